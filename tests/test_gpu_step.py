"""The fused decoding step (sgd_step) against the oracle.

sgd_step is sgd_propose_with_update followed by sgd_ingest of the step's
finished docs; up to 32 docs run inside the same kernel launch (one extra CTA
appends them once their rows are updated).  Drafts, the updated rows, the
ring and every snapshot built from it must equal the oracle's, step after
step, whether the step runs as one launch or as the two calls.
"""
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _mods():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from model_free_suffix_gb300 import build
    build.build()
    from model_free_suffix_gb300 import workload as W
    from oracle import oracle as O
    import harness as H
    return W, O, H


def _ring_matches(ls):
    live, nd = ls.dr.corpus_stats()
    assert (live, nd) == (ls.ring.live, ls.ring.ndocs)


@pytest.mark.parametrize("finish_frac", [0.1, 0.6])
def test_fused_step_matches_oracle(finish_frac):
    """0.1: a few docs per step (in-kernel ingest); 0.6: more than 32 docs (two calls)."""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=2048)
    ls = H.Lockstep(cfg, seed=3, B=64, steps=14, finish_frac=finish_frac, corpus=1 << 16, fused=True)
    ls.prefill(seed=3)
    docs = 0
    for _ in range(14):
        sd = ls.step(check_state=True)
        docs += sd.finished.shape[0]
        _ring_matches(ls)
    assert docs > 0 and ls.generation >= 2
    ls.build_and_swap()
    text, sa, _ = ls.dr.export_snapshot()
    assert text.cpu().numpy().tolist() == ls.X.tolist()
    assert np.array_equal(sa.cpu().numpy(), O.suffix_array(ls.X))
    assert ls.dr.get_error() == 0
    ls.close()


def test_fused_step_graph_replays():
    """One captured sgd_step replayed with new inputs staged into its buffers:
    every replay must wait for its own rows' updates (fresh epoch per launch)."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B, T, m = 97, 256, 24, 5, 6
    rng = np.random.default_rng(11)
    C = 2048
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=8, max_tree_depth=16,
                       max_occurrences=16, max_sampled=T, corpus_capacity=C, max_docs=256)
    ring = O.Ring(C, 256, V)
    p = O.Params(S=S, V=V, k=8, D=16, R=16)
    tok = np.zeros((B, S), dtype=np.int32)
    n = rng.integers(40, 120, size=B).astype(np.int32)
    base = rng.integers(0, 12, size=64)
    for b in range(B):
        tok[b, :n[b]] = np.resize(np.roll(base, b % 5), n[b])
    g_tok, g_n = torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda()
    d_samp = torch.zeros((B, T), dtype=torch.int32, device="cuda")
    d_rows = torch.zeros(m, dtype=torch.int32, device="cuda")
    d_st = torch.zeros(m, dtype=torch.int32, device="cuda")
    d_ln = torch.zeros(m, dtype=torch.int32, device="cuda")
    out = dr.new_outputs(B)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dr.step(g_tok, g_n, d_samp, d_rows, d_st, d_ln, out=out, stream=stream)
    torch.cuda.synchronize()
    assert (g_n.cpu().numpy() == n).all()  # capture ran nothing
    side = torch.cuda.Stream()
    X = None
    for it in range(8):
        samp = rng.integers(0, 12, size=(B, T)).astype(np.int32)
        samp[rng.random((B, T)) < 0.1] = -1
        rows = rng.choice(B, size=m, replace=False).astype(np.int32)
        n_after = n.copy()
        O.update_state(tok, n_after, samp, V)
        starts = (n_after[rows] // 3).astype(np.int32)
        lens = (n_after[rows] - starts).astype(np.int32)
        d_samp.copy_(torch.from_numpy(samp))
        d_rows.copy_(torch.from_numpy(rows))
        d_st.copy_(torch.from_numpy(starts))
        d_ln.copy_(torch.from_numpy(lens))
        graph.replay()
        torch.cuda.synchronize()
        n[:] = n_after
        orc = O.propose(p, tok, n, X=X)
        H.compare(out, orc, ctx="replay %d" % it)
        assert np.array_equal(g_n.cpu().numpy(), n)
        assert np.array_equal(g_tok.cpu().numpy(), tok)
        ring.ingest(tok, rows, starts, lens, num_tokens=n)
        live, nd = dr.corpus_stats()
        assert (live, nd) == (ring.live, ring.ndocs)
        if it % 3 == 2:
            dr.build_sa(side)
            assert dr.poll(wait=True)[0] == 1
            X = ring.snapshot()
            text, sa, _ = dr.export_snapshot()
            assert text.cpu().numpy().tolist() == X.tolist()
    assert dr.get_error() == 0
    dr.close()


def test_step_wait_injection_skips_docs_and_recovers():
    """A bounded wait that runs out (test injection: the awaited signal is never
    sent) skips the step's docs with SGD_ERR_INGEST_WAIT; drafting is unaffected
    and the next step ingests normally."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter, _lib as L
    V, S, B, T = 31, 128, 8, 3
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=4, max_sampled=T,
                       corpus_capacity=1024)
    p = O.Params(S=S, V=V, k=4)
    tok = np.tile(np.arange(20, dtype=np.int32) % 7, (B, 1))
    full = np.zeros((B, S), dtype=np.int32)
    full[:, :20] = tok
    n = np.full(B, 20, dtype=np.int32)
    g_tok, g_n = torch.from_numpy(full.copy()).cuda(), torch.from_numpy(n.copy()).cuda()
    samp = np.tile(np.array([[1, 2, 3]], dtype=np.int32), (B, 1))
    rows = torch.tensor([0, 3], dtype=torch.int32, device="cuda")
    st = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    ln = torch.tensor([10, 12], dtype=torch.int32, device="cuda")
    dr.debug_inject(L.INJECT_STEP_WAIT)
    out = dr.step(g_tok, g_n, torch.from_numpy(samp).cuda(), rows, st, ln)
    torch.cuda.synchronize()
    O.update_state(full, n, samp, V)
    H.compare(out, O.propose(p, full, n, X=None), ctx="injected step")
    assert dr.get_error(clear=True) == L.ERR_INGEST_WAIT
    assert dr.corpus_stats() == (0, 0)
    out = dr.step(g_tok, g_n, torch.from_numpy(samp).cuda(), rows, st, ln)
    torch.cuda.synchronize()
    O.update_state(full, n, samp, V)
    H.compare(out, O.propose(p, full, n, X=None), ctx="next step")
    assert dr.get_error() == 0
    assert dr.corpus_stats() == (10 + 1 + 12 + 1, 2)
    dr.close()
