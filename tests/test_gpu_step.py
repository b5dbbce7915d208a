"""The fused decoding step (sgd_step) against the oracle.

sgd_step is sgd_propose_with_update followed by sgd_ingest of the step's
finished docs; up to 64 docs run inside the same kernel launch (one extra CTA
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


@pytest.mark.parametrize("mode", [1, 2], ids=["one-launch", "two-launch"])
@pytest.mark.parametrize("finish_frac,B", [(0.1, 64), (0.45, 128), (0.6, 128)],
                         ids=["6-docs", "57-docs", "76-docs"])
def test_fused_step_matches_oracle(finish_frac, B, mode):
    """A few docs per step and 33-64 docs (in-kernel ingest); more than 64
    docs (two calls)."""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=2048)
    ls = H.Lockstep(cfg, seed=3, B=B, steps=14, finish_frac=finish_frac, corpus=1 << 16, fused=True,
                    drafter_over=dict(propose_mode=mode))
    ls.prefill(seed=3)
    docs = 0
    for _ in range(14):
        sd = ls.step(check_state=True)
        docs += sd.finished.shape[0]
        _ring_matches(ls)
    assert docs > 0 and ls.generation >= 2
    if ls.build_pending:  # (a rebuild the last steps started)
        ls.swap()
    ls.build_and_swap()
    text, sa, _ = ls.dr.export_snapshot()
    assert text.cpu().numpy().tolist() == ls.X.tolist()
    assert np.array_equal(sa.cpu().numpy(), O.suffix_array(ls.X))
    assert ls.dr.get_error() == 0
    ls.close()


@pytest.mark.parametrize("delta", [0, 2048], ids=["no-delta", "delta"])
@pytest.mark.parametrize("mode", [1, 2], ids=["one-launch", "two-launch"])
def test_fused_step_graph_replays(mode, delta):
    """One captured sgd_step replayed with new inputs staged into its buffers:
    every replay must wait for its own rows' updates (fresh epoch per launch).
    With a delta the rows also match the docs ingested since the last swap."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B, T, m = 97, 256, 24, 5, 6
    rng = np.random.default_rng(11)
    C = 2048
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=8, max_tree_depth=16,
                       max_occurrences=16, max_sampled=T, corpus_capacity=C, max_docs=256,
                       propose_mode=mode, delta_capacity=delta)
    ring = O.Ring(C, 256, V)
    since = 0
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
        Xc = O.corpus_text(X, ring.delta(since, delta)) if delta else X
        orc = O.propose(p, tok, n, X=Xc)
        H.compare(out, orc, ctx="replay %d" % it)
        assert np.array_equal(g_n.cpu().numpy(), n)
        assert np.array_equal(g_tok.cpu().numpy(), tok)
        ring.ingest(tok, rows, starts, lens, num_tokens=n)
        live, nd = dr.corpus_stats()
        assert (live, nd) == (ring.live, ring.ndocs)
        if it % 3 == 2:
            dr.build_sa(side)
            assert dr.poll(wait=True)[0] == 1
            X, since = ring.snapshot(), ring.pushed
            text, sa, _ = dr.export_snapshot()
            assert text.cpu().numpy().tolist() == X.tolist()
    assert dr.get_error() == 0
    dr.close()


@pytest.mark.parametrize("delta", [0, 1024], ids=["no-delta", "delta"])
def test_step_wait_injection_skips_docs_and_recovers(delta):
    """A bounded wait that runs out (test injection: the awaited signal is never
    sent) skips the step's docs with SGD_ERR_INGEST_WAIT; drafting is unaffected
    and the next step ingests normally."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter, _lib as L
    V, S, B, T = 31, 128, 8, 3
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=4, max_sampled=T,
                       corpus_capacity=1024, delta_capacity=delta)
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
    if delta:  # the two docs are in the delta: the next step matches them
        ring = O.Ring(1024, 65536, V)
        ring.ingest(full, [0, 3], [0, 5], [10, 12], num_tokens=n)  # (tokens the updates left alone)
        out = dr.step(g_tok, g_n, torch.from_numpy(samp).cuda(), rows[:0], st[:0], ln[:0])
        torch.cuda.synchronize()
        O.update_state(full, n, samp, V)
        H.compare(out, O.propose(p, full, n, X=ring.delta(0, delta)), ctx="delta step")
    dr.close()


@pytest.mark.parametrize("nb", [1, 4], ids=["longest", "backoff4"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned-in-place", "pageable-staged"])
def test_step_host_matches_device_step(pinned, nb):
    """sgd_step_host gives exactly what sgd_step gives on device buffers, step
    after step: with page-locked host buffers the kernels read and write them
    in place, with pageable ones the library stages copies; also with
    multi-length backoff (update, backoff and ingest launches)."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    V, S, B, T, k = 97, 256, 24, 5, 8
    rng = np.random.default_rng(21)
    kw = dict(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=16, max_occurrences=16,
              max_sampled=T, corpus_capacity=2048, max_docs=256, num_backoff=nb)
    A, Bd = SuffixDrafter(**kw), SuffixDrafter(**kw)
    tok = np.zeros((B, S), dtype=np.int32)
    n = rng.integers(40, 120, size=B).astype(np.int32)
    base = rng.integers(0, 12, size=64)
    for b in range(B):
        tok[b, :n[b]] = np.resize(np.roll(base, b % 5), n[b])
    ta, na = torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda()
    tb, nb = ta.clone(), na.clone()
    outa = A.new_outputs(B)
    # outputs as views of one host block in the library's order (one copy back when staged)
    ob = pin(torch.empty(B * k + B + B + B * k + 2 * B, dtype=torch.int32))
    h_drafts, h_nv = ob[:B * k].view(B, k), ob[B * k:B * k + B]
    h_score = ob[B * k + B:B * k + 2 * B].view(torch.float32)
    h_probs = ob[B * k + 2 * B:2 * B * k + 2 * B].view(torch.float32).view(B, k)
    h_mi = ob[2 * B * k + 2 * B:].view(B, 2)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    for it in range(8):
        samp = rng.integers(0, 12, size=(B, T)).astype(np.int32)
        m = int(rng.integers(0, 6))
        rows = rng.choice(B, size=m, replace=False).astype(np.int32)
        # docs: the first 30 tokens of each row, always inside the row after the update;
        # odd steps pass the inputs as views of one host block (moved at once when staged)
        if it % 2:
            blk = pin(torch.from_numpy(np.concatenate([samp.ravel(), rows, np.zeros(m, np.int32),
                                                       np.full(m, 30, np.int32)]).astype(np.int32)))
            h_samp = blk[:B * T].view(B, T)
            h_rows, h_st, h_ln = blk[B * T:B * T + m], blk[B * T + m:B * T + 2 * m], blk[B * T + 2 * m:]
        else:
            h_samp = pin(torch.from_numpy(samp))
            h_rows = pin(torch.from_numpy(rows))
            h_st = pin(torch.zeros(m, dtype=torch.int32))
            h_ln = pin(torch.full((m,), 30, dtype=torch.int32))
        A.step(ta, na, h_samp.cuda(), h_rows.cuda(), h_st.cuda(), h_ln.cuda(), out=outa)
        Bd.step_host(tb, nb, h_samp, h_rows, h_st, h_ln, h_drafts, h_nv, h_score, h_probs, h_mi,
                     stream=stream)
        stream.synchronize()
        assert torch.equal(outa.drafts.cpu(), h_drafts) and torch.equal(outa.num_valid.cpu(), h_nv)
        assert torch.equal(outa.score.cpu(), h_score) and torch.equal(outa.probs.cpu(), h_probs)
        assert torch.equal(outa.match_info.cpu(), h_mi)
        assert torch.equal(ta, tb) and torch.equal(na, nb)
        assert A.corpus_stats() == Bd.corpus_stats()
        if it % 3 == 2:
            for d in (A, Bd):
                d.build_sa(side)
                assert d.poll(wait=True)[0] == 1
    assert A.get_error() == 0 and Bd.get_error() == 0
    A.close()
    Bd.close()


def test_bound_step_host_reuses_buffers():
    """bind_step_host: one marshalled call reused over fixed pinned buffers whose
    contents change between steps gives the same results as step()."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B, T, k, m = 61, 128, 12, 4, 6, 3
    rng = np.random.default_rng(33)
    kw = dict(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=12, max_occurrences=8,
              max_sampled=T, corpus_capacity=1024, max_docs=128)
    A, Bd = SuffixDrafter(**kw), SuffixDrafter(**kw)
    tok = rng.integers(0, 7, size=(B, S)).astype(np.int32)
    n = np.full(B, 40, dtype=np.int32)
    ta, na = torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda()
    tb, nb = ta.clone(), na.clone()
    outa = A.new_outputs(B)
    h_in = torch.empty(B * T + 3 * m, dtype=torch.int32).pin_memory()
    h_out = torch.empty(B * k + B, dtype=torch.int32).pin_memory()
    h_drafts, h_nv = h_out[:B * k].view(B, k), h_out[B * k:]
    stream = torch.cuda.current_stream()
    step = Bd.bind_step_host(tb, nb, h_in[:B * T].view(B, T), h_in[B * T:B * T + m],
                             h_in[B * T + m:B * T + 2 * m], h_in[B * T + 2 * m:], h_drafts, h_nv,
                             stream=stream)
    for it in range(6):
        samp = rng.integers(0, 7, size=(B, T)).astype(np.int32)
        rows = rng.choice(B, size=m, replace=False).astype(np.int32)
        blk = np.concatenate([samp.ravel(), rows, np.zeros(m, np.int32), np.full(m, 20, np.int32)])
        h_in.numpy()[:] = blk
        d = torch.from_numpy(blk).cuda()
        A.step(ta, na, d[:B * T].view(B, T), d[B * T:B * T + m], d[B * T + m:B * T + 2 * m],
               d[B * T + 2 * m:], out=outa)
        step()
        stream.synchronize()
        assert torch.equal(outa.drafts.cpu(), h_drafts) and torch.equal(outa.num_valid.cpu(), h_nv)
        assert torch.equal(ta, tb) and torch.equal(na, nb)
        assert A.corpus_stats() == Bd.corpus_stats()
    A.close()
    Bd.close()


@pytest.mark.parametrize("mode", [1, 2], ids=["one-launch", "two-launch"])
def test_fixed_length_drafts_lockstep(mode):
    """Model Runner V2 drafts (draft_mode 1: k tokens, the unstopped vote, the
    row's last token in the empty slots) through the fused step, with the
    corpus and rebuilds, against the oracle's fixed_length rule."""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=4096)
    ls = H.Lockstep(cfg, seed=9, B=64, steps=10, finish_frac=0.1, corpus=1 << 16, fused=True,
                    drafter_over=dict(propose_mode=mode, draft_mode=1),
                    param_over=dict(fixed_length=True))
    ls.prefill(seed=9)
    for _ in range(10):
        ls.step(check_state=True)
        nv = ls.out.num_valid.cpu().numpy()
        assert (nv == cfg.k).all()  # every row here is active and non-empty
    assert ls.dr.get_error() == 0
    ls.close()


SCORE_CASES = [
    (dict(propose_mode=1), {}, 0),
    (dict(propose_mode=2), {}, 0),
    (dict(propose_mode=1), {}, 1 << 16),
    (dict(propose_mode=1, draft_mode=1), dict(fixed_length=True), 0),
    (dict(propose_mode=1, corpus_records=0, corpus_gram_index=0), {}, 0),
]


@pytest.mark.parametrize("over,pover,delta", SCORE_CASES,
                         ids=["one-launch", "two-launch", "one-launch+delta", "fixed-length",
                              "text+descent"])
def test_select_by_score_lockstep(over, pover, delta):
    """Score-ranked selection (select_by_score 1: the row's and the corpus's
    candidates both voted, the better score wins) through the fused step,
    with rebuilds, against the oracle -- in both launch modes, with a delta,
    with Model Runner V2 drafts and through the text / descent corpus path."""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=4096)
    ls = H.Lockstep(cfg, seed=13, B=64, steps=10, finish_frac=0.1, corpus=1 << 16, fused=True,
                    drafter_over=dict(over, select_by_score=1),
                    param_over=dict(pover, select_by_score=True), delta=delta)
    ls.prefill(seed=13)
    switched = 0
    for i in range(10):
        ls.step(check_state=True)
        if i >= 1:  # the rule must change some rows' source for the test to mean anything
            a = O.propose(ls.p, ls.o_tok, ls.o_n, X=ls.oracle_corpus(), threads=H.THREADS)
            p2 = O.Params(**{k: getattr(ls.p, k) for k in ("S", "V", "k", "D", "R", "offset")},
                          factor=ls.p.factor, min_prob=ls.p.min_prob,
                          fixed_length=ls.p.fixed_length)
            b2 = O.propose(p2, ls.o_tok, ls.o_n, X=ls.oracle_corpus(), threads=H.THREADS)
            switched += int((a.match_info[:, 1] != b2.match_info[:, 1]).sum())
    assert switched > 0
    assert ls.dr.get_error() == 0
    ls.close()
