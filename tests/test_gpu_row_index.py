"""The per-row bigram position index (row_index = 1) against the oracle.

With the index on, a row's own match comes from the earlier positions of its
last two tokens (kept by every update, rebuilt by sgd_reset_rows) instead of
a scan of the row; rows whose last bigram is frequent, or new with no corpus
match of 2 or more, are still scanned.  The drafts must stay those of the
plain definition (the oracle), bit for bit, through serving traces with rows
restarting, updates through every entry point, inactive rows, rows changed
without a reset, repeated resets (the 8-bit generation wraps) and edge knobs.
Row statistics show that the index path is taken.
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
    from model_free_suffix_gb300 import SuffixDrafter, workload as W
    from oracle import oracle as O
    import harness as H
    return SuffixDrafter, W, O, H


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a)).to(dtype).cuda()


def _how(stats, B):
    return (stats.view(-1, 4)[:B, 3].cpu().numpy() >> 8) & 15


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused-step"])
@pytest.mark.parametrize("cfg_name", ["c2", "c3", "c5"])
def test_serving_trace_lockstep(cfg_name, fused):
    """Serving traces (rows finishing and restarting) with the index on."""
    SuffixDrafter, W, O, H = _mods()
    cfg = W.CONFIGS[cfg_name]
    B, corpus = {"c2": (48, 0), "c3": (96, 1 << 16), "c5": (24, 1 << 17)}[cfg_name]
    cfg = dataclasses.replace(cfg, rebuild_tokens=4096)
    ls = H.Lockstep(cfg, seed=11, B=B, steps=10, finish_frac=0.1, corpus=corpus,
                    fused=fused, drafter_over=dict(row_index=1))
    if corpus:
        ls.prefill(seed=11)
    stats = torch.zeros(B * 4, dtype=torch.int32, device=ls.dr.device)
    ls.dr.set_row_stats(stats)
    used = 0
    for _ in range(10):
        ls.step(check_state=True)
        used += int((_how(stats, B) != 0).sum())
    assert used > 0, "the index never replaced a scan"
    assert ls.dr.get_error() == 0
    ls.close()


def _rows(rng, B, S, V, kinds):
    tok = np.full((B, S), -1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        kind = kinds[b % len(kinds)]
        if kind == "periodic":   # the last bigram occurs many times: scanned
            nb = int(rng.integers(S // 4, S // 2))
            p = int(rng.integers(1, 6))
            base = rng.integers(0, V, size=p)
            tok[b, :nb] = base[np.arange(nb) % p]
        elif kind == "few":      # a span repeated 2-5 times among fresh ids, also at the end
            nb = int(rng.integers(64, S // 2))
            x = rng.integers(0, V, size=nb)
            L = int(rng.integers(3, 30))
            span = rng.integers(0, V, size=L)
            for _ in range(int(rng.integers(1, 5))):
                at = int(rng.integers(0, nb - 2 * L))
                x[at:at + L] = span
            x[nb - L:] = span
            tok[b, :nb] = x
        elif kind == "short":
            nb = int(rng.integers(0, 4))
            tok[b, :nb] = rng.integers(0, V, size=nb)
        elif kind == "full":
            nb = S - int(rng.integers(0, 3))
            tok[b, :nb] = rng.integers(0, V, size=nb)
        else:                    # random
            nb = int(rng.integers(2, S - 40))
            tok[b, :nb] = rng.integers(0, V, size=nb)
        n[b] = nb
    return tok, n


GRID = [
    # (V, S, k, D, R, T, corpus)
    (3, 512, 8, 24, 64, 9, False),
    (50, 1024, 16, 24, 64, 17, True),
    (1000, 2048, 16, 32, 64, 33, True),
    (7, 512, 4, 2, 1, 5, False),
    (20, 1024, 32, 128, 128, 40, False),
    (151936, 4096, 16, 24, 64, 17, True),
]


@pytest.mark.parametrize("grid", GRID, ids=lambda g: "V%d_S%d_k%d_D%d_R%d_T%d" % g[:6])
def test_structured_rows_multi_step(grid):
    """Rows where the last bigram is new, rare or frequent, short and full
    rows, updates of every width, inactive rows; propose with and without an
    update, and the standalone update followed by a propose."""
    SuffixDrafter, W, O, H = _mods()
    V, S, k, D, R, T, with_corpus = grid
    rng = np.random.default_rng(V * 7 + S)
    B = 64
    tok, n = _rows(rng, B, S, V, ["periodic", "few", "short", "full", "random", "few"])
    C = 1 << 14
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=D,
                       max_occurrences=R, max_sampled=T, corpus_capacity=C if with_corpus else 0,
                       row_index=1)
    p = O.Params(S=S, V=V, k=k, D=D, R=R)
    X = None
    if with_corpus:  # a corpus made of pieces of the rows, so that it matches
        docs = []
        for b in range(B):
            if n[b] > 40:
                s0 = int(rng.integers(0, n[b] - 32))
                docs.append(tok[b, s0:s0 + int(rng.integers(8, 32))])
        m = len(docs)
        buf = np.full((m, S), -1, dtype=np.int32)
        lens = np.array([d.shape[0] for d in docs], dtype=np.int32)
        for i, d in enumerate(docs):
            buf[i, :d.shape[0]] = d
        dr.ingest(_dev(buf), _dev(np.arange(m)), _dev(np.zeros(m)), _dev(lens))
        ring = O.Ring(C, 65536, V)
        ring.ingest(buf, np.arange(m), np.zeros(m), lens)
        dr.build_sa(torch.cuda.Stream())
        assert dr.poll(wait=True)[0] == 1
        X = ring.snapshot()
    g_tok, g_n = _dev(tok), _dev(n)
    dr.reset_rows(g_tok, g_n, _dev(np.arange(B)))
    stats = torch.zeros(B * 4, dtype=torch.int32, device="cuda")
    dr.set_row_stats(stats)
    used = 0
    for it in range(8):
        active = (rng.random(B) < 0.85).astype(np.uint8)
        if it % 4 == 3:  # no update: the same rows again
            out = dr.propose(g_tok, g_n, active=_dev(active, torch.uint8))
        else:
            samp = np.full((B, T), -1, dtype=np.int32)
            for b in range(B):
                a = int(rng.integers(0, T + 1))
                # continue the row's own text at times (matches extend), else fresh ids
                if n[b] > a + 2 and rng.random() < 0.5:
                    s0 = int(rng.integers(0, n[b] - a))
                    samp[b, :a] = tok[b, s0:s0 + a]
                else:
                    samp[b, :a] = rng.integers(0, V, size=a)
            if it % 4 == 2:  # the standalone update, then a propose
                dr.update_state(g_tok, g_n, _dev(samp))
                out = dr.propose(g_tok, g_n, active=_dev(active, torch.uint8))
            else:
                out = dr.propose_with_update(g_tok, g_n, _dev(samp), active=_dev(active, torch.uint8))
            O.update_state(tok, n, samp, V)
        orc = O.propose(p, tok, n, X=X, active=active, threads=H.THREADS)
        H.compare(out, orc, ctx="iteration %d" % it)
        used += int((_how(stats, B) == 1).sum())
        assert np.array_equal(g_n.cpu().numpy(), n) and np.array_equal(g_tok.cpu().numpy(), tok)
    assert used > 0
    assert dr.get_error() == 0
    dr.close()


def test_rows_changed_without_reset_stay_exact_and_resets_repeat():
    """A row rewritten with a new length but no reset is scanned (stale index
    detected); a row rewritten with the same length and reset drafts from its
    new contents; 300 resets of the same rows wrap the generation; a row
    listed twice in one reset call is reset once."""
    SuffixDrafter, W, O, H = _mods()
    V, S, B = 5, 1024, 8
    rng = np.random.default_rng(3)
    tok, n = _rows(rng, B, S, V, ["few", "random"])
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=8, max_tree_depth=24,
                       max_occurrences=64, max_sampled=9, row_index=1)
    p = O.Params(S=S, V=V, k=8, D=24, R=64)
    g_tok, g_n = _dev(tok), _dev(n)
    dr.reset_rows(g_tok, g_n, _dev(np.arange(B)))
    H.compare(dr.propose(g_tok, g_n), O.propose(p, tok, n))
    # rewritten, new lengths, no reset
    tok2, n2 = _rows(rng, B, S, V, ["random", "few"])
    for b in range(B):  # (every length differs from the indexed one)
        if n2[b] == n[b]:
            tok2[b, n2[b] - 1] = -1
            n2[b] -= 1
    g_tok.copy_(_dev(tok2))
    g_n.copy_(_dev(n2))
    H.compare(dr.propose(g_tok, g_n), O.propose(p, tok2, n2), ctx="stale, scanned")
    # same lengths, new contents, reset (rows listed twice and out of range too)
    tok3 = np.where(tok2 >= 0, (tok2 + 1) % V, -1).astype(np.int32)
    g_tok.copy_(_dev(tok3))
    dr.reset_rows(g_tok, g_n, _dev(np.concatenate([np.arange(B), np.arange(B), [B + 5, -1]])))
    H.compare(dr.propose(g_tok, g_n), O.propose(p, tok3, n2), ctx="after reset")
    for r in range(300):
        dr.reset_rows(g_tok, g_n, _dev(np.arange(B)))
    samp = rng.integers(0, V, size=(B, 9)).astype(np.int32)
    out = dr.propose_with_update(g_tok, g_n, _dev(samp))
    O.update_state(tok3, n2, samp, V)
    H.compare(out, O.propose(p, tok3, n2), ctx="after 300 resets")
    dr.close()


def test_row_index_knob_validation():
    SuffixDrafter, W, O, H = _mods()
    from model_free_suffix_gb300 import _lib as L
    for over in [dict(propose_mode=2), dict(delta_capacity=1024, corpus_capacity=1 << 14),
                 dict(select_by_score=1), dict(num_backoff=2), dict(vocab_size=1 << 25)]:
        kw = dict(max_batch=4, seq_capacity=256, vocab_size=100, row_index=1)
        kw.update(over)
        with pytest.raises(L.SgdError):
            SuffixDrafter(**kw)
