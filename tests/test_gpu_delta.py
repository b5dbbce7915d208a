"""The delta: docs placed after the current snapshot was linearised, matched by
a brute-force scan before the next rebuild indexes them.

The oracle's corpus is the snapshot followed by the delta's text (oracle
Ring.delta, cut at the capacity); the GPU reads the delta in place from the
ring.  Drafts, counts and match info bit-exact, scores and probabilities
bit-equal as float32 words, through every path: one fused launch per step (the
ingest CTA appending while the rows scan), the two-launch mode, the plain
propose, a ring that wraps and evicts, a delta larger than its capacity.
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


MODES = [
    dict(propose_mode=1),
    dict(propose_mode=2),
    dict(propose_mode=1, corpus_records=0, corpus_gram_index=0),
]


@pytest.mark.parametrize("over", MODES, ids=["one-launch", "two-launch", "text+descent"])
@pytest.mark.parametrize("fused", [True, False], ids=["step", "propose+ingest"])
@pytest.mark.parametrize("delta", [1 << 16, 700], ids=["whole-delta", "cut-delta"])
def test_delta_lockstep(delta, fused, over):
    """A serving trace with rebuilds every 4096 new tokens: between swaps the
    rows also match the docs finished since the snapshot was taken."""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=4096)
    ls = H.Lockstep(cfg, seed=5, B=64, steps=16, finish_frac=0.15, corpus=1 << 16, fused=fused,
                    drafter_over=over, delta=delta)
    ls.prefill(seed=5)
    changed = 0
    for i in range(16):
        ls.step(check_state=True)
        if i >= 2:  # the delta must decide some rows for the test to mean anything
            with_d = O.propose(ls.p, ls.o_tok, ls.o_n, X=ls.oracle_corpus(), threads=H.THREADS)
            without = O.propose(ls.p, ls.o_tok, ls.o_n, X=ls.X, threads=H.THREADS)
            changed += int((with_d.match_info != without.match_info).any(axis=1).sum())
        live, nd = ls.dr.corpus_stats()
        assert (live, nd) == (ls.ring.live, ls.ring.ndocs)
    assert changed > 0
    assert ls.dr.get_error() == 0
    ls.close()


def _docs_rows(rng, V, S, base, m, lo, hi):
    """m docs cut from a shared base sequence (so rows and docs share n-grams)."""
    buf = np.zeros((m, S), dtype=np.int32)
    lens = rng.integers(lo, hi, size=m).astype(np.int32)
    for i in range(m):
        off = int(rng.integers(0, base.shape[0] - lens[i]))
        buf[i, :lens[i]] = base[off:off + lens[i]]
    return buf, lens


@pytest.mark.parametrize("C,delta", [(1024, 1024), (1024, 384), (2048, 2048)])
def test_delta_wraps_and_evicts(C, delta):
    """A small ring that wraps many times: the delta runs across the ring's end,
    the snapshot's docs are evicted while it stays current, and with no swap
    for a while every live doc is a delta doc (and the oldest of those are
    evicted in turn)."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B, k, D, R = 23, 256, 16, 8, 16, 16
    rng = np.random.default_rng(C + delta)
    base = rng.integers(0, V, size=400).astype(np.int32)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=D,
                       max_occurrences=R, corpus_capacity=C, max_docs=64, delta_capacity=delta)
    ring = O.Ring(C, 64, V)
    p = O.Params(S=S, V=V, k=k, D=D, R=R)
    side = torch.cuda.Stream()
    X, since = None, 0
    tok = np.zeros((B, S), dtype=np.int32)
    n = rng.integers(24, 200, size=B).astype(np.int32)
    for b in range(B):
        off = int(rng.integers(0, base.shape[0] - n[b]))
        tok[b, :n[b]] = base[off:off + n[b]]
        tok[b, n[b] - 6:n[b]] = rng.integers(0, V, size=6)  # a tail the row itself may not hold
    g_tok, g_n = torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda()
    for it in range(24):
        buf, lens = _docs_rows(rng, V, S, base, int(rng.integers(1, 5)), 20, 160)
        g = torch.from_numpy(buf).cuda()
        rows = torch.arange(buf.shape[0], dtype=torch.int32, device="cuda")
        dr.ingest(g, rows, torch.zeros_like(rows), torch.from_numpy(lens).cuda())
        ring.ingest(buf, np.arange(buf.shape[0]), np.zeros(buf.shape[0]), lens)
        if it % 8 == 3:  # a swap now and then; long stretches without
            dr.build_sa(side)
            assert dr.poll(wait=True)[0] == 1
            X, since = ring.snapshot(), ring.pushed
        out = dr.propose(g_tok, g_n)
        torch.cuda.synchronize()
        Xd = O.corpus_text(X, ring.delta(since, delta))
        H.compare(out, O.propose(p, tok, n, X=Xd), ctx="iteration %d" % it)
    assert dr.get_error() == 0
    dr.close()


@pytest.mark.parametrize("mode", [1, 2], ids=["one-launch", "two-launch"])
def test_fused_step_appending_over_the_visible_delta(mode):
    """No swap at all and a ring that fills: every live doc is in the delta and
    each step's docs overwrite the oldest of them, which the same launch's
    rows may be reading.  The ingest CTA then waits for every row to finish
    with the ring; results stay those of propose-then-ingest."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B, T, k = 29, 256, 32, 4, 8
    C = 1024
    rng = np.random.default_rng(8)
    base = rng.integers(0, V, size=300).astype(np.int32)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=16,
                       max_occurrences=16, max_sampled=T, corpus_capacity=C, max_docs=128,
                       delta_capacity=C, propose_mode=mode)
    ring = O.Ring(C, 128, V)
    p = O.Params(S=S, V=V, k=k, D=16, R=16)
    tok = np.zeros((B, S), dtype=np.int32)
    n = rng.integers(30, 150, size=B).astype(np.int32)
    for b in range(B):
        off = int(rng.integers(0, base.shape[0] - n[b]))
        tok[b, :n[b]] = base[off:off + n[b]]
    g_tok, g_n = torch.from_numpy(tok.copy()).cuda(), torch.from_numpy(n.copy()).cuda()
    for it in range(20):
        samp = rng.integers(0, V, size=(B, T)).astype(np.int32)
        m = int(rng.integers(2, 7))
        rows = rng.choice(B, size=m, replace=False).astype(np.int32)
        n_after = n.copy()
        O.update_state(tok, n_after, samp, V)
        starts = np.zeros(m, dtype=np.int32)
        lens = np.minimum(n_after[rows], 200).astype(np.int32)
        out = dr.step(g_tok, g_n, torch.from_numpy(samp).cuda(), torch.from_numpy(rows).cuda(),
                      torch.from_numpy(starts).cuda(), torch.from_numpy(lens).cuda())
        torch.cuda.synchronize()
        n[:] = n_after
        H.compare(out, O.propose(p, tok, n, X=ring.delta(0, C)), ctx="step %d" % it)
        ring.ingest(tok, rows, starts, lens, num_tokens=n)
        assert dr.corpus_stats() == (ring.live, ring.ndocs)
        assert dr.get_error() == 0
    assert ring.pushed > ring.ndocs  # the ring wrapped: docs were evicted
    dr.close()


def test_delta_results_equal_the_rebuilt_index():
    """Without evictions, what the rows draft from snapshot + delta is what they
    draft once the same docs are indexed by a rebuild and swapped in."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B = 41, 512, 48
    rng = np.random.default_rng(3)
    base = rng.integers(0, V, size=1500).astype(np.int32)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=12, max_tree_depth=24,
                       max_occurrences=32, corpus_capacity=1 << 16, delta_capacity=1 << 16)
    ring = O.Ring(1 << 16, 65536, V)
    p = O.Params(S=S, V=V, k=12, D=24, R=32)
    side = torch.cuda.Stream()
    # 20 docs indexed, then 40 more in one call (more than the in-CTA ingest
    # takes: the multi-kernel path, whose signature kernel then runs)
    buf, lens = _docs_rows(rng, V, S, base, 60, 50, 400)
    rows = torch.arange(60, dtype=torch.int32, device="cuda")
    g = torch.from_numpy(buf).cuda()
    dr.ingest(g[:20], rows[:20], torch.zeros_like(rows[:20]), torch.from_numpy(lens[:20]).cuda())
    ring.ingest(buf[:20], np.arange(20), np.zeros(20), lens[:20])
    dr.build_sa(side)
    assert dr.poll(wait=True)[0] == 1
    since = ring.pushed
    dr.ingest(g[20:], rows[:40], torch.zeros_like(rows[:40]), torch.from_numpy(lens[20:]).cuda())
    ring.ingest(buf[20:], np.arange(40), np.zeros(40), lens[20:])
    tok = np.zeros((B, S), dtype=np.int32)
    n = rng.integers(16, 400, size=B).astype(np.int32)
    for b in range(B):
        off = int(rng.integers(0, base.shape[0] - n[b]))
        tok[b, :n[b]] = base[off:off + n[b]]
    g_tok, g_n = torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda()
    before = dr.propose(g_tok, g_n)
    torch.cuda.synchronize()
    # no doc was evicted: the snapshot taken now is the old one followed by the delta
    H.compare(before, O.propose(p, tok, n, X=ring.snapshot()), ctx="before the swap")
    snap = [t.clone() for t in (before.drafts, before.num_valid, before.score, before.probs,
                                before.match_info)]
    dr.build_sa(side)
    assert dr.poll(wait=True)[0] == 1
    after = dr.propose(g_tok, g_n)
    torch.cuda.synchronize()
    for x, y in zip(snap, (after.drafts, after.num_valid, after.score, after.probs,
                           after.match_info)):
        assert torch.equal(x, y)
    assert ring.pushed > since
    assert dr.get_error() == 0
    dr.close()
