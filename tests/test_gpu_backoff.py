"""Multi-length backoff (num_backoff > 1): every support threshold's length is
a candidate on each path and the best score wins.

The oracle computes every match length by brute force and ranks the
candidates; the GPU measures lengths exactly too (row ends, the hits of the
last two tokens' suffix-array interval, every delta position) and selects the
R most recent ends per candidate.  Drafts, counts and match info bit-exact,
scores and probabilities bit-equal as float32 words.
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


CASES = [
    (2, dict(), {}, 0, True),
    (8, dict(), {}, 0, True),
    (8, dict(), {}, 1 << 16, True),
    (4, dict(), {}, 1 << 16, False),
    (8, dict(draft_mode=1), dict(fixed_length=True), 0, True),
    (3, dict(propose_mode=2, corpus_records=0, corpus_gram_index=0), {}, 0, False),
]


@pytest.mark.parametrize("nb,over,pover,delta,fused", CASES,
                         ids=["nb2", "nb8", "nb8+delta", "nb4+delta-unfused", "nb8-fixed-length",
                              "nb3-text-descent-unfused"])
def test_backoff_lockstep(nb, over, pover, delta, fused):
    """A serving trace with rebuilds: every step's drafts against the oracle.
    (On this workload the longest match usually wins anyway -- its repeated
    spans continue alike; test_backoff_structured makes shorter lengths win.)"""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=4096)
    ls = H.Lockstep(cfg, seed=21, B=64, steps=10, finish_frac=0.1, corpus=1 << 16, fused=fused,
                    drafter_over=dict(over, num_backoff=nb), param_over=dict(pover, num_backoff=nb),
                    delta=delta)
    ls.prefill(seed=21)
    for i in range(10):
        ls.step(check_state=True)
    assert ls.dr.get_error() == 0
    ls.close()


def _patterns(rng, V, count):
    return [([int(x) for x in rng.integers(0, V, int(rng.integers(2, 5)))],
             [int(x) for x in rng.integers(0, V, 3)]) for _ in range(count)]


def _structured(rng, V, L, pool):
    """Tokens ending in a pattern P (2-4 ids, from a pool shared by rows and
    docs) whose earlier full occurrences each continue differently, while its
    shorter suffix recurs (after another id) with one continuation: the case
    backoff is for."""
    P, cont = pool[int(rng.integers(0, len(pool)))]
    segs = [P + [int(rng.integers(0, V))] for _ in range(int(rng.integers(1, 4)))]
    for _ in range(int(rng.integers(2, 7))):
        x = int(rng.integers(0, V))
        while x == P[0]:
            x = int(rng.integers(0, V))
        segs.append([x] + P[1:] + cont)
    out = []
    for i in rng.permutation(len(segs)):
        out += [int(x) for x in rng.integers(0, V, int(rng.integers(0, 6)))] + segs[i]
    out += [int(x) for x in rng.integers(0, V, int(rng.integers(0, 6)))] + P
    return np.array(out[-L:], dtype=np.int32)


@pytest.mark.parametrize("nb,delta", [(4, 0), (8, 1 << 14)], ids=["nb4", "nb8+delta"])
def test_backoff_structured(nb, delta):
    """Rows and corpus docs whose longest match is unreliable and whose
    shorter suffix is well supported: shorter lengths win some rows, on both
    paths, and every row matches the oracle."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    V, S, B, C = 64, 256, 64, 1 << 15
    rng = np.random.default_rng(nb + delta)
    kw = dict(k=8, D=16, R=16)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, max_tree_depth=kw["D"],
                       max_occurrences=kw["R"], k=kw["k"], min_token_prob=(1, 2),
                       max_spec_offset=2, corpus_capacity=C, delta_capacity=delta,
                       num_backoff=nb)
    p = O.Params(S=S, V=V, min_prob=(1, 2), offset=2, num_backoff=nb, **kw)
    ring = O.Ring(C, 65536, V)
    pool = _patterns(rng, V, 24)

    def add(m):
        buf = np.zeros((m, S), dtype=np.int32)
        lens = np.zeros(m, dtype=np.int32)
        for i in range(m):
            d = _structured(rng, V, S, pool)
            buf[i, :len(d)] = d
            lens[i] = len(d)
        rows = torch.arange(m, dtype=torch.int32, device="cuda")
        dr.ingest(torch.from_numpy(buf).cuda(), rows, torch.zeros_like(rows), torch.from_numpy(lens).cuda())
        ring.ingest(buf, np.arange(m), np.zeros(m), lens)

    add(48)  # few docs per pattern: the corpus's thresholds reach the shorter suffix too
    dr.build_sa(torch.cuda.Stream())
    assert dr.poll(wait=True)[0] == 1
    X, since = ring.snapshot(), ring.pushed
    add(24)
    tok = np.zeros((B, S), dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        r = _structured(rng, V, S, pool)
        tok[b, :len(r)] = r
        n[b] = len(r)
    out = dr.propose(torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda())
    torch.cuda.synchronize()
    Xd = O.corpus_text(X, ring.delta(since, delta)) if delta else X
    orc = O.propose(p, tok, n, X=Xd, threads=H.THREADS)
    H.compare(out, orc)
    one = O.propose(O.Params(S=S, V=V, min_prob=(1, 2), offset=2, select_by_score=True, **kw),
                    tok, n, X=Xd, threads=H.THREADS)
    changed = (orc.match_info != one.match_info).any(axis=1)
    assert changed.sum() > 0
    assert dr.get_error() == 0
    dr.close()


def _doc_text(docs, V):
    out = []
    for d in docs:
        out += list(d) + [V]
    return np.array(out, dtype=np.int32)


def test_backoff_worked_example():
    """The worked examples of the oracle's pins, through the library: the
    row's length 3 drafts nothing, its length 2 drafts 5 6 at 4/7, a corpus
    doc (3, 1, 2, 5, 6) drafts 5 6 at 1/1 and wins; with five docs the
    corpus's own thresholds pick its length 3, then its length 2."""
    W, O, H = _mods()
    V, S = 20, 64
    row = [3, 1, 2, 7, 8, 3, 1, 2, 9, 8, 3, 1, 2, 11, 8] + [4, 1, 2, 5, 6] * 4 + [3, 1, 2]
    five = [[4, 1, 2, 9]] * 3 + [[3, 1, 2, 7], [3, 1, 2, 8]]
    for docs, nb, want in (([], 4, [2, 1]), ([[3, 1, 2, 5, 6]], 4, [3, 2]), ([[3, 1, 2, 5]], 4, [2, 1]),
                           (five, 2, [3, 2]), (five, 3, [2, 2]), (five, 4, [2, 1])):
        from model_free_suffix_gb300 import SuffixDrafter
        dr = SuffixDrafter(max_batch=2, seq_capacity=S, vocab_size=V, k=4, max_tree_depth=8,
                           max_occurrences=8, min_token_prob=(1, 2), corpus_capacity=1024,
                           num_backoff=nb)
        p = O.Params(S=S, V=V, k=4, D=8, R=8, min_prob=(1, 2), num_backoff=nb)
        X = None
        if docs:
            buf = np.zeros((len(docs), S), dtype=np.int32)
            lens = np.array([len(d) for d in docs], dtype=np.int32)
            for i, d in enumerate(docs):
                buf[i, :len(d)] = d
            rows = torch.arange(len(docs), dtype=torch.int32, device="cuda")
            dr.ingest(torch.from_numpy(buf).cuda(), rows, torch.zeros_like(rows),
                      torch.from_numpy(lens).cuda())
            dr.build_sa(torch.cuda.Stream())
            assert dr.poll(wait=True)[0] == 1
            X = _doc_text(docs, V)
        tok = np.zeros((2, S), dtype=np.int32)
        tok[0, :len(row)] = row
        tok[1, :5] = [1, 2, 1, 2, 1]
        n = np.array([len(row), 5], dtype=np.int32)
        out = dr.propose(torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda())
        torch.cuda.synchronize()
        orc = O.propose(p, tok, n, X=X)
        assert orc.match_info[0].tolist() == want
        H.compare(out, orc, ctx=str(docs))
        assert dr.get_error() == 0
        dr.close()


@pytest.mark.parametrize("V,C,delta,R,k,D,nb,S", [
    (2, 1 << 16, 0, 8, 6, 12, 8, 512),
    (2, 1 << 16, 1 << 15, 16, 8, 16, 5, 512),
    (3, 1 << 14, 1 << 12, 1, 1, 2, 2, 512),
    (5, 1 << 14, 1 << 14, 128, 16, 128, 8, 512),
    (7, 1 << 16, 1 << 14, 64, 64, 32, 8, 8192),
], ids=["wide-interval", "wide+delta", "R1-k1-D2", "R128-D128", "k64-S8192"])
def test_backoff_edges(V, C, delta, R, k, D, nb, S):
    """Few ids, so the interval of the last two tokens holds thousands of hits
    (more than the on-chip length cache: lengths evaluated again, ends chosen
    by the radix selection); the extreme knobs; rows that are empty, one or
    two tokens long, full, or inactive; docs both indexed and in the delta."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    B = 40
    rng = np.random.default_rng(V * 1000 + R)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=D,
                       max_occurrences=R, min_token_prob=(1, 4), max_spec_offset=2,
                       corpus_capacity=C, delta_capacity=delta, num_backoff=nb)
    p = O.Params(S=S, V=V, k=k, D=D, R=R, min_prob=(1, 4), offset=2, num_backoff=nb)
    ring = O.Ring(C, 65536, V)

    def add(m):
        lens = rng.integers(20, 300, size=m).astype(np.int32)
        buf = rng.integers(0, V, size=(m, S)).astype(np.int32)
        rows = torch.arange(m, dtype=torch.int32, device="cuda")
        dr.ingest(torch.from_numpy(buf).cuda(), rows, torch.zeros_like(rows), torch.from_numpy(lens).cuda())
        ring.ingest(buf, np.arange(m), np.zeros(m), lens)

    while ring.live < 3 * C // 4:
        add(32)
    dr.build_sa(torch.cuda.Stream())
    assert dr.poll(wait=True)[0] == 1
    X, since = ring.snapshot(), ring.pushed
    add(24)  # placed after the snapshot: the delta (if any)
    tok = rng.integers(0, V, size=(B, S)).astype(np.int32)
    n = rng.integers(3, S + 1, size=B).astype(np.int32)
    n[:4] = [0, 1, 2, S]
    active = np.ones(B, dtype=np.uint8)
    active[5] = 0
    out = dr.propose(torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda(),
                     active=torch.from_numpy(active).cuda())
    torch.cuda.synchronize()
    Xd = O.corpus_text(X, ring.delta(since, delta)) if delta else X
    H.compare(out, O.propose(p, tok, n, X=Xd, active=active, threads=H.THREADS))
    assert dr.get_error() == 0
    dr.close()


@pytest.mark.parametrize("V,D,nb", [(40, 12, 8), (6, 12, 8), (6, 3, 4), (6, 2, 2), (40, 4, 3), (3, 24, 8)],
                         ids=["2gram-blocks", "2-3gram-blocks", "blocks-D3", "blocks-D2",
                              "2gram-blocks-D4", "V3"])
@pytest.mark.parametrize("gd", [1, 0], ids=["gram-drafts", "no-gram-drafts"])
def test_backoff_gram_blocks(V, D, nb, gd):
    """The corpus side from the snapshot's gram draft blocks: with V = 40 the
    last 2-gram has a block and the 3-gram's interval is walked; with V = 6
    both have blocks and only the 4-gram's interval is walked (D = 3, 2: no
    walk at all).  The same rows with blocks off walk the 2-gram's interval;
    both against the oracle."""
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    B, S, C, R, k = 48, 1024, 1 << 16, 16, 8
    rng = np.random.default_rng(V * 100 + D)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=D,
                       max_occurrences=R, min_token_prob=(1, 3), max_spec_offset=1,
                       corpus_capacity=C, num_backoff=nb, gram_drafts=gd)
    p = O.Params(S=S, V=V, k=k, D=D, R=R, min_prob=(1, 3), offset=1, num_backoff=nb)
    ring = O.Ring(C, 65536, V)
    while ring.live < 3 * C // 4:
        m = 32
        lens = rng.integers(20, 400, size=m).astype(np.int32)
        buf = rng.integers(0, V, size=(m, S)).astype(np.int32)
        # repeated spans, so that longer matches and their continuations agree
        for i in range(m):
            if lens[i] > 60:
                at = int(rng.integers(0, lens[i] - 40))
                buf[i, at:at + 24] = buf[(i + 1) % m, 10:34]
        rows = torch.arange(m, dtype=torch.int32, device="cuda")
        dr.ingest(torch.from_numpy(buf).cuda(), rows, torch.zeros_like(rows), torch.from_numpy(lens).cuda())
        ring.ingest(buf, np.arange(m), np.zeros(m), lens)
    dr.build_sa(torch.cuda.Stream())
    assert dr.poll(wait=True)[0] == 1
    X = ring.snapshot()
    tok = rng.integers(0, V, size=(B, S)).astype(np.int32)
    n = rng.integers(3, S - 16, size=B).astype(np.int32)
    n[:3] = [1, 2, 3]
    for b in range(3, B, 2):  # rows ending in a corpus span
        d = X[int(rng.integers(0, X.shape[0] - 40)):][:32]
        if n[b] >= 32 and (d < V).all():
            tok[b, n[b] - 32:n[b]] = d
    out = dr.propose(torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda())
    torch.cuda.synchronize()
    H.compare(out, O.propose(p, tok, n, X=X, threads=H.THREADS))
    assert dr.get_error() == 0
    dr.close()


def test_backoff_full_serving_size_sampled_rows():
    """The serving workload at its full size (B = 256, S = 4096, 1M-token
    corpus, rebuilds), num_backoff = 8 through the step as the benchmark runs
    it: 48 sampled rows per step against the oracle."""
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=8192)
    ls = H.Lockstep(cfg, seed=3, steps=6, fused=True, drafter_over=dict(num_backoff=8),
                    param_over=dict(num_backoff=8))
    ls.prefill(seed=3)
    rng = np.random.default_rng(3)
    for _ in range(6):
        ls.step(check_rows=np.sort(rng.choice(cfg.B, size=48, replace=False)), check_state=True)
    assert ls.dr.get_error() == 0
    ls.close()
