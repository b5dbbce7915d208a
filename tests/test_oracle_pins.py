"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here calls the CUDA library.  The oracle is checked against
hand-worked examples (tests/golden), an independent brute-force formulation
(tests/bruteforce.py), closed forms and invariants.
"""
import json
import os
import random
from fractions import Fraction

import numpy as np
import pytest

from bruteforce import brute_propose, brute_suffix_array

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _params(orc, case, corpus=False):
    pr = dict(S=1000, V=100, k=8, D=24, R=64, factor=(1, 1), offset=0, min_prob=(1, 10),
              depth_sum_cap=False)
    for key, val in case.get("params", {}).items():
        pr[key] = tuple(val) if isinstance(val, list) else val
    return orc.Params(**pr), pr


@pytest.mark.parametrize("case", GOLDEN["cases"], ids=lambda c: c["name"])
def test_worked_example(orc, case):
    p, pr = _params(orc, case)
    t = case["t"]
    X = case.get("X")
    r = orc.propose_row(p, t, len(t), X=X, active=case.get("active", True))
    exp = case["expect"]
    L = len(exp["drafts"])
    assert r.num_valid == L
    assert r.drafts[:L].tolist() == exp["drafts"]
    assert (r.drafts[L:] == -1).all()
    assert r.match_info.tolist() == [exp["M"], exp["source"]]
    want_score = np.float32(Fraction(*exp["score"]))
    assert np.float32(r.score) == want_score
    for d, (a, b) in enumerate(exp["probs"]):
        assert r.probs[d] == np.float32(Fraction(a, b))
    assert (r.probs[L:] == 0).all()


@pytest.mark.parametrize("case", GOLDEN["suffix_arrays"], ids=lambda c: c["name"])
def test_suffix_array_examples(orc, case):
    assert orc.suffix_array(case["X"]).tolist() == case["SA"]
    assert orc.check_suffix_array(case["X"], case["SA"]) == 0


@pytest.mark.parametrize("case", GOLDEN["updates"], ids=lambda c: c["name"])
def test_update_examples(orc, case):
    row = np.array([case["row"]], dtype=np.int32)
    n = np.array([case["n"]], dtype=np.int32)
    f = orc.update_state(row, n, np.array([case["sampled"]], dtype=np.int32), case["V"])
    assert row[0].tolist() == case["expect_row"]
    assert int(n[0]) == case["expect_n"]
    assert f == case["expect_flags"]


@pytest.mark.parametrize("case", GOLDEN["rings"], ids=lambda c: c["name"])
def test_ring_examples(orc, case):
    docs = case["docs"]
    width = max(1, max(len(d) for d in docs))
    buf = np.full((len(docs), width), -1, dtype=np.int32)
    for i, d in enumerate(docs):
        buf[i, :len(d)] = d
    ring = orc.Ring(case["C"], case["max_docs"], case["V"])
    f = ring.ingest(buf, np.arange(len(docs)), np.zeros(len(docs)), [len(d) for d in docs])
    assert f == case["expect_flags"]
    assert ring.live == case["expect_live"]
    assert ring.snapshot().tolist() == case["expect_snapshot"]


# --------------------------------------------------------------------------
# brute force over every suffix length and every occurrence

def _rand_params(rng):
    k = rng.randint(1, 10)
    D = rng.randint(1, 9)
    factor = rng.choice([(1, 1), (2, 1), (1, 2), (3, 2), (0, 1)])
    offset = rng.choice([0, 0, 1, 2])
    min_prob = rng.choice([(0, 1), (1, 10), (1, 4), (1, 3), (1, 2), (2, 3), (1, 1)])
    return k, D, factor, offset, min_prob


def _compare(orc, t, n, S, V, k, D, R, factor, offset, min_prob, X=None, dsc=False):
    p = orc.Params(S=S, V=V, k=k, D=D, R=R if R is not None else 4096, factor=factor,
                   offset=offset, min_prob=min_prob, depth_sum_cap=dsc)
    r = orc.propose_row(p, np.asarray(t, dtype=np.int32), n, X=X)
    b = brute_propose(t, n, k, D, R, S, factor, offset, min_prob, X=X, Z=V, depth_sum_cap=dsc)
    ctx = dict(t=list(t[:n]), X=None if X is None else list(X), k=k, D=D, R=R, S=S,
               factor=factor, offset=offset, min_prob=min_prob)
    assert r.match_info.tolist() == [b.M, b.source], ctx
    assert r.num_valid == len(b.drafts), ctx
    assert r.drafts[:r.num_valid].tolist() == b.drafts, ctx
    assert (r.drafts[r.num_valid:] == -1).all()
    assert np.float32(r.score) == np.float32(b.score), ctx
    for d, pr in enumerate(b.probs):
        assert r.probs[d] == np.float32(pr), ctx


@pytest.mark.parametrize("seed", range(6))
def test_self_vs_bruteforce_unbounded(orc, seed):
    rng = random.Random(1000 + seed)
    for _ in range(150):
        V = rng.choice([2, 3, 4])
        n = rng.randint(0, 48)
        S = n + rng.choice([0, 1, 2, 5, 40])
        t = [rng.randrange(V) for _ in range(n)]
        k, D, factor, offset, min_prob = _rand_params(rng)
        _compare(orc, t, n, S, V, k, D, None, factor, offset, min_prob,
                 dsc=rng.random() < 0.2)


@pytest.mark.parametrize("seed", range(4))
def test_self_vs_bruteforce_budget(orc, seed):
    rng = random.Random(2000 + seed)
    for _ in range(150):
        V = rng.choice([2, 3])
        n = rng.randint(2, 48)
        S = n + 40
        t = [rng.randrange(V) for _ in range(n)]
        k, D, factor, offset, min_prob = _rand_params(rng)
        R = rng.randint(1, 4)
        _compare(orc, t, n, S, V, k, D, R, factor, offset, min_prob)


def _rand_corpus(rng, V, ndocs, maxlen):
    X = []
    for _ in range(ndocs):
        L = rng.randint(1, maxlen)
        X += [rng.randrange(V) for _ in range(L)] + [V]
    return X


@pytest.mark.parametrize("seed", range(4))
def test_corpus_vs_bruteforce(orc, seed):
    rng = random.Random(3000 + seed)
    for _ in range(120):
        V = rng.choice([2, 3, 4])
        n = rng.randint(0, 24)
        S = n + rng.choice([1, 3, 40])
        t = [rng.randrange(V) for _ in range(n)]
        X = _rand_corpus(rng, V, rng.randint(1, 6), 12)
        k, D, factor, offset, min_prob = _rand_params(rng)
        R = rng.choice([None, None, 1, 2, 3])
        _compare(orc, t, n, S, V, k, D, R, factor, offset, min_prob, X=X)


def test_corpus_match_scan_vs_substrings(orc):
    """Mc and its occurrence set against a naive search over all lengths."""
    rng = random.Random(77)
    from bruteforce import ends_of
    for _ in range(400):
        V = rng.choice([2, 3])
        X = _rand_corpus(rng, V, rng.randint(1, 5), 10)
        n = rng.randint(0, 12)
        t = [rng.randrange(V) for _ in range(n)]
        D = rng.randint(1, 8)
        R = rng.randint(1, 6)
        M, occ = orc.corpus_match(X, V, t, n, D, R)
        best = 0
        ends = []
        if D >= 2 and n >= 2:
            for l in range(min(D, n), 1, -1):
                es = [e for e in ends_of(X, t[n - l:]) if e + 1 < len(X) and X[e + 1] != V]
                if es:
                    best, ends = l, sorted(es, reverse=True)[:R]
                    break
        assert M == best
        assert occ.tolist() == ends


def test_self_match_occurrences_vs_substrings(orc):
    rng = random.Random(78)
    from bruteforce import ends_of
    for _ in range(400):
        V = rng.choice([2, 3])
        n = rng.randint(0, 30)
        t = [rng.randrange(V) for _ in range(n)]
        D = rng.randint(1, 10)
        R = rng.randint(1, 6)
        M, occ = orc.self_match(t, n, D, R)
        best, ends = 0, []
        for l in range(min(D, n - 1), 0, -1):
            es = [e for e in ends_of(t, t[n - l:]) if e <= n - 2]
            if es:
                best, ends = l, sorted(es, reverse=True)[:R]
                break
        assert M == best
        assert occ.tolist() == ends


# --------------------------------------------------------------------------
# closed forms

@pytest.mark.parametrize("p,n,D,k", [(3, 40, 8, 8), (2, 31, 6, 10), (5, 64, 7, 16),
                                     (4, 9, 8, 8), (7, 10, 24, 16), (1, 20, 5, 8)])
def test_periodic_closed_form(orc, p, n, D, k):
    """A period-p text: if n - p >= D then M = D, the draft continues the period,
    and depth d keeps c0 - floor(d / p) survivors (occurrences run off the end
    one period at a time); otherwise M = n - p with one occurrence."""
    base = list(range(10, 10 + p))
    t = [base[i % p] for i in range(n)]
    S = 10 * n
    prm = orc.Params(S=S, V=100, k=k, D=D, R=4096, factor=(100, 1), offset=0, min_prob=(0, 1))
    r = orc.propose_row(prm, t, n)
    if n - p >= D:
        M = D
        # ends j <= n-2 with j = n-1 (mod p) and j >= D-1
        occ = [j for j in range(D - 1, n - 1) if (j - (n - 1)) % p == 0]
        c0 = len(occ)
        L = k
        exp_probs = [Fraction(c0 - d // p, c0) for d in range(L)]
        assert r.match_info.tolist() == [M, 1]
        assert r.num_valid == L
        assert r.drafts.tolist() == [t[(n + d) % p] if False else base[(n + d) % p] for d in range(L)]
        for d in range(L):
            assert r.probs[d] == np.float32(exp_probs[d])
    else:
        M = n - p
        assert r.match_info.tolist() == [M, 1 if M > 0 else 0]
        if M > 0:
            L = min(k, p, S - n - 1)
            assert r.num_valid == L
            assert r.drafts[:L].tolist() == [base[(n + d) % p] for d in range(L)]


def test_all_distinct_and_short(orc):
    prm = orc.Params(S=100, V=1000, k=8, D=24, R=64)
    r = orc.propose_row(prm, list(range(50)), 50)
    assert r.num_valid == 0 and r.match_info.tolist() == [0, 0]
    for n in (0, 1):
        r = orc.propose_row(prm, [3, 3], n)
        assert r.num_valid == 0


def test_no_room_near_capacity(orc):
    t = [1, 2] * 10
    for S, want in ((20, 0), (21, 0), (22, 1), (23, 2)):
        prm = orc.Params(S=S, V=10, k=8, D=24, R=64, factor=(10, 1))
        r = orc.propose_row(prm, t, 20)
        assert r.num_valid == want


# --------------------------------------------------------------------------
# suffix array

def test_suffix_array_vs_python_sort(orc):
    rng = random.Random(5)
    for _ in range(300):
        N = rng.randint(0, 60)
        V = rng.choice([1, 2, 3, 50])
        X = [rng.randrange(V) - (1 if rng.random() < 0.1 else 0) for _ in range(N)]
        sa = orc.suffix_array(X)
        assert sa.tolist() == brute_suffix_array(X)
        assert orc.check_suffix_array(X, sa) == 0


def test_suffix_array_checker_rejects(orc):
    X = [3, 1, 2, 1, 2, 100]
    good = brute_suffix_array(X)
    assert orc.check_suffix_array(X, good) == 0
    bad = list(good)
    bad[1], bad[2] = bad[2], bad[1]
    assert orc.check_suffix_array(X, bad) != 0
    dup = list(good)
    dup[0] = dup[1]
    assert orc.check_suffix_array(X, dup) != 0


def test_suffix_array_large_sorted(orc):
    rng = np.random.default_rng(3)
    X = rng.integers(0, 4, size=20000).astype(np.int32)
    X[rng.integers(0, 20000, size=200)] = 4
    X[-1] = 4
    sa = orc.suffix_array(X)
    assert orc.check_suffix_array(X, sa) == 0


# --------------------------------------------------------------------------
# ring and update

def test_ring_vs_fifo_model(orc):
    """The ring holds the newest docs whose tokens + sentinels fit in C."""
    rng = random.Random(9)
    for _ in range(50):
        C = rng.randint(5, 60)
        max_docs = rng.randint(1, 8)
        ring = orc.Ring(C, max_docs, 50)
        model = []
        for _step in range(20):
            m = rng.randint(0, 4)
            docs = [[rng.randrange(50) for _ in range(rng.randint(0, 15))] for _ in range(m)]
            if m == 0:
                continue
            width = max(1, max(len(d) for d in docs))
            buf = np.full((m, width), -1, dtype=np.int32)
            for i, d in enumerate(docs):
                buf[i, :len(d)] = d
            ring.ingest(buf, np.arange(m), np.zeros(m), [len(d) for d in docs])
            for d in docs:
                if len(d) == 0 or len(d) + 1 > C:
                    continue
                model.append(d)
                while sum(len(x) + 1 for x in model) > C or len(model) > max_docs:
                    model.pop(0)
            snap = []
            for d in model:
                snap += d + [50]
            assert ring.snapshot().tolist() == snap
            assert ring.live == len(snap) <= C
            assert ring.ndocs == len(model)


def test_ring_rejects_bad_args(orc):
    ring = orc.Ring(100, 8, 50)
    buf = np.array([[1, 2, 3, 4]], dtype=np.int32)
    assert ring.ingest(buf, [1], [0], [2]) == orc.ERR_DOC_ARGS        # row out of range
    assert ring.ingest(buf, [0], [3], [2]) == orc.ERR_DOC_ARGS        # past the row
    assert ring.ingest(buf, [0], [-1], [2]) == orc.ERR_DOC_ARGS
    assert ring.ingest(buf, [0], [0], [3], num_tokens=[2]) == orc.ERR_DOC_ARGS
    assert ring.live == 0
    assert ring.ingest(buf, [0], [1], [2], num_tokens=[4]) == 0
    assert ring.snapshot().tolist() == [2, 3, 50]


def test_update_batch(orc):
    rng = np.random.default_rng(1)
    B, S, T, V = 8, 32, 5, 20
    tok = np.full((B, S), -1, dtype=np.int32)
    n = rng.integers(0, S + 1, size=B).astype(np.int32)
    for b in range(B):
        tok[b, :n[b]] = rng.integers(0, V, size=n[b])
    sampled = rng.integers(-1, V, size=(B, T)).astype(np.int32)
    tok0, n0 = tok.copy(), n.copy()
    orc.update_state(tok, n, sampled, V)
    for b in range(B):
        c = 0
        while c < T and 0 <= sampled[b, c] < V:
            c += 1
        assert n[b] == min(S, n0[b] + c)
        assert tok[b, :n0[b]].tolist() == tok0[b, :n0[b]].tolist()
        assert tok[b, n0[b]:n[b]].tolist() == sampled[b, :n[b] - n0[b]].tolist()
        assert (tok[b, n[b]:] == tok0[b, n[b]:]).all()


def test_invariants_random_rows(orc):
    """num_valid <= cap, -1 padding, non-increasing probs >= min_prob, score = sum."""
    rng = np.random.default_rng(11)
    for _ in range(200):
        V = int(rng.integers(2, 6))
        n = int(rng.integers(0, 80))
        t = rng.integers(0, V, size=n).astype(np.int32)
        k = int(rng.integers(1, 12))
        prm = orc.Params(S=n + 30, V=V, k=k, D=int(rng.integers(1, 12)), R=int(rng.integers(1, 9)),
                         min_prob=(1, 5))
        r = orc.propose_row(prm, t, n)
        L = r.num_valid
        assert 0 <= L <= k
        assert (r.drafts[L:] == -1).all() and (r.drafts[:L] >= 0).all()
        pr = r.probs[:L]
        assert (np.diff(pr) <= 0).all()
        assert (pr >= np.float32(0.2) - 1e-7).all()
        assert abs(float(r.score) - float(pr.astype(np.float64).sum())) < 1e-5
        if L:
            M = r.match_info[0]
            W = list(t[n - M:]) + r.drafts[:L].tolist()
            s = "," + ",".join(map(str, t.tolist())) + ","
            assert ("," + ",".join(map(str, W)) + ",") in s


def test_vote_is_a_prefix_whatever_the_cap(orc):
    """The vote at a depth never depends on where it will stop: with the cap
    set by the offset alone (factor 0), a smaller cap gives a prefix of a
    larger cap's draft with the same probabilities, and num_valid =
    min(cap, the larger cap's num_valid).  (This is what lets a precomputed
    depth-k vote of a gram serve every row whose candidate it is, cut at the
    row's own cap.)"""
    rng = np.random.default_rng(23)
    for _ in range(150):
        V = int(rng.integers(2, 6))
        n = int(rng.integers(2, 60))
        t = rng.integers(0, V, size=n).astype(np.int32)
        X = None
        if rng.random() < 0.6:
            X = rng.integers(0, V + 1, size=int(rng.integers(10, 120))).astype(np.int32)
            X[-1] = V
        k = int(rng.integers(2, 12))
        kw = dict(S=n + 40, V=V, k=k, D=int(rng.integers(2, 10)), R=int(rng.integers(1, 9)),
                  factor=(0, 1), min_prob=(1, int(rng.integers(2, 6))))
        full = orc.propose_row(orc.Params(offset=k, **kw), t, n, X=X)
        for cap in range(k + 1):
            r = orc.propose_row(orc.Params(offset=cap, **kw), t, n, X=X)
            L = r.num_valid
            assert L == min(cap, full.num_valid), (cap, L, full.num_valid)
            assert r.drafts[:L].tolist() == full.drafts[:L].tolist()
            assert np.array_equal(r.probs[:L].view(np.uint32), full.probs[:L].view(np.uint32))
            if L:
                assert r.match_info.tolist() == full.match_info.tolist()


# --------------------------------------------------------------------------
# delta (docs placed after the snapshot was taken, not yet indexed)

def _ingest_docs(ring, docs):
    width = max(1, max(len(d) for d in docs))
    buf = np.full((len(docs), width), -1, dtype=np.int32)
    for i, d in enumerate(docs):
        buf[i, :len(d)] = d
    ring.ingest(buf, np.arange(len(docs)), np.zeros(len(docs)), [len(d) for d in docs])


def test_delta_vs_sequence_model(orc):
    """The delta of a snapshot taken after `since` placements is the live docs
    placed after it, oldest first, each followed by the sentinel, cut at cap
    (checked against a list model that numbers every placed doc)."""
    rng = random.Random(21)
    for _ in range(60):
        C = rng.randint(5, 80)
        max_docs = rng.randint(1, 9)
        ring = orc.Ring(C, max_docs, 50)
        model = []   # (sequence number, tokens) of the live docs, oldest first
        placed = 0
        marks = [0]  # pushed counts at which snapshots were "taken"
        for _step in range(25):
            m = rng.randint(1, 4)
            docs = [[rng.randrange(50) for _ in range(rng.randint(0, 15))] for _ in range(m)]
            _ingest_docs(ring, docs)
            for d in docs:
                if len(d) == 0 or len(d) + 1 > C:
                    continue
                model.append((placed, d))
                placed += 1
                while sum(len(x) + 1 for _, x in model) > C or len(model) > max_docs:
                    model.pop(0)
            assert ring.pushed == placed
            if rng.random() < 0.3:
                marks.append(placed)
            for since in marks[-3:] + [placed]:
                for cap in (0, 1, rng.randint(1, 40), 10 ** 6):
                    want = []
                    for sq, d in model:
                        if sq >= since:
                            want += d + [50]
                    assert ring.delta(since, cap).tolist() == want[:cap], (since, cap)


def test_delta_completes_the_snapshot(orc):
    """While nothing has been evicted since a snapshot, that snapshot followed
    by its full delta is the snapshot the ring would give now; a smaller cap
    gives a prefix of the full delta."""
    rng = random.Random(5)
    for _ in range(40):
        ring = orc.Ring(10 ** 6, 10 ** 4, 30)
        _ingest_docs(ring, [[rng.randrange(30) for _ in range(rng.randint(1, 12))]
                            for _ in range(rng.randint(1, 6))])
        X0, since = ring.snapshot(), ring.pushed
        _ingest_docs(ring, [[rng.randrange(30) for _ in range(rng.randint(0, 12))]
                            for _ in range(rng.randint(1, 6))])
        full = ring.delta(since, 10 ** 9)
        assert np.concatenate([X0, full]).tolist() == ring.snapshot().tolist()
        cap = rng.randint(0, full.shape[0] + 2)
        assert ring.delta(since, cap).tolist() == full[:cap].tolist()
        # a ring never snapshotted: every live doc is in the delta
        assert ring.delta(0, 10 ** 9).tolist() == ring.snapshot().tolist()


def test_delta_proposals_equal_the_rebuilt_index(orc):
    """Matching against snapshot + delta gives the proposals that matching
    against a snapshot rebuilt over the same docs gives (no evictions)."""
    rng = np.random.default_rng(17)
    V, S = 12, 64
    p = orc.Params(S=S, V=V, k=6, D=8, R=8, min_prob=(1, 10))
    for trial in range(20):
        ring = orc.Ring(10 ** 6, 10 ** 4, V)
        docs = [list(rng.integers(0, V, rng.integers(2, 20))) for _ in range(6)]
        _ingest_docs(ring, docs[:3])
        X0, since = ring.snapshot(), ring.pushed
        _ingest_docs(ring, docs[3:])
        Xd = orc.corpus_text(X0, ring.delta(since, 10 ** 9))
        tok = rng.integers(0, V, (8, S)).astype(np.int32)
        n = rng.integers(2, S - 8, 8).astype(np.int32)
        a = orc.propose(p, tok, n, X=Xd)
        b = orc.propose(p, tok, n, X=ring.snapshot())
        assert np.array_equal(a.drafts, b.drafts) and np.array_equal(a.match_info, b.match_info)
        assert np.array_equal(a.num_valid, b.num_valid) and np.array_equal(a.score, b.score)


# --------------------------------------------------------------------------
# Model Runner V2 drafts ("Suffix Decoding" (vLLM docs), Model Runner V2: the
# draft always has k tokens; slots without a match hold the last sampled token;
# max_spec_factor and min_token_prob are not used)

def _row(orc, p, t, X=None):
    S = p.S
    tok = np.zeros((1, S), dtype=np.int32)
    tok[0, :len(t)] = t
    return orc.propose(p, tok, np.array([len(t)], dtype=np.int32), X=X)


def test_fixed_length_worked_examples(orc):
    # row 5 6 7 5 6: the tail (5, 6) occurs once before, at 0..1, followed by 7 5 6
    # and then nothing: the vote gives 7 5 6 (each 1/1), the fourth slot is the last
    # token 6.  The default rule stops at floor(1.0 * 2) + 0 = 2 tokens instead.
    p = orc.Params(S=16, V=10, k=4, D=8, R=4, fixed_length=True)
    r = _row(orc, p, [5, 6, 7, 5, 6])
    assert r.drafts[0].tolist() == [7, 5, 6, 6] and r.num_valid[0] == 4
    assert r.probs[0].tolist() == [1.0, 1.0, 1.0, 0.0] and float(r.score[0]) == 3.0
    assert r.match_info[0].tolist() == [2, 1]
    r = _row(orc, orc.Params(S=16, V=10, k=4, D=8, R=4), [5, 6, 7, 5, 6])
    assert r.drafts[0].tolist() == [7, 5, -1, -1] and r.num_valid[0] == 2
    # no earlier 3 in 1 2 3: every slot is the last token, probability 0
    r = _row(orc, p, [1, 2, 3])
    assert r.drafts[0].tolist() == [3, 3, 3, 3] and r.num_valid[0] == 4
    assert r.probs[0].tolist() == [0.0] * 4 and float(r.score[0]) == 0.0
    assert r.match_info[0].tolist() == [0, 0]
    # 9 1 9 2 9 3 9: three ends of length 1 (at 4, 2, 0) continue with 3, 2, 1; the
    # tie goes to 1 (count 1 of 3), whose end (0) continues 9 2 9.  min_token_prob
    # 0.5 would stop the default rule before the first token; here it is unused.
    p = orc.Params(S=16, V=10, k=4, D=8, R=4, min_prob=(1, 2), fixed_length=True)
    r = _row(orc, p, [9, 1, 9, 2, 9, 3, 9])
    assert r.drafts[0].tolist() == [1, 9, 2, 9] and r.num_valid[0] == 4
    assert np.allclose(r.probs[0], [1 / 3] * 4) and abs(float(r.score[0]) - 4 / 3) < 1e-6
    r = _row(orc, orc.Params(S=16, V=10, k=4, D=8, R=4, min_prob=(1, 2), factor=(100, 1)),
             [9, 1, 9, 2, 9, 3, 9])
    assert r.num_valid[0] == 0 and r.drafts[0].tolist() == [-1] * 4


def test_fixed_length_is_the_unstopped_vote_then_the_last_token(orc):
    """On random rows (and a corpus): the voted part of a fixed-length draft is the
    default draft with no probability floor and no factor cap; the rest is the
    row's last token; inactive or empty rows stay empty."""
    rng = np.random.default_rng(8)
    V, S, k = 7, 96, 6
    X = np.concatenate([np.append(rng.integers(0, V, rng.integers(5, 40)), V) for _ in range(12)])
    for trial in range(40):
        B = 6
        tok = rng.integers(0, V, (B, S)).astype(np.int32)
        n = rng.integers(0, S - 2, B).astype(np.int32)
        n[0] = 0
        act = np.ones(B, np.uint8)
        act[1] = 0
        Xc = X if trial % 2 else None
        f = orc.propose(orc.Params(S=S, V=V, k=k, D=12, R=8, fixed_length=True), tok, n, X=Xc,
                        active=act)
        d = orc.propose(orc.Params(S=S, V=V, k=k, D=12, R=8, min_prob=(0, 1), factor=(10 ** 6, 1)),
                        tok, n, X=Xc, active=act)
        for b in range(B):
            if not act[b] or n[b] == 0:
                assert f.num_valid[b] == 0 and (f.drafts[b] == -1).all()
                continue
            m = d.num_valid[b]
            assert f.num_valid[b] == k
            assert f.drafts[b, :m].tolist() == d.drafts[b, :m].tolist()
            assert (f.drafts[b, m:] == tok[b, n[b] - 1]).all()
            assert np.array_equal(f.probs[b, :m], d.probs[b, :m]) and (f.probs[b, m:] == 0).all()
            assert f.score[b] == d.score[b] and np.array_equal(f.match_info[b], d.match_info[b])


# --------------------------------------------------------------------------
# score-ranked selection ("SuffixGPU" (PyPI), How it works, step 3: the local
# and global winners compete by the same score)

def _doc_text(docs, V):
    out = []
    for d in docs:
        out += list(d) + [V]
    return np.array(out, dtype=np.int32)


def test_select_by_score_worked_examples(orc):
    V = 20
    row = [1, 2, 9, 8, 7, 1, 2, 9, 8, 7, 5, 1, 2]
    # the row: (1, 2) occurs at 0..1 and 5..6 (length 2 each, 5 before the tail
    # breaks the third token), both followed by 9 8: two tokens of 2/2, score 2.
    # the corpus: (5, 1, 2) three times, followed by 3, 4 and 6: length 3, one
    # token 3 of 1/3 (the tie goes to the smallest id), then the sentinel.
    X = _doc_text([[5, 1, 2, 3], [5, 1, 2, 4], [5, 1, 2, 6]], V)
    base = dict(S=32, V=V, k=4, D=8, R=4)
    r = _row(orc, orc.Params(**base), row, X=X)          # the longer match wins
    assert r.match_info[0].tolist() == [3, 2] and r.drafts[0].tolist() == [3, -1, -1, -1]
    assert abs(float(r.score[0]) - 1 / 3) < 1e-7
    r = _row(orc, orc.Params(**base, select_by_score=True), row, X=X)  # the better score wins
    assert r.match_info[0].tolist() == [2, 1] and r.drafts[0].tolist() == [9, 8, -1, -1]
    assert r.probs[0].tolist() == [1.0, 1.0, 0.0, 0.0] and float(r.score[0]) == 2.0
    # equal scores: with max_spec_factor 1/2 each side emits one token of 1/1
    # (the corpus holds (5, 1, 2) once); the longer match, the corpus's, wins
    X1 = _doc_text([[5, 1, 2, 3]], V)
    r = _row(orc, orc.Params(**base, factor=(1, 2), select_by_score=True), row, X=X1)
    assert r.match_info[0].tolist() == [3, 2] and r.drafts[0].tolist() == [3, -1, -1, -1]
    assert float(r.score[0]) == 1.0


def test_select_by_score_picks_the_better_of_the_two(orc):
    """Where the longer match is the corpus's, its draft is the default rule's
    and the row's own candidate is the draft without a corpus: the score rule
    returns the better of those two (ties: the longer match)."""
    rng = np.random.default_rng(31)
    V, S, k = 6, 80, 5
    checked = 0
    for trial in range(60):
        X = _doc_text([rng.integers(0, V, rng.integers(4, 30)) for _ in range(15)], V)
        B = 8
        tok = rng.integers(0, V, (B, S)).astype(np.int32)
        n = rng.integers(4, S - 2, B).astype(np.int32)
        kw = dict(S=S, V=V, k=k, D=10, R=6, min_prob=(1, 5))
        sc = orc.propose(orc.Params(**kw, select_by_score=True), tok, n, X=X)
        ln = orc.propose(orc.Params(**kw), tok, n, X=X)
        own = orc.propose(orc.Params(**kw), tok, n, X=None)
        for b in range(B):
            if ln.match_info[b, 1] != 2 or own.match_info[b, 1] != 1:
                continue
            checked += 1
            s_c, s_s = float(ln.score[b]), float(own.score[b])
            win = ln if s_c >= s_s else own  # (equal: the longer match, the corpus's)
            assert sc.drafts[b].tolist() == win.drafts[b].tolist(), (trial, b)
            assert sc.match_info[b].tolist() == win.match_info[b].tolist()
            assert sc.score[b] == win.score[b] and np.array_equal(sc.probs[b], win.probs[b])
    assert checked > 20


def test_backoff_lengths_worked_examples(orc):
    """[PYPI] How it works, step 1: for support threshold t the candidate is the
    largest length occurring at least t times, the t-th largest match_back
    value; thresholds 1..nb name the distinct values among the nb largest."""
    L = [3, 1, 3, 2, 0, 5, 2]  # sorted: 5 3 3 2 2 1 0
    assert orc.backoff_lengths(L, 1, 1) == [(5, 1)]
    assert orc.backoff_lengths(L, 1, 2) == [(5, 1), (3, 3)]
    assert orc.backoff_lengths(L, 1, 3) == [(5, 1), (3, 3)]           # t = 3 is still 3
    assert orc.backoff_lengths(L, 1, 4) == [(5, 1), (3, 3), (2, 5)]
    assert orc.backoff_lengths(L, 1, 8) == [(5, 1), (3, 3), (2, 5), (1, 6)]  # no 0: not a match
    assert orc.backoff_lengths(L, 2, 8) == [(5, 1), (3, 3), (2, 5)]   # the corpus needs >= 2
    assert orc.backoff_lengths([0, 0, 1], 2, 8) == []
    assert orc.backoff_lengths([], 1, 4) == []


def test_backoff_lengths_are_the_t_th_largest(orc):
    """The same lengths read off a descending sort: entry t - 1 for t <= nb."""
    rng = np.random.default_rng(4)
    for _ in range(200):
        L = rng.integers(0, 9, rng.integers(0, 40))
        nb, minlen = int(rng.integers(1, 10)), int(rng.integers(1, 3))
        srt = sorted([int(x) for x in L if x >= minlen], reverse=True)
        want = []
        for t in range(1, nb + 1):
            if t <= len(srt) and (not want or want[-1][0] != srt[t - 1]):
                want.append((srt[t - 1], sum(1 for x in srt if x >= srt[t - 1])))
        assert orc.backoff_lengths(L, minlen, nb) == want


def test_backoff_worked_examples(orc):
    V = 20
    # Ends of the row's last token 2 (before the tail itself): 2, 7, 12 match
    # (3, 1, 2), length 3, continued by 7, 9, 11; 17, 22, 27, 32 match (1, 2)
    # only, length 2, each continued by 5 6.
    row = [3, 1, 2, 7, 8, 3, 1, 2, 9, 8, 3, 1, 2, 11, 8] + [4, 1, 2, 5, 6] * 4 + [3, 1, 2]
    base = dict(S=64, V=V, k=4, D=8, R=8, min_prob=(1, 2))
    # the longest match alone: three ends that disagree, 1/3 < 1/2 stops the vote
    for nb in (1, 2, 3):
        r = _row(orc, orc.Params(**base, num_backoff=nb), row)
        assert r.match_info[0].tolist() == [3, 1] and r.drafts[0].tolist() == [-1] * 4
        assert int(r.num_valid[0]) == 0 and float(r.score[0]) == 0.0
    # threshold 4 reaches length 2: all seven ends vote, 5 (4/7) then 6 (4/7),
    # capped at factor 1 x 2 tokens; score 8/7 beats the empty draft
    r = _row(orc, orc.Params(**base, num_backoff=4), row)
    assert r.match_info[0].tolist() == [2, 1] and r.drafts[0].tolist() == [5, 6, -1, -1]
    assert r.probs[0].tolist() == [np.float32(4 / 7)] * 2 + [0.0, 0.0]
    assert abs(float(r.score[0]) - 8 / 7) < 1e-6 and int(r.num_valid[0]) == 2
    # a corpus doc holding (3, 1, 2, 5, 6): corpus length 3, one end, 5 and 6
    # at 1/1 (then the sentinel): score 2 > 8/7, the corpus wins
    r = _row(orc, orc.Params(**base, num_backoff=4), row, X=_doc_text([[3, 1, 2, 5, 6]], V))
    assert r.match_info[0].tolist() == [3, 2] and r.drafts[0].tolist() == [5, 6, -1, -1]
    assert r.probs[0].tolist() == [1.0, 1.0, 0.0, 0.0] and float(r.score[0]) == 2.0
    # (3, 1, 2, 5): one token at 1/1, score 1 < 8/7: the row's length 2 wins
    # although the corpus match is longer
    r = _row(orc, orc.Params(**base, num_backoff=4), row, X=_doc_text([[3, 1, 2, 5]], V))
    assert r.match_info[0].tolist() == [2, 1] and r.drafts[0].tolist() == [5, 6, -1, -1]
    # the corpus's own backoff: (4, 1, 2, 9) x3 and (3, 1, 2, 7), (3, 1, 2, 8):
    # length 3 has two ends (thresholds 1, 2): 7 at 1/2 (the tie goes to the
    # smaller id), then the sentinel, score 1/2; threshold 3 reaches length 2:
    # five ends, 9 at 3/5, then the sentinel, score 3/5.  The row's length 3
    # covers thresholds 1..3 and drafts nothing, its length 2 needs 4.
    X = _doc_text([[4, 1, 2, 9]] * 3 + [[3, 1, 2, 7], [3, 1, 2, 8]], V)
    r = _row(orc, orc.Params(**base, num_backoff=2), row, X=X)
    assert r.match_info[0].tolist() == [3, 2] and r.drafts[0].tolist() == [7, -1, -1, -1]
    assert r.probs[0].tolist() == [0.5, 0.0, 0.0, 0.0] and float(r.score[0]) == 0.5
    r = _row(orc, orc.Params(**base, num_backoff=3), row, X=X)
    assert r.match_info[0].tolist() == [2, 2] and r.drafts[0].tolist() == [9, -1, -1, -1]
    assert abs(float(r.score[0]) - 3 / 5) < 1e-6
    r = _row(orc, orc.Params(**base, num_backoff=4), row, X=X)  # the row's 8/7 wins
    assert r.match_info[0].tolist() == [2, 1] and r.drafts[0].tolist() == [5, 6, -1, -1]


def test_backoff_reduces_to_score_selection(orc):
    """A row whose ends all match the same length has one candidate per path
    whatever num_backoff is: the result is score-ranked selection's.  The row
    repeats a unit of distinct ids and D is at most the unit's length, so
    every earlier end of its last id matches D tokens; each corpus doc is the
    unit followed by ids the unit does not hold."""
    rng = np.random.default_rng(12)
    V, S = 12, 96
    for trial in range(40):
        u = int(rng.integers(3, 7))
        unit = list(rng.permutation(6)[:u])
        row = unit * int(rng.integers(2, 8))
        D = int(rng.integers(2, u + 1))
        X = _doc_text([unit + list(rng.integers(6, V, rng.integers(0, 5))) for _ in range(4)], V)
        assert len(set(l for l in _self_lengths(row, D) if l > 0)) == 1
        assert len(set(l for l in _corpus_lengths(X.tolist(), row, D, V) if l >= 2)) <= 1
        kw = dict(S=S, V=V, k=6, D=D, R=int(rng.integers(1, 9)), offset=int(rng.integers(0, 3)))
        one = _row(orc, orc.Params(**kw, select_by_score=True), row, X=X)
        for nb in (2, 5, 9):
            r = _row(orc, orc.Params(**kw, num_backoff=nb), row, X=X)
            assert r.match_info.tolist() == one.match_info.tolist(), trial
            assert r.drafts.tolist() == one.drafts.tolist() and r.score[0] == one.score[0]
            assert r.probs.tolist() == one.probs.tolist()


def _self_lengths(t, D):
    n = len(t)
    out = []
    for j in range(n - 1):
        l = 0
        while l < min(D, j + 1) and t[j - l] == t[n - 1 - l]:
            l += 1
        out.append(l)
    return out


def _corpus_lengths(X, t, D, Z):
    n = len(t)
    out = []
    for e in range(len(X) - 1):
        l = 0
        if X[e + 1] != Z:
            while l < min(D, n, e + 1) and X[e - l] == t[n - 1 - l]:
                l += 1
        out.append(l)
    return out


def test_backoff_never_scores_below_fewer_candidates(orc):
    """Thresholds 1..nb name a superset of those of 1..nb-1, and the best score
    over a superset is no lower: the winner's score never drops as nb grows,
    and nb = 2 never scores below score-ranked selection over the longest
    matches.  The winner's length is one of its path's candidate lengths."""
    rng = np.random.default_rng(23)
    V, S, B = 3, 72, 8  # few ids and short docs: continuations often run out
    seen_shorter = 0
    for trial in range(25):
        X = _doc_text([rng.integers(0, V, rng.integers(3, 8)) for _ in range(10)], V)
        tok = rng.integers(0, V, (B, S)).astype(np.int32)
        n = rng.integers(3, S - 2, B).astype(np.int32)
        kw = dict(S=S, V=V, k=8, D=9, R=6, offset=1, min_prob=(1, 2))
        prev = orc.propose(orc.Params(**kw, select_by_score=True), tok, n, X=X)
        for nb in (2, 3, 5, 8):
            cur = orc.propose(orc.Params(**kw, num_backoff=nb), tok, n, X=X)
            for b in range(B):
                assert cur.score[b] >= prev.score[b], (trial, nb, b)
                M, src = cur.match_info[b].tolist()
                t = tok[b, :n[b]].tolist()
                own = orc.backoff_lengths(_self_lengths(t, 9), 1, nb)
                other = orc.backoff_lengths(_corpus_lengths(X.tolist(), t, 9, V), 2, nb)
                if M == 0:
                    assert own == [] and other == []
                    continue
                cands = [l for l, _ in (own if src == 1 else other)]
                assert M in cands, (trial, nb, b)
                seen_shorter += int(M != cands[0])
            prev = cur
    assert seen_shorter > 10  # shorter lengths do win


def test_backoff_matches_substring_count_brute_force(orc):
    """The oracle's backoff (per-end match lengths, their t-th largest values)
    against a literal reading of the pages (for each threshold t the largest
    length whose string occurs at least t times, by counting substring
    occurrences), on tiny random rows and corpora."""
    from bruteforce import brute_backoff
    rng = np.random.default_rng(77)
    checked = shorter = 0
    for trial in range(300):
        V = int(rng.integers(2, 5))
        n = int(rng.integers(0, 28))
        t = [int(x) for x in rng.integers(0, V, n)]
        X = None
        if rng.random() < 0.7:
            X = _doc_text([rng.integers(0, V, rng.integers(1, 9)) for _ in range(int(rng.integers(1, 5)))], V)
        kw = dict(S=40, V=V, k=int(rng.integers(1, 6)), D=int(rng.integers(1, 8)),
                  R=int(rng.integers(1, 6)), factor=(int(rng.integers(1, 3)), 1),
                  offset=int(rng.integers(0, 3)), min_prob=(int(rng.integers(1, 3)), 4))
        nb = int(rng.integers(2, 9))
        r = _row(orc, orc.Params(**kw, num_backoff=nb), t, X=X) if n > 0 else None
        b = brute_backoff(t, n, kw["k"], kw["D"], kw["R"], kw["S"], kw["factor"], kw["offset"],
                          kw["min_prob"], nb, X=None if X is None else X.tolist(), Z=V)
        if r is None:
            continue
        L = len(b.drafts)
        assert r.match_info[0].tolist() == [b.M, b.source], (trial, t, X)
        assert int(r.num_valid[0]) == L and r.drafts[0, :L].tolist() == b.drafts
        assert np.float32(r.score[0]) == np.float32(b.score)
        assert [np.float32(x) for x in r.probs[0, :L]] == [np.float32(x) for x in b.probs]
        checked += 1
        one = _row(orc, orc.Params(**kw, select_by_score=True), t, X=X)
        shorter += int(one.match_info[0].tolist() != [b.M, b.source])
    assert checked > 200 and shorter > 10
