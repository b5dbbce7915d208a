"""CUDA library vs CPU oracle, element by element, on the same seeded inputs.

Drafts, valid counts, match info, token buffers and suffix arrays must be
bit-exact; scores and per-slot probabilities bit-equal as float32 words (both
sides round the same integer quotient over c0 to float32, which lands on the
same float: tests/test_arith.py).
"""
import dataclasses
import json
import os
import random

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from model_free_suffix_gb300 import build
    build.build()
    from oracle import oracle as O
    O.build()


def _mods():
    from model_free_suffix_gb300 import SuffixDrafter, workload as W
    from oracle import oracle as O
    import harness as H
    return SuffixDrafter, W, O, H


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a)).to(dtype).cuda()


def _ingest_text(dr, X, V, S):
    """Feed a sentinel-separated text into the ring, doc by doc."""
    from model_free_suffix_gb300 import workload as W
    docs, lens = W.docs_from_text(np.asarray(X, dtype=np.int32), V)
    assert docs.shape[1] <= S
    for s in range(0, docs.shape[0], 2048):
        d = docs[s:s + 2048]
        m = d.shape[0]
        buf = np.full((m, S), -1, dtype=np.int32)
        buf[:, :d.shape[1]] = d
        dr.ingest(_dev(buf), _dev(np.arange(m)), _dev(np.zeros(m)), _dev(lens[s:s + 2048]))


# ---------------------------------------------------------------------------
# Every parameter a worked example may set, and the drafter argument it becomes.
# A key missing here fails the test instead of being dropped silently.
GOLDEN_KNOBS = {"S": "seq_capacity", "V": "vocab_size", "k": "k", "D": "max_tree_depth",
                "R": "max_occurrences", "factor": "max_spec_factor", "offset": "max_spec_offset",
                "min_prob": "min_token_prob", "depth_sum_cap": "depth_sum_cap",
                "num_backoff": "num_backoff"}


@pytest.mark.parametrize("case", GOLDEN["cases"], ids=lambda c: c["name"])
def test_golden_case(case):
    SuffixDrafter, W, O, H = _mods()
    pr = dict(S=1000, V=100, k=8, D=24, R=64, factor=(1, 1), offset=0, min_prob=(1, 10),
              depth_sum_cap=False, num_backoff=1)
    unknown = set(case.get("params", {})) - set(GOLDEN_KNOBS)
    assert not unknown, "golden parameters with no drafter argument: %s" % sorted(unknown)
    for key, val in case.get("params", {}).items():
        pr[key] = tuple(val) if isinstance(val, list) else val
    if pr["S"] % 4:
        pytest.skip("row capacity must be a multiple of 4 on the GPU (oracle-only case)")
    X = case.get("X")
    dr = SuffixDrafter(max_batch=1, corpus_capacity=64 if X else 0,
                       **{GOLDEN_KNOBS[key]: val for key, val in pr.items()})
    t = case["t"]
    row = np.full((1, pr["S"]), -1, dtype=np.int32)
    row[0, :len(t)] = t
    if X:
        _ingest_text(dr, X, pr["V"], pr["S"])
        dr.build_sa(torch.cuda.Stream())
        assert dr.poll(wait=True)[0] == 1
    act = _dev([1 if case.get("active", True) else 0], torch.uint8)
    out = dr.propose(_dev(row), _dev([len(t)]), active=act)
    exp = case["expect"]
    L = len(exp["drafts"])
    d = out.drafts.cpu().numpy()[0]
    assert int(out.num_valid[0]) == L
    assert d[:L].tolist() == exp["drafts"] and (d[L:] == -1).all()
    assert out.match_info.cpu().numpy()[0].tolist() == [exp["M"], exp["source"]]
    from fractions import Fraction
    assert float(out.score[0]) == float(np.float32(Fraction(*exp["score"])))
    for i, (a, b) in enumerate(exp["probs"]):
        assert float(out.probs[0, i]) == float(np.float32(Fraction(a, b)))
    dr.close()


@pytest.mark.parametrize("case", GOLDEN["suffix_arrays"], ids=lambda c: c["name"])
def test_golden_suffix_array(case):
    SuffixDrafter, W, O, H = _mods()
    dr = SuffixDrafter(max_batch=1, seq_capacity=8, vocab_size=200, corpus_capacity=64)
    sa = dr.suffix_array(_dev(case["X"]))
    assert sa.cpu().numpy().tolist() == case["SA"]
    dr.close()


# ---------------------------------------------------------------------------
SELF_GRID = [
    # (V, S, k, D, R, factor, offset, min_prob, depth_sum_cap, self_warps)
    (2, 256, 8, 24, 64, (1, 1), 0, (1, 10), False, 0),
    (3, 256, 16, 5, 3, (2, 1), 1, (1, 4), False, 0),
    (2, 1024, 64, 128, 128, (4, 1), 0, (0, 1), False, 0),
    (5, 1024, 1, 1, 1, (1, 1), 0, (1, 10), False, 0),
    (3, 512, 12, 2, 7, (3, 2), 2, (1, 3), True, 0),
    (50, 2048, 32, 32, 64, (1, 1), 0, (1, 10), False, 3),
    (4, 4096, 16, 24, 64, (1, 1), 0, (1, 2), False, 16),
    (2, 128, 8, 3, 2, (1, 1), 0, (2, 3), False, 1),
]


@pytest.mark.parametrize("mode", [1, 2], ids=["one-launch", "two-launch"])
@pytest.mark.parametrize("grid", SELF_GRID, ids=lambda g: "V%d_S%d_k%d_D%d_R%d" % g[:5])
def test_fuzz_self(grid, mode):
    SuffixDrafter, W, O, H = _mods()
    V, S, k, D, R, f, off, mp, dsc, sw = grid
    rng = np.random.default_rng(hash(grid) & 0xffff)
    B = 96
    tok = np.full((B, S), -1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        kind = b % 6
        nb = {0: rng.integers(0, S + 1), 1: rng.integers(0, 4), 2: S - rng.integers(0, 3),
              3: rng.integers(S // 2, S + 1), 4: rng.integers(1, 200), 5: rng.integers(0, S + 1)}[kind]
        nb = int(min(max(nb, 0), S))
        if kind == 5:  # periodic rows: long matches, many occurrences
            p = int(rng.integers(1, 9))
            base = rng.integers(0, V, size=p)
            tok[b, :nb] = base[np.arange(nb) % p]
        else:
            tok[b, :nb] = rng.integers(0, V, size=nb)
        n[b] = nb
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=D,
                       max_occurrences=R, max_spec_factor=f, max_spec_offset=off, min_token_prob=mp,
                       depth_sum_cap=dsc, self_warps=sw, propose_mode=mode)
    active = (rng.random(B) < 0.9).astype(np.uint8)
    out = dr.propose(_dev(tok), _dev(n), active=_dev(active, torch.uint8))
    p = O.Params(S=S, V=V, k=k, D=D, R=R, factor=f, offset=off, min_prob=mp, depth_sum_cap=dsc)
    orc = O.propose(p, tok, n, active=active, threads=H.THREADS)
    H.compare(out, orc, ctx=str(grid))
    dr.close()


CORPUS_GRID = [
    # (V, D, R, k, cand_cap, n_docs, doc_len)
    (2, 24, 64, 8, 2048, 40, 30),
    (3, 4, 5, 6, 64, 60, 20),
    (3, 3, 8, 8, 64, 30, 25),
    (2, 2, 3, 4, 64, 50, 10),
    (4, 8, 1, 16, 128, 200, 40),
    (5, 24, 128, 32, 256, 300, 60),
]


# snapshot indexes: (records, n-gram table); drafts must be the same for each
INDEX_MODES = [(1, 1, 1), (1, 0, 1), (0, 0, 1), (1, 1, 2), (0, 0, 2)]
INDEX_IDS = ["records+grams", "records+descent", "text+descent", "records+grams-2launch",
             "text+descent-2launch"]


@pytest.mark.parametrize("mode", INDEX_MODES, ids=INDEX_IDS)
@pytest.mark.parametrize("grid", CORPUS_GRID, ids=lambda g: "V%d_D%d_R%d_cap%d" % (g[0], g[1], g[2], g[4]))
def test_fuzz_corpus(grid, mode):
    records, grams, launches = mode
    SuffixDrafter, W, O, H = _mods()
    V, D, R, k, cc, nd, dl = grid
    rng = np.random.default_rng(sum(grid))
    S = 256
    X = []
    for _ in range(nd):
        X += rng.integers(0, V, size=int(rng.integers(1, dl + 1))).tolist() + [V]
    X = np.asarray(X, dtype=np.int32)
    B = 128
    tok = np.full((B, S), -1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        nb = int(rng.integers(0, 48)) if b % 3 else int(rng.integers(0, S + 1))
        if b % 4 == 0 and len(X) > 20:  # tails copied from the corpus
            s = int(rng.integers(0, len(X) - 10))
            seg = [x for x in X[s:s + 12].tolist() if x != V][:nb]
            tok[b, :len(seg)] = seg
            nb = len(seg)
        else:
            tok[b, :nb] = rng.integers(0, V, size=nb)
        n[b] = nb
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=k, max_tree_depth=D,
                       max_occurrences=R, corpus_capacity=max(1024, len(X)), corpus_cand_cap=cc,
                       max_spec_factor=(2, 1), min_token_prob=(1, 8), corpus_records=records,
                       corpus_gram_index=grams, propose_mode=launches)
    _ingest_text(dr, X, V, S)
    dr.build_sa(torch.cuda.Stream())
    assert dr.poll(wait=True)[0] == 1
    text, sa, gen = dr.export_snapshot()
    assert gen == 1 and text.cpu().numpy().tolist() == X.tolist()
    assert sa.cpu().numpy().tolist() == O.suffix_array(X).tolist()
    out = dr.propose(_dev(tok), _dev(n))
    p = O.Params(S=S, V=V, k=k, D=D, R=R, factor=(2, 1), min_prob=(1, 8))
    orc = O.propose(p, tok, n, X=X, threads=H.THREADS)
    H.compare(out, orc, ctx=str(grid))
    assert (orc.match_info[:, 1] == 2).sum() > 0  # the corpus path is exercised
    dr.close()


def test_large_match_set_multi_pass_selection():
    """A frequent bigram: thousands of equal-length corpus ends, more than the
    on-chip candidate buffer holds; the R most recent must still be exact."""
    SuffixDrafter, W, O, H = _mods()
    rng = np.random.default_rng(5)
    V, S = 1000, 64
    X = []
    for i in range(3000):
        X += [7, 9, int(rng.integers(10, 1000)), int(rng.integers(10, 1000)), V]
    X = np.asarray(X, dtype=np.int32)
    tok = np.full((4, S), -1, dtype=np.int32)
    tok[0, :3] = [500, 7, 9]          # no self match: the bigram interval decides
    tok[1, :2] = [7, 9]
    tok[2, :4] = [1, 2, 7, 9]
    tok[3, :5] = [9, 3, 9, 7, 9]      # self M=1 (9), corpus 2 wins
    n = np.array([3, 2, 4, 5], dtype=np.int32)
    for cc, R, grams in ((64, 16, 1), (64, 64, 0), (128, 100, 1), (4096, 64, 0)):
        dr = SuffixDrafter(max_batch=4, seq_capacity=S, vocab_size=V, k=4, max_tree_depth=24,
                           max_occurrences=R, corpus_capacity=len(X), corpus_cand_cap=cc,
                           min_token_prob=(0, 1), max_docs=4096, corpus_gram_index=grams)
        _ingest_text(dr, X, V, S)
        dr.build_sa(torch.cuda.Stream())
        assert dr.poll(wait=True)[0] == 1
        out = dr.propose(_dev(tok), _dev(n))
        p = O.Params(S=S, V=V, k=4, D=24, R=R, min_prob=(0, 1))
        orc = O.propose(p, tok, n, X=X)
        H.compare(out, orc, ctx="cand_cap %d R %d" % (cc, R))
        assert (orc.match_info[:, 1] == 2).all()
        dr.close()


@pytest.mark.parametrize("mode", INDEX_MODES, ids=INDEX_IDS)
@pytest.mark.parametrize("R", [16, 128])
def test_small_p4_interval_long_matches(R, mode):
    """A 4-token pattern with ~100 hits whose matches run back 10 tokens: the
    small-interval path evaluates them from one round of on-chip context and
    selects the R most recent (on-chip radix select when R < hits)."""
    SuffixDrafter, W, O, H = _mods()
    rng = np.random.default_rng(77 + R)
    V, S = 1000, 128
    A = rng.integers(0, V, size=30).tolist()
    X = []
    for i in range(110):
        L = int(rng.integers(10, 31))
        X += rng.integers(0, V, size=5).tolist() + A[:L] + rng.integers(0, V, size=3).tolist() + [V]
    X += A[:10] + [V]                       # a hit whose continuation is the sentinel
    X = np.asarray(X, dtype=np.int32)
    tok = np.full((3, S), -1, dtype=np.int32)
    tok[0, :12] = [3, 4] + A[:10]            # M_c = 10 (the prefix breaks the match)
    tok[1, :10] = A[:10]                     # match bounded by the row start
    tok[2, :26] = [5] + A[:25]               # long match, capped by D
    n = np.array([12, 10, 26], dtype=np.int32)
    dr = SuffixDrafter(max_batch=3, seq_capacity=S, vocab_size=V, k=8, max_tree_depth=24,
                       max_occurrences=R, corpus_capacity=len(X), min_token_prob=(1, 20),
                       max_docs=4096, corpus_records=mode[0], corpus_gram_index=mode[1],
                       propose_mode=mode[2])
    _ingest_text(dr, X, V, S)
    dr.build_sa(torch.cuda.Stream())
    assert dr.poll(wait=True)[0] == 1
    out = dr.propose(_dev(tok), _dev(n))
    p = O.Params(S=S, V=V, k=8, D=24, R=R, min_prob=(1, 20))
    orc = O.propose(p, tok, n, X=X)
    H.compare(out, orc, ctx="R %d" % R)
    assert (orc.match_info[:, 1] == 2).all()
    dr.close()


def test_update_and_error_flags():
    SuffixDrafter, W, O, H = _mods()
    rng = np.random.default_rng(2)
    B, S, T, V = 64, 64, 9, 20
    tok = np.full((B, S), -1, dtype=np.int32)
    n = rng.integers(-3, S + 3, size=B).astype(np.int32)
    for b in range(B):
        m = int(min(max(n[b], 0), S))
        tok[b, :m] = rng.integers(0, V, size=m)
    sampled = rng.integers(-1, V + 2, size=(B, T)).astype(np.int32)
    sampled[::3, :4] = rng.integers(0, V, size=(len(range(0, B, 3)), 4))
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=8, max_sampled=T)
    g_tok, g_n = _dev(tok), _dev(n)
    dr.update_state(g_tok, g_n, _dev(sampled))
    o_tok, o_n = tok.copy(), n.copy()
    flags = O.update_state(o_tok, o_n, sampled, V)
    assert np.array_equal(g_n.cpu().numpy(), o_n)
    assert np.array_equal(g_tok.cpu().numpy(), o_tok)
    assert dr.get_error(clear=True) == flags and flags & 1 and flags & 2
    assert dr.get_error() == 0
    # fused form: same buffers, then drafts
    out = dr.propose_with_update(g_tok, g_n, _dev(sampled))
    flags = O.update_state(o_tok, o_n, sampled, V)
    orc = O.propose(O.Params(S=S, V=V, k=8), o_tok, o_n)
    assert np.array_equal(g_tok.cpu().numpy(), o_tok) and np.array_equal(g_n.cpu().numpy(), o_n)
    H.compare(out, orc)
    assert dr.get_error(clear=True) == flags
    dr.close()


def test_empty_batch_and_small_rows():
    SuffixDrafter, W, O, H = _mods()
    S, V = 16, 5
    dr = SuffixDrafter(max_batch=8, seq_capacity=S, vocab_size=V, k=4, max_sampled=3)
    z = torch.zeros((0, S), dtype=torch.int32, device="cuda")
    out = dr.propose(z, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert out.drafts.shape == (0, 4)
    tok = np.full((6, S), -1, dtype=np.int32)
    rows = [[], [1], [1, 1], [1, 2, 1, 2], [1] * 15, [2] * 16]
    for i, r in enumerate(rows):
        tok[i, :len(r)] = r
    n = np.array([len(r) for r in rows], dtype=np.int32)
    out = dr.propose(_dev(tok), _dev(n))
    orc = O.propose(O.Params(S=S, V=V, k=4), tok, n)
    H.compare(out, orc)
    assert out.num_valid.cpu().numpy().tolist()[4:] == [0, 0]  # no room left in the row
    sampled = np.array([[1, -1, 3]] * 6, dtype=np.int32)
    out = dr.propose_with_update(_dev(tok), _dev(n), _dev(sampled[:, :1]))
    dr.close()


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("max_m", [8, 64])
def test_ring_and_snapshot_match_oracle(max_m):
    """Small calls run as one CTA, larger ones as measure/plan/copy kernels."""
    SuffixDrafter, W, O, H = _mods()
    rng = np.random.default_rng(8 + max_m)
    V, S, C, MD = 50, 64, 500 if max_m == 8 else 2000, 12 if max_m == 8 else 40
    dr = SuffixDrafter(max_batch=16, seq_capacity=S, vocab_size=V, k=4, corpus_capacity=C,
                       max_docs=MD, max_ingest_docs=max_m)
    ring = O.Ring(C, MD, V)
    side = torch.cuda.Stream()
    for it in range(40):
        m = int(rng.integers(1, max_m + 1))
        buf = rng.integers(0, V, size=(m, S)).astype(np.int32)
        buf[rng.random((m, S)) < 0.01] = V + 3          # occasional bad id -> truncation
        rows = np.arange(m, dtype=np.int32)
        starts = rng.integers(0, 8, size=m).astype(np.int32)
        lens = rng.integers(0, 80, size=m).astype(np.int32)
        lens[0] = min(lens[0], S - starts[0])
        if it % 7 == 3:
            rows[-1] = 99                                 # bad row -> skipped
        num = rng.integers(S // 2, S + 1, size=max_m).astype(np.int32)  # some docs end past it
        dr.ingest(_dev(buf), _dev(rows), _dev(starts), _dev(lens), num_tokens=_dev(num[:m]))
        f_orc = ring.ingest(buf, rows, starts, lens, num_tokens=num[:m])
        assert dr.get_error(clear=True) == f_orc
        live, nd = dr.corpus_stats()
        assert (live, nd) == (ring.live, ring.ndocs)
        if it % 5 == 4:
            dr.build_sa(side)
            assert dr.poll(wait=True)[0] == 1
            text, sa, gen = dr.export_snapshot()
            X = ring.snapshot()
            assert text.cpu().numpy().tolist() == X.tolist()
            assert O.check_suffix_array(X, sa.cpu().numpy()) == 0
    dr.close()


def test_failure_injection_keeps_old_index():
    SuffixDrafter, W, O, H = _mods()
    from model_free_suffix_gb300 import _lib as L
    V, S = 10, 32
    dr = SuffixDrafter(max_batch=2, seq_capacity=S, vocab_size=V, k=4, corpus_capacity=256)
    side = torch.cuda.Stream()
    _ingest_text(dr, [1, 2, 3, 4, V], V, S)
    dr.build_sa(side)
    assert dr.poll(wait=True)[0] == L.SGD_OK_SWAPPED
    tok = np.full((1, S), -1, dtype=np.int32)
    tok[0, :2] = [2, 3]
    before = dr.propose(_dev(tok), _dev([2]))
    assert before.drafts.cpu().numpy()[0, :1].tolist() == [4]
    _ingest_text(dr, [2, 3, 9, V, 2, 3, 9, V], V, S)
    dr.debug_inject(L.INJECT_BUILD_FAIL)
    dr.build_sa(side)
    st, gen = dr.poll(wait=True)
    assert st == L.SGD_EBUILD and gen == 1
    after = dr.propose(_dev(tok), _dev([2]))
    assert after.drafts.cpu().numpy().tolist() == before.drafts.cpu().numpy().tolist()
    dr.debug_inject(L.INJECT_BUILD_HANG)
    dr.build_sa(side)
    assert dr.poll(wait=True, timeout_us=50_000)[0] == L.SGD_ETIMEDOUT
    assert dr.poll(wait=False)[0] == L.SGD_PENDING
    assert dr.try_build_sa(side) == L.SGD_EBUSY
    dr.debug_inject(L.INJECT_NONE)                      # the build is released
    st, gen = dr.poll(wait=True)
    assert st == L.SGD_OK_SWAPPED and gen == 2
    new = dr.propose(_dev(tok), _dev([2]))
    assert new.drafts.cpu().numpy()[0, :1].tolist() == [9]
    dr.close()


def test_graph_capture_and_swap_under_capture():
    SuffixDrafter, W, O, H = _mods()
    V, S, B = 40, 128, 16
    rng = np.random.default_rng(4)
    dr = SuffixDrafter(max_batch=B, seq_capacity=S, vocab_size=V, k=8, max_sampled=5,
                       corpus_capacity=4096)
    side = torch.cuda.Stream()
    X1 = []
    for _ in range(20):
        X1 += rng.integers(0, V, size=int(rng.integers(5, 40))).tolist() + [V]
    _ingest_text(dr, X1, V, S)
    dr.build_sa(side)
    assert dr.poll(wait=True)[0] == 1
    tok = np.full((B, S), -1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        s = int(rng.integers(0, len(X1) - 8))
        seg = [x for x in X1[s:s + 6] if x != V]
        tok[b, :len(seg)] = seg
        n[b] = len(seg)
    g_tok, g_n = _dev(tok), _dev(n)
    out = dr.new_outputs(B)
    sampled = _dev(np.full((B, 5), -1, dtype=np.int32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dr.propose_with_update(g_tok, g_n, sampled, out=out)   # warm-up outside capture
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            dr.propose_with_update(g_tok, g_n, sampled, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    graph.replay()
    torch.cuda.synchronize()
    p = O.Params(S=S, V=V, k=8)
    H.compare(out, O.propose(p, tok, n, X=np.asarray(X1, dtype=np.int32)), ctx="graph, snapshot 1")
    eager = dr.propose(g_tok, g_n)
    H.compare(eager, O.propose(p, tok, n, X=np.asarray(X1, dtype=np.int32)), ctx="eager")
    # new corpus; swap; replay the graph captured before the swap
    X2 = X1 + tok[0, :n[0]].tolist() + [33, 34, 35, V]
    _ingest_text(dr, tok[0, :n[0]].tolist() + [33, 34, 35, V], V, S)
    dr.build_sa(side)
    assert dr.poll(wait=True)[0] == 1
    graph.replay()
    torch.cuda.synchronize()
    H.compare(out, O.propose(p, tok, n, X=np.asarray(X2, dtype=np.int32)), ctx="graph after swap")
    dr.close()


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["c1", "c2"])
def test_self_configs_full(name):
    SuffixDrafter, W, O, H = _mods()
    cfg = W.CONFIGS[name]
    ls = H.Lockstep(cfg, seed=0, corpus=0)
    ls.step(check_state=True)  # also covers the initial buffers
    for _ in range(cfg.steps - 1):
        ls.step(check_state=True)
    assert ls.dr.get_error() == 0
    ls.close()


def test_c3_full_corpus():
    SuffixDrafter, W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=2048)
    ls = H.Lockstep(cfg, seed=0)
    ls.prefill(seed=0)
    text, sa, gen = ls.dr.export_snapshot()
    X = ls.X
    assert text.cpu().numpy().tolist() == X.tolist()
    assert np.array_equal(sa.cpu().numpy(), O.suffix_array(X))
    srcs = np.zeros(3, dtype=np.int64)
    for _ in range(cfg.steps):
        ls.step()
        mi = ls.out.match_info.cpu().numpy()
        srcs += np.bincount(mi[:, 1], minlength=3)
    assert ls.generation >= 2          # at least one rebuild was swapped in mid-run
    assert srcs[2] > 0 and srcs[1] > 0  # both sources won somewhere
    assert ls.dr.get_error() == 0
    ls.close()


def test_c5_sampled_rows():
    SuffixDrafter, W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c5"], rebuild_tokens=8192)
    ls = H.Lockstep(cfg, seed=0, steps=6)
    ls.prefill(seed=0)
    X = ls.X
    text, sa, gen = ls.dr.export_snapshot()
    assert text.cpu().numpy().tolist() == X.tolist()
    assert O.check_suffix_array(X, sa.cpu().numpy()) == 0
    rng = np.random.default_rng(0)
    for _ in range(6):
        rows = np.sort(rng.choice(cfg.B, size=48, replace=False))
        ls.step(check_rows=rows)
    assert ls.generation >= 2
    ls.close()


@pytest.mark.parametrize("N", [1 << 20, 1 << 24])
def test_c4_suffix_array(N):
    SuffixDrafter, W, O, H = _mods()
    X = W.sa_corpus(N, seed=0)
    dr = SuffixDrafter(max_batch=1, seq_capacity=8, vocab_size=151936, corpus_capacity=N)
    sa = dr.suffix_array(_dev(X)).cpu().numpy()
    if N <= 1 << 20:
        assert np.array_equal(sa, O.suffix_array(X))
    else:
        assert O.check_suffix_array(X, sa) == 0   # permutation + strictly increasing suffixes
    st = dr.build_stats()
    assert st["status"] == 0 and st["n"] == N and st["rounds"] >= 5
    dr.close()


@pytest.mark.parametrize("lo,hi", [(0, 1), (0, (1 << 16) - 2), (0, 151936), (-5, (1 << 21) - 6),
                                   (-(1 << 31), (1 << 31) - 1)])
def test_suffix_array_token_ranges(lo, hi):
    """Round 0 packs as many tokens per key as the text's token range allows
    (4, 4, 3, 2 and 1 token here); every range must give the oracle's array."""
    SuffixDrafter, W, O, H = _mods()
    rng = np.random.default_rng(hi & 0xffff)
    n = 30000
    X = rng.integers(lo, hi, size=n, endpoint=True, dtype=np.int64)
    span = rng.integers(lo, hi, size=300, endpoint=True, dtype=np.int64)
    for s0 in range(0, n - 300, 3000):  # long repeats force many doubling rounds
        X[s0:s0 + 300] = span
    X[0], X[-1] = lo, hi
    X = X.astype(np.int32)
    dr = SuffixDrafter(max_batch=1, seq_capacity=8, vocab_size=16, corpus_capacity=n)
    sa = dr.suffix_array(_dev(X)).cpu().numpy()
    assert np.array_equal(sa, O.suffix_array(X))
    assert dr.build_stats()["status"] == 0
    dr.close()


def test_c4_background_build_while_proposing():
    """The 1M corpus built on a side stream while proposes run; a graph
    captured before the swap reads the new index after it."""
    SuffixDrafter, W, O, H = _mods()
    N = 1 << 20
    X = W.sa_corpus(N, seed=1)
    cfg = W.CONFIGS["c3"]
    dr = H.drafter_for(cfg, B=cfg.B, corpus=N)
    _ingest_text(dr, X, cfg.V, cfg.S)
    tr = W.ServingTrace(cfg, seed=1, steps=2)
    tok, n = tr.initial()
    g_tok, g_n = _dev(tok), _dev(n)
    out = dr.propose(g_tok, g_n)   # empty index: self matches only
    p = H.params_for(cfg)
    H.compare(out, O.propose(p, tok, n, threads=H.THREADS), ctx="before swap")
    side = torch.cuda.Stream()
    dr.build_sa(side)
    for _ in range(20):            # drafting keeps running during the build
        dr.propose(g_tok, g_n, out=out)
    assert dr.poll(wait=True)[0] == 1
    text, sa, gen = dr.export_snapshot()
    assert np.array_equal(text.cpu().numpy(), X)
    assert np.array_equal(sa.cpu().numpy(), O.suffix_array(X))
    dr.propose(g_tok, g_n, out=out)
    H.compare(out, O.propose(p, tok, n, X=X, threads=H.THREADS), ctx="after swap")
    dr.close()
