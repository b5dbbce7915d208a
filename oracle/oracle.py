"""ctypes wrapper of the CPU oracle (test infrastructure only).

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg import this module.  The product path never does.  Arrays are numpy;
every call releases the GIL (ctypes does), so rows can be spread over a
thread pool without touching the oracle itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from fractions import Fraction
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgd_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

ERR_SAMPLED_TOKEN = 0x1
ERR_NUM_TOKENS = 0x2
ERR_DOC_ARGS = 0x4
ERR_DOC_TOKEN = 0x8
ERR_DOC_TOO_LONG = 0x10


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (plain gcc)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    srcs = [_SRC, os.path.join(_HERE, "sgd_oracle.h")]
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(s) for s in srcs)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared",
                           "-fPIC", "-o", tmp, _SRC])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int32), ("V", ctypes.c_int32), ("k", ctypes.c_int32),
                ("D", ctypes.c_int32), ("R", ctypes.c_int32),
                ("fN", ctypes.c_int64), ("fD", ctypes.c_int64), ("offset", ctypes.c_int64),
                ("pN", ctypes.c_int64), ("pD", ctypes.c_int64),
                ("depth_sum_cap", ctypes.c_int32), ("fixed_length", ctypes.c_int32),
                ("select_by_score", ctypes.c_int32), ("num_backoff", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
        _lib.orc_update_row.restype = u32
        _lib.orc_update_row.argtypes = [P, P, P, i32, i32, i32]
        _lib.orc_update_state.restype = u32
        _lib.orc_update_state.argtypes = [P, P, P, i32, i32, i32, i32]
        _lib.orc_self_match.restype = i32
        _lib.orc_self_match.argtypes = [P, i32, i32, i32, P, P]
        _lib.orc_corpus_match.restype = i32
        _lib.orc_corpus_match.argtypes = [P, i64, i32, P, i32, i32, i32, P, P]
        _lib.orc_backoff_lengths.restype = i32
        _lib.orc_backoff_lengths.argtypes = [P, i64, i32, i32, P, P]
        _lib.orc_propose_row.restype = None
        _lib.orc_propose_row.argtypes = [P, P, i32, P, i64, i32, P, P, P, P, P, P]
        _lib.orc_propose.restype = u32
        _lib.orc_propose.argtypes = [P, P, P, P, i32, P, i64, P, P, P, P, P]
        _lib.orc_suffix_array.restype = None
        _lib.orc_suffix_array.argtypes = [P, i64, P]
        _lib.orc_check_suffix_array.restype = i64
        _lib.orc_check_suffix_array.argtypes = [P, i64, P]
        _lib.orc_ring_create.restype = P
        _lib.orc_ring_create.argtypes = [i64, i32, i32]
        _lib.orc_ring_destroy.restype = None
        _lib.orc_ring_destroy.argtypes = [P]
        _lib.orc_ring_ingest.restype = u32
        _lib.orc_ring_ingest.argtypes = [P, P, P, i32, i32, P, P, P, i32]
        _lib.orc_ring_live.restype = i64
        _lib.orc_ring_live.argtypes = [P]
        _lib.orc_ring_ndocs.restype = i32
        _lib.orc_ring_ndocs.argtypes = [P]
        _lib.orc_ring_snapshot.restype = i64
        _lib.orc_ring_snapshot.argtypes = [P, P]
        _lib.orc_ring_pushed.restype = i64
        _lib.orc_ring_pushed.argtypes = [P]
        _lib.orc_ring_delta.restype = i64
        _lib.orc_ring_delta.argtypes = [P, i64, i64, P]
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def rational(x, denom: int = 10 ** 6):
    """A float knob as the rational the library uses (x rounded to 1e-6)."""
    if isinstance(x, tuple):
        return int(x[0]), int(x[1])
    f = Fraction(int(round(float(x) * denom)), denom)
    return f.numerator, f.denominator


class Params:
    """Drafter knobs (S, V, k, D, R, factor, offset, min_prob, depth_sum_cap, fixed_length,
    select_by_score, num_backoff)."""

    def __init__(self, S, V, k=16, D=24, R=64, factor=(1, 1), offset=0,
                 min_prob=(1, 10), depth_sum_cap=False, fixed_length=False, select_by_score=False,
                 num_backoff=1):
        self.S, self.V, self.k, self.D, self.R = int(S), int(V), int(k), int(D), int(R)
        self.factor = rational(factor)
        self.offset = int(offset)
        self.min_prob = rational(min_prob)
        self.depth_sum_cap = bool(depth_sum_cap)
        self.fixed_length = bool(fixed_length)
        self.select_by_score = bool(select_by_score)
        self.num_backoff = int(num_backoff)

    def c(self) -> _Params:
        return _Params(self.S, self.V, self.k, self.D, self.R, self.factor[0], self.factor[1],
                       self.offset, self.min_prob[0], self.min_prob[1], int(self.depth_sum_cap),
                       int(self.fixed_length), int(self.select_by_score), self.num_backoff)


def update_state(token_ids: np.ndarray, num_tokens: np.ndarray, sampled: np.ndarray, V: int) -> int:
    """In place on (token_ids [B,S], num_tokens [B]); returns error flags."""
    assert token_ids.dtype == np.int32 and token_ids.flags.c_contiguous
    assert num_tokens.dtype == np.int32 and num_tokens.flags.c_contiguous
    sampled = _i32(sampled)
    B, S = token_ids.shape
    return int(lib().orc_update_state(_p(token_ids), _p(num_tokens), _p(sampled), B,
                                      sampled.shape[1], S, V))


def self_match(t, n: int, D: int, R: int):
    t = _i32(t)
    occ = np.zeros(max(R, 1), dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    M = lib().orc_self_match(_p(t), int(n), D, R, _p(occ), _p(cnt))
    return int(M), occ[:cnt[0]].copy()


def corpus_match(X, Z: int, t, n: int, D: int, R: int):
    X = _i32(X)
    t = _i32(t)
    occ = np.zeros(max(R, 1), dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    M = lib().orc_corpus_match(_p(X), X.shape[0], Z, _p(t), int(n), D, R, _p(occ), _p(cnt))
    return int(M), occ[:cnt[0]].copy()


class Proposal:
    def __init__(self, drafts, num_valid, score, probs, match_info, flags):
        self.drafts, self.num_valid, self.score = drafts, num_valid, score
        self.probs, self.match_info, self.flags = probs, match_info, flags


def backoff_lengths(L, minlen: int, nb: int):
    """Candidate lengths of multi-length backoff ([PYPI] How it works, step 1):
    the distinct values among the nb largest match lengths >= minlen, longest
    first, with the number of ends reaching each."""
    L = _i32(L)
    lens = np.zeros(max(nb, 1), dtype=np.int32)
    sup = np.zeros(max(nb, 1), dtype=np.int64)
    c = lib().orc_backoff_lengths(_p(L), L.shape[0], minlen, nb, _p(lens), _p(sup))
    return [(int(lens[i]), int(sup[i])) for i in range(c)]


def propose_row(p: Params, t, n: int, X=None, active: bool = True) -> Proposal:
    t = _i32(t)
    Xa = None if X is None else _i32(X)
    drafts = np.zeros(p.k, dtype=np.int32)
    nv = np.zeros(1, dtype=np.int32)
    score = np.zeros(1, dtype=np.float32)
    probs = np.zeros(p.k, dtype=np.float32)
    mi = np.zeros(2, dtype=np.int32)
    flags = np.zeros(1, dtype=np.uint32)
    prm = p.c()
    lib().orc_propose_row(ctypes.byref(prm), _p(t), int(n), _p(Xa),
                          0 if Xa is None else Xa.shape[0], int(bool(active)),
                          _p(drafts), _p(nv), _p(score), _p(probs), _p(mi), _p(flags))
    return Proposal(drafts, int(nv[0]), float(score[0]), probs, mi, int(flags[0]))


def propose(p: Params, token_ids: np.ndarray, num_tokens: np.ndarray, X=None,
            active=None, rows=None, threads: int = 1) -> Proposal:
    """Batch proposal; `rows` restricts the work to a subset (others stay empty).

    With threads > 1 the rows are spread over a thread pool; each call of the
    oracle still runs single-threaded on its own row.
    """
    token_ids = _i32(token_ids)
    num_tokens = _i32(num_tokens)
    B = token_ids.shape[0]
    assert token_ids.shape[1] == p.S
    Xa = None if X is None else _i32(X)
    NX = 0 if Xa is None else Xa.shape[0]
    act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
    drafts = np.full((B, p.k), -1, dtype=np.int32)
    nv = np.zeros(B, dtype=np.int32)
    score = np.zeros(B, dtype=np.float32)
    probs = np.zeros((B, p.k), dtype=np.float32)
    mi = np.zeros((B, 2), dtype=np.int32)
    flags = np.zeros(B, dtype=np.uint32)
    prm = p.c()
    L = lib()
    row_list = range(B) if rows is None else [int(r) for r in rows]

    def one(b):
        L.orc_propose_row(ctypes.byref(prm), _p(token_ids[b]), int(num_tokens[b]), _p(Xa), NX,
                          1 if act is None else int(act[b]), _p(drafts[b]), _p(nv[b:b + 1]),
                          _p(score[b:b + 1]), _p(probs[b]), _p(mi[b]), _p(flags[b:b + 1]))

    if threads > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, row_list))
    else:
        for b in row_list:
            one(b)
    f = 0
    for x in flags:
        f |= int(x)
    return Proposal(drafts, nv, score, probs, mi, f)


def suffix_array(X) -> np.ndarray:
    X = _i32(X)
    SA = np.zeros(X.shape[0], dtype=np.int32)
    lib().orc_suffix_array(_p(X), X.shape[0], _p(SA))
    return SA


def check_suffix_array(X, SA) -> int:
    """0 if SA is the suffix array of X, else 1 + the first failing index."""
    X = _i32(X)
    SA = _i32(SA)
    if SA.shape[0] != X.shape[0]:
        return 1
    return int(lib().orc_check_suffix_array(_p(X), X.shape[0], _p(SA)))


class Ring:
    """FIFO corpus model (documents of finished responses, oldest out first)."""

    def __init__(self, capacity: int, max_docs: int, V: int):
        self.V = V
        self._h = lib().orc_ring_create(int(capacity), int(max_docs), int(V))

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_ring_destroy(self._h)
            self._h = None

    def ingest(self, token_ids, rows, starts, lengths, num_tokens=None) -> int:
        token_ids = _i32(token_ids)
        B, S = token_ids.shape
        rows, starts, lengths = _i32(rows), _i32(starts), _i32(lengths)
        nt = None if num_tokens is None else _i32(num_tokens)
        return int(lib().orc_ring_ingest(self._h, _p(token_ids), _p(nt), B, S, _p(rows),
                                         _p(starts), _p(lengths), rows.shape[0]))

    @property
    def live(self) -> int:
        return int(lib().orc_ring_live(self._h))

    @property
    def ndocs(self) -> int:
        return int(lib().orc_ring_ndocs(self._h))

    def snapshot(self) -> np.ndarray:
        X = np.zeros(max(self.live, 1), dtype=np.int32)
        n = lib().orc_ring_snapshot(self._h, _p(X))
        return X[:n].copy()

    @property
    def pushed(self) -> int:
        return int(lib().orc_ring_pushed(self._h))

    def delta(self, since: int, cap: int) -> np.ndarray:
        """Docs not yet indexed by a snapshot taken at pushed == since, cut at cap tokens."""
        Y = np.zeros(max(min(int(cap), self.live), 1), dtype=np.int32)
        n = lib().orc_ring_delta(self._h, int(since), int(cap), _p(Y))
        return Y[:n].copy()


def corpus_text(X: Optional[np.ndarray], Y: Optional[np.ndarray]) -> Optional[np.ndarray]:
    """The text a row is matched against: the snapshot, then the not-yet-indexed
    docs ([PYPI] How it works, step 2: the suffix array plus a brute-force scan
    of the delta buffer)."""
    parts = [a for a in (X, Y) if a is not None and a.shape[0] > 0]
    if not parts:
        return None
    return np.concatenate(parts).astype(np.int32)
