"""Seeded synthetic workloads for the suffix-decoding drafter.

This module only produces data: token buffers, per-step sampled ids, finished
requests and corpus documents.  It contains none of the drafter's arithmetic
(no matching, voting or suffix sorting), so both the CUDA path and the CPU
oracle can be fed from it without sharing method code.

The public pages measure on Spec-Bench and GSM8K, which are not available
here; the generators below stand in for their repetition structure: each
sequence is a mix of fresh tokens (uniform or Zipf) and spans drawn from a
seeded pool, so that suffixes recur both within a request and across
requests, the way agentic and code-editing traffic repeats itself.

All randomness comes from ``numpy.random.Generator`` seeded through
``SeedSequence([config_id, purpose, seed])``.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

# purposes (distinct random streams per use)
_P_POOL, _P_ROWS, _P_STEPS, _P_CORPUS, _P_FINISH, _P_RESET, _P_C4 = range(7)


@dataclasses.dataclass(frozen=True)
class Config:
    """One workload: shapes, drafter knobs and the token recipe."""
    name: str
    cid: int
    B: int                      # batch rows
    S: int                      # row capacity (int32 tokens)
    V: int                      # vocabulary size; the corpus sentinel is V
    k: int                      # max draft tokens
    D: int                      # max_tree_depth
    R: int                      # max_occurrences
    T: int                      # sampled width per step (k + 1)
    steps: int                  # propose_with_update steps
    fresh: str                  # "uniform" or "zipf"
    zipf_s: float
    pool_size: int
    span_lo: int
    span_hi: int
    p_repeat: float
    n_lo: int
    n_hi: int
    factor: Tuple[int, int] = (1, 1)        # max_spec_factor as a rational
    offset: int = 0                         # max_spec_offset
    min_prob: Tuple[int, int] = (1, 10)     # min_token_prob as a rational
    corpus_tokens: int = 0                  # ring capacity (0: no corpus)
    doc_lo: int = 64
    doc_hi: int = 512
    finish_frac: float = 0.0                # rows finishing per step
    rebuild_tokens: int = 1 << 16           # rebuild once this many tokens were ingested


CONFIGS: Dict[str, Config] = {
    # self-match only, tiny
    "c1": Config("c1", 1, B=4, S=2048, V=32000, k=8, D=24, R=64, T=9, steps=32,
                 fresh="uniform", zipf_s=0.0, pool_size=64, span_lo=8, span_hi=64,
                 p_repeat=0.7, n_lo=512, n_hi=2048),
    # self-match only, Zipf tokens
    "c2": Config("c2", 2, B=64, S=8192, V=151936, k=16, D=24, R=64, T=17, steps=32,
                 fresh="zipf", zipf_s=1.1, pool_size=256, span_lo=16, span_hi=128,
                 p_repeat=0.5, n_lo=1024, n_hi=8192),
    # global corpus, the headline shape B=256, S=4096
    "c3": Config("c3", 3, B=256, S=4096, V=151936, k=16, D=24, R=64, T=17, steps=32,
                 fresh="zipf", zipf_s=1.1, pool_size=256, span_lo=16, span_hi=128,
                 p_repeat=0.5, n_lo=1024, n_hi=4096, corpus_tokens=1 << 20,
                 finish_frac=0.05),
    # long-context agentic scale
    "c5": Config("c5", 5, B=1024, S=32768, V=151936, k=32, D=32, R=64, T=33, steps=64,
                 fresh="zipf", zipf_s=1.1, pool_size=1024, span_lo=32, span_hi=512,
                 p_repeat=0.8, n_lo=8192, n_hi=32768, corpus_tokens=1 << 22,
                 finish_frac=0.05),
}


def _rng(cfg_id: int, purpose: int, seed: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([cfg_id, purpose, seed]))


class FreshSampler:
    """Fresh (non-repeated) tokens: uniform over [0, V) or bounded Zipf(s)."""

    def __init__(self, V: int, kind: str, s: float = 1.1):
        self.V = V
        self.kind = kind
        if kind == "zipf":
            ranks = np.arange(1, V + 1, dtype=np.float64)
            w = ranks ** (-s)
            cdf = np.cumsum(w)
            self.cdf = cdf / cdf[-1]
        elif kind != "uniform":
            raise ValueError(kind)

    def sample(self, rng: np.random.Generator, size: int) -> np.ndarray:
        if self.kind == "uniform":
            return rng.integers(0, self.V, size=size, dtype=np.int64).astype(np.int32)
        u = rng.random(size)
        r = np.searchsorted(self.cdf, u, side="right")
        return np.minimum(r, self.V - 1).astype(np.int32)


def span_pool(cfg: Config, seed: int) -> List[np.ndarray]:
    rng = _rng(cfg.cid, _P_POOL, seed)
    fresh = FreshSampler(cfg.V, cfg.fresh, cfg.zipf_s)
    out = []
    for _ in range(cfg.pool_size):
        ln = int(rng.integers(cfg.span_lo, cfg.span_hi + 1))
        out.append(fresh.sample(rng, ln))
    return out


def mixed_sequence(rng: np.random.Generator, length: int, p_repeat: float,
                   pool: List[np.ndarray], fresh: FreshSampler) -> np.ndarray:
    """Append pool spans (prob p_repeat) or 1..32 fresh tokens until `length`."""
    chunks = []
    total = 0
    # fresh tokens are drawn in blocks to keep the Python loop short
    blk = int(min(4096, max(64, length)))
    buf = fresh.sample(rng, blk)
    bpos = 0
    while total < length:
        if rng.random() < p_repeat:
            c = pool[int(rng.integers(len(pool)))]
        else:
            a = int(rng.integers(1, 33))
            if bpos + a > buf.shape[0]:
                buf = fresh.sample(rng, blk)
                bpos = 0
            c = buf[bpos:bpos + a]
            bpos += a
        chunks.append(c)
        total += c.shape[0]
    return np.concatenate(chunks)[:length].astype(np.int32)


@dataclasses.dataclass
class StepData:
    """Inputs of one serving step."""
    sampled: np.ndarray                 # [B, T] int32, leading accepted prefix then -1
    finished: np.ndarray                # [m] rows that finish after this step's propose
    ingest_starts: np.ndarray           # [m] start of each finished row's response
    ingest_lengths: np.ndarray          # [m] response length (capped by the row capacity)
    reset_tokens: Optional[np.ndarray]  # [m, S] new row contents (-1 beyond reset_n)
    reset_n: np.ndarray                 # [m]


class ServingTrace:
    """Rows, their continuation streams and the per-step finish/reset schedule.

    Each row owns one token stream: its first n tokens fill the buffer, the rest
    is the continuation that later steps' sampled ids reveal (a uniform 1..T
    accepted prefix per step, the remainder -1).  Continuations are generated
    on demand, in blocks, from the same mixed process.  When rows finish, their
    response (the tokens appended since the row started) is handed to the
    corpus and the row restarts with a fresh stream.
    """

    BLOCK = 256

    def __init__(self, cfg: Config, seed: int = 0, steps: Optional[int] = None,
                 finish_frac: Optional[float] = None, B: Optional[int] = None):
        self.cfg = cfg
        self.B = cfg.B if B is None else B
        self.steps = cfg.steps if steps is None else steps
        self.finish_frac = cfg.finish_frac if finish_frac is None else finish_frac
        self.pool = span_pool(cfg, seed)
        self.fresh = FreshSampler(cfg.V, cfg.fresh, cfg.zipf_s)
        self.seed = seed
        self._rows_rng = _rng(cfg.cid, _P_ROWS, seed)
        self._steps_rng = _rng(cfg.cid, _P_STEPS, seed)
        self._fin_rng = _rng(cfg.cid, _P_FINISH, seed)
        self._reset_rng = _rng(cfg.cid, _P_RESET, seed)
        S, B = cfg.S, self.B
        self.tokens = np.full((B, S), -1, dtype=np.int32)
        self.n0 = np.zeros(B, dtype=np.int32)
        self.stream: List[np.ndarray] = []
        self.pos = np.zeros(B, dtype=np.int64)       # consumed continuation tokens
        for b in range(B):
            tok, n = self._new_row(self._rows_rng)
            self.tokens[b, :n] = tok[:n]
            self.n0[b] = n
            self.stream.append(tok[n:])
        self.step_index = 0

    def _new_row(self, rng: np.random.Generator) -> Tuple[np.ndarray, int]:
        cfg = self.cfg
        n = int(rng.integers(cfg.n_lo, cfg.n_hi + 1))
        return mixed_sequence(rng, n + self.BLOCK, cfg.p_repeat, self.pool, self.fresh), n

    def _continuation(self, b: int, need: int, rng: np.random.Generator) -> np.ndarray:
        p = int(self.pos[b])
        while self.stream[b].shape[0] < p + need:
            ext = mixed_sequence(rng, max(self.BLOCK, need), self.cfg.p_repeat, self.pool,
                                 self.fresh)
            self.stream[b] = np.concatenate([self.stream[b], ext])
        return self.stream[b][p:p + need]

    def initial(self) -> Tuple[np.ndarray, np.ndarray]:
        return self.tokens.copy(), self.n0.copy()

    def next_step(self) -> StepData:
        cfg, B, T, S = self.cfg, self.B, self.cfg.T, self.cfg.S
        rng = self._steps_rng
        a = rng.integers(1, T + 1, size=B)
        sampled = np.full((B, T), -1, dtype=np.int32)
        for b in range(B):
            sampled[b, :a[b]] = self._continuation(b, int(a[b]), self._rows_rng)
            self.pos[b] += a[b]
        m = int(np.floor(self.finish_frac * B))
        if m > 0:
            fin = np.sort(self._fin_rng.choice(B, size=m, replace=False)).astype(np.int32)
            starts = self.n0[fin].copy()
            # response = tokens appended since the row started, bounded by the row
            lengths = np.minimum(self.pos[fin], S - starts).astype(np.int32)
            reset_tokens = np.full((m, S), -1, dtype=np.int32)
            reset_n = np.zeros(m, dtype=np.int32)
            for i, b in enumerate(fin):
                tok, n = self._new_row(self._reset_rng)
                reset_tokens[i, :n] = tok[:n]
                reset_n[i] = n
                self.n0[b] = n
                self.stream[b] = tok[n:]
                self.pos[b] = 0
        else:
            fin = np.zeros(0, dtype=np.int32)
            starts = np.zeros(0, dtype=np.int32)
            lengths = np.zeros(0, dtype=np.int32)
            reset_tokens = None
            reset_n = np.zeros(0, dtype=np.int32)
        self.step_index += 1
        return StepData(sampled, fin, starts, lengths, reset_tokens, reset_n)


def corpus_docs(cfg: Config, seed: int = 0, capacity: Optional[int] = None,
                pool: Optional[List[np.ndarray]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Documents that fill a ring of `capacity` tokens (each doc costs len + 1).

    Docs have U[doc_lo, doc_hi] tokens from the config's mixed generator and
    span pool.  Generation stops when the next doc would not fit.
    Returns (docs [m, doc_hi] int32 padded with -1, lengths [m] int32).
    """
    cap = cfg.corpus_tokens if capacity is None else capacity
    rng = _rng(cfg.cid, _P_CORPUS, seed)
    fresh = FreshSampler(cfg.V, cfg.fresh, cfg.zipf_s)
    pool = span_pool(cfg, seed) if pool is None else pool
    docs, lens = [], []
    used = 0
    while True:
        ln = int(rng.integers(cfg.doc_lo, cfg.doc_hi + 1))
        if used + ln + 1 > cap:
            break
        docs.append(mixed_sequence(rng, ln, cfg.p_repeat, pool, fresh))
        lens.append(ln)
        used += ln + 1
    out = np.full((len(docs), cfg.doc_hi), -1, dtype=np.int32)
    for i, d in enumerate(docs):
        out[i, :d.shape[0]] = d
    return out, np.asarray(lens, dtype=np.int32)


def sa_corpus(N: int, seed: int = 0, V: int = 151936, repeat_frac: float = 0.3,
              n_spans: int = 512, span_lo: int = 32, span_hi: int = 256,
              doc_lo: int = 64, doc_hi: int = 512) -> np.ndarray:
    """Text of exactly N int32 tokens for the suffix-array workload.

    Docs of U[doc_lo, doc_hi] tokens, each followed by the sentinel V.  Fresh
    tokens are Zipf(1.1) over V; before each chunk a deterministic controller
    picks a repeat (a span from a pool of `n_spans` spans of U[span_lo,
    span_hi] Zipf tokens) iff repeated tokens so far are below `repeat_frac`
    of all tokens, else 1..32 fresh tokens.  The last doc is truncated so that
    it and its sentinel end exactly at N.
    """
    rng = _rng(4, _P_C4, seed)
    fresh = FreshSampler(V, "zipf", 1.1)
    spans = [fresh.sample(rng, int(rng.integers(span_lo, span_hi + 1))) for _ in range(n_spans)]
    out = np.empty(N, dtype=np.int32)
    pos = 0
    rep = 0
    total = 0
    fbuf = fresh.sample(rng, 1 << 16)
    fpos = 0
    while pos < N:
        ln = int(rng.integers(doc_lo, doc_hi + 1))
        ln = min(ln, N - pos - 1)
        filled = 0
        while filled < ln:
            if rep < repeat_frac * max(total, 1):
                c = spans[int(rng.integers(n_spans))]
                is_rep = True
            else:
                a = int(rng.integers(1, 33))
                if fpos + a > fbuf.shape[0]:
                    fbuf = fresh.sample(rng, 1 << 16)
                    fpos = 0
                c = fbuf[fpos:fpos + a]
                fpos += a
                is_rep = False
            take = min(c.shape[0], ln - filled)
            out[pos + filled:pos + filled + take] = c[:take]
            filled += take
            total += take
            if is_rep:
                rep += take
        pos += ln
        out[pos] = V
        pos += 1
    return out


def docs_from_text(text: np.ndarray, sentinel: int) -> Tuple[np.ndarray, np.ndarray]:
    """Split a sentinel-terminated text into a padded doc matrix and lengths."""
    ends = np.flatnonzero(text == sentinel)
    starts = np.concatenate([[0], ends[:-1] + 1])
    lens = (ends - starts).astype(np.int32)
    width = int(max(1, lens.max(initial=1)))
    out = np.full((lens.shape[0], width), -1, dtype=np.int32)
    for i, (s, l) in enumerate(zip(starts, lens)):
        out[i, :l] = text[s:s + l]
    return out, lens
