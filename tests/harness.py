"""Lockstep runner: the CUDA library and the CPU oracle on the same seeded inputs.

Inputs come from model_free_suffix_gb300.workload; the oracle never sees a
value produced by the CUDA path.  Build and swap points of the corpus index
are fixed in advance (a build is started after a step's ingest once enough
tokens arrived, and swapped in with a blocking poll before the next step),
so both sides use the same snapshot at every step.  With a delta capacity the
oracle's corpus is that snapshot followed by the docs placed since it was
linearised (oracle Ring.delta), cut at the capacity.
"""
from __future__ import annotations

import os
from typing import List, Optional

import numpy as np
import torch

from model_free_suffix_gb300 import SuffixDrafter
from model_free_suffix_gb300 import workload as W
from oracle import oracle as O

THREADS = max(1, min(16, os.cpu_count() or 1))


def drafter_for(cfg: W.Config, B: Optional[int] = None, corpus: Optional[int] = None,
                **over) -> SuffixDrafter:
    kw = dict(max_batch=B or cfg.B, seq_capacity=cfg.S, vocab_size=cfg.V, k=cfg.k,
              max_tree_depth=cfg.D, max_occurrences=cfg.R, max_sampled=cfg.T,
              max_spec_factor=cfg.factor, max_spec_offset=cfg.offset, min_token_prob=cfg.min_prob,
              corpus_capacity=cfg.corpus_tokens if corpus is None else corpus)
    kw.update(over)
    return SuffixDrafter(**kw)


def params_for(cfg: W.Config, **over) -> O.Params:
    kw = dict(S=cfg.S, V=cfg.V, k=cfg.k, D=cfg.D, R=cfg.R, factor=cfg.factor, offset=cfg.offset,
              min_prob=cfg.min_prob)
    kw.update(over)
    return O.Params(**kw)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def _f32_words(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def compare(gpu, orc, rows=None, ctx="", check_probs=True):
    """Bit-exact drafts / counts / match info, and bit-equal float32 scores and
    per-slot probabilities.

    Both sides round the same integer quotient (a chain count or a count sum
    over c0) to float32: the oracle from the double quotient, the kernel by one
    single-precision division of exact integers.  tests/test_arith.py checks
    exhaustively that these land on the same float for every quotient the
    drafter can form, so the float words must be identical, which is stricter
    than a 1e-6 relative tolerance."""
    gd, gn, gs = to_np(gpu.drafts), to_np(gpu.num_valid), to_np(gpu.score)
    gp, gm = to_np(gpu.probs), to_np(gpu.match_info)
    gs_w, os_w = _f32_words(gs), _f32_words(orc.score)
    gp_w, op_w = _f32_words(gp), _f32_words(orc.probs)
    idx = np.arange(gd.shape[0]) if rows is None else np.asarray(rows)
    bad = []
    for b in idx:
        ok = (np.array_equal(gd[b], orc.drafts[b]) and gn[b] == orc.num_valid[b]
              and np.array_equal(gm[b], orc.match_info[b]) and gs_w[b] == os_w[b])
        if ok and check_probs:
            ok = bool(np.array_equal(gp_w[b], op_w[b]))
        if not ok:
            bad.append(b)
    if bad:
        b = bad[0]
        msg = ("%s: %d/%d rows differ; first row %d:\n gpu drafts %s nv %d score %r mi %s probs %s\n"
               " orc drafts %s nv %d score %r mi %s probs %s" % (
                   ctx, len(bad), len(idx), b, gd[b].tolist(), gn[b], float(gs[b]), gm[b].tolist(),
                   gp[b].tolist(), orc.drafts[b].tolist(), orc.num_valid[b], float(orc.score[b]),
                   orc.match_info[b].tolist(), orc.probs[b].tolist()))
        raise AssertionError(msg)


def invariants(gpu, k, min_prob=(1, 10)):
    """Properties that hold at any size: -1 padding, counts, monotone probs."""
    d, n, s, p = to_np(gpu.drafts), to_np(gpu.num_valid), to_np(gpu.score), to_np(gpu.probs)
    assert ((n >= 0) & (n <= k)).all()
    pos = np.arange(k)[None, :]
    assert ((d == -1) == (pos >= n[:, None])).all()
    valid = pos < n[:, None]
    assert (p[~valid] == 0).all()
    assert (np.diff(np.where(valid, p, 0), axis=1)[valid[:, 1:]] <= 0).all()
    assert (p[valid] >= np.float32(min_prob[0] / min_prob[1]) - 1e-6).all()
    assert np.allclose(s, np.where(valid, p.astype(np.float64), 0).sum(1), rtol=1e-5, atol=1e-5)


def invariants_fixed(gpu, k):
    """Model Runner V2 drafts: k tokens or none, probabilities non-increasing
    and 0 from the first filled slot on."""
    d, n, p = to_np(gpu.drafts), to_np(gpu.num_valid), to_np(gpu.probs)
    assert np.isin(n, [0, k]).all()
    assert ((d == -1) == (n[:, None] == 0)).all()
    assert (np.diff(p, axis=1) <= 0).all()


class Lockstep:
    """One serving trace run on the GPU and the oracle side by side."""

    def __init__(self, cfg: W.Config, seed: int = 0, B: Optional[int] = None,
                 steps: Optional[int] = None, finish_frac: Optional[float] = None,
                 corpus: Optional[int] = None, drafter_over: Optional[dict] = None,
                 param_over: Optional[dict] = None, fused: bool = False, delta: int = 0):
        self.cfg = cfg
        self.delta = delta  # delta capacity in tokens (0: only swapped snapshots are matched)
        self.fused = fused  # drive each step through sgd_step (update + propose + ingest)
        self.trace = W.ServingTrace(cfg, seed=seed, steps=steps, finish_frac=finish_frac, B=B)
        self.B = self.trace.B
        self.corpus = cfg.corpus_tokens if corpus is None else corpus
        over = dict(drafter_over or {})
        if delta:
            over["delta_capacity"] = delta
        self.dr = drafter_for(cfg, B=self.B, corpus=self.corpus, **over)
        self.p = params_for(cfg, **(param_over or {}))
        tok, n = self.trace.initial()
        self.o_tok, self.o_n = tok.copy(), n.copy()
        dev = self.dr.device
        self.tok = torch.from_numpy(tok).to(dev)
        self.n = torch.from_numpy(n).to(dev)
        # rows written by the caller: their bigram indexes start from them
        self.row_index = bool(over.get("row_index"))
        if self.row_index:
            self.dr.reset_rows(self.tok, self.n, torch.arange(self.B, dtype=torch.int32, device=dev))
        self.out = self.dr.new_outputs(self.B)
        self.X = None            # oracle's current snapshot
        self.X_pending = None
        self.since = 0           # ring docs placed when the current snapshot was linearised
        self.since_pending = 0
        self.ring = O.Ring(self.corpus, 65536, cfg.V) if self.corpus else None
        self.ingested_since_build = 0
        self.build_pending = False
        self.side = torch.cuda.Stream(device=dev)
        self.generation = 0

    # corpus ------------------------------------------------------------------
    def prefill(self, seed: int = 0, docs=None, lens=None, chunk: int = 0):
        if chunk <= 0:  # keep the staging buffer near 64 MB
            chunk = max(1, min(2048, (64 << 20) // (self.cfg.S * 4)))
        if docs is None:
            docs, lens = W.corpus_docs(self.cfg, seed=seed, capacity=self.corpus, pool=self.trace.pool)
        dev = self.dr.device
        for s in range(0, docs.shape[0], chunk):
            d = np.ascontiguousarray(docs[s:s + chunk])
            m = d.shape[0]
            rows = np.arange(m, dtype=np.int32)
            starts = np.zeros(m, dtype=np.int32)
            ln = np.ascontiguousarray(lens[s:s + chunk]).astype(np.int32)
            dd = torch.zeros((m, self.cfg.S), dtype=torch.int32, device=dev)
            dd[:, :d.shape[1]] = torch.from_numpy(d).to(dev)
            self.dr.ingest(dd, torch.from_numpy(rows).to(dev), torch.from_numpy(starts).to(dev),
                           torch.from_numpy(ln).to(dev))
            buf = np.zeros((m, self.cfg.S), dtype=np.int32)
            buf[:, :d.shape[1]] = d
            self.ring.ingest(buf, rows, starts, ln)
        self.build_and_swap()

    def start_build(self):
        self.dr.build_sa(self.side)
        self.X_pending = self.ring.snapshot()
        self.since_pending = self.ring.pushed
        self.build_pending = True
        self.ingested_since_build = 0

    def swap(self):
        st, gen = self.dr.poll(wait=True, timeout_us=-1)
        assert st == 1, st
        self.generation = gen
        self.X = self.X_pending
        self.since = self.since_pending
        self.build_pending = False

    def build_and_swap(self):
        self.start_build()
        self.swap()

    def oracle_corpus(self):
        """The oracle's corpus text for the next propose."""
        if not self.delta or self.ring is None:
            return self.X
        return O.corpus_text(self.X, self.ring.delta(self.since, self.delta))

    # steps -------------------------------------------------------------------
    def step(self, check_rows=None, check=True, check_state=False):
        sd = self.trace.next_step()
        if self.build_pending:
            self.swap()
        dev = self.dr.device
        sampled = torch.from_numpy(sd.sampled).to(dev)
        m = sd.finished.shape[0]
        fused = self.fused and self.ring is not None
        if fused:
            self.dr.step(self.tok, self.n, sampled, torch.from_numpy(sd.finished).to(dev),
                         torch.from_numpy(sd.ingest_starts).to(dev),
                         torch.from_numpy(sd.ingest_lengths).to(dev), out=self.out)
        else:
            self.dr.propose_with_update(self.tok, self.n, sampled, out=self.out)
        O.update_state(self.o_tok, self.o_n, sd.sampled, self.cfg.V)
        if check:
            orc = O.propose(self.p, self.o_tok, self.o_n, X=self.oracle_corpus(), rows=check_rows,
                            threads=THREADS)
            compare(self.out, orc, rows=check_rows, ctx="step %d" % self.trace.step_index)
            if self.p.fixed_length:
                invariants_fixed(self.out, self.cfg.k)
            else:
                invariants(self.out, self.cfg.k, self.p.min_prob)
        if check_state:
            assert np.array_equal(to_np(self.n), self.o_n)
            assert np.array_equal(to_np(self.tok), self.o_tok)
        if m:
            if self.ring is not None:
                if not fused:
                    rows_t = torch.from_numpy(sd.finished).to(dev)
                    self.dr.ingest(self.tok, rows_t, torch.from_numpy(sd.ingest_starts).to(dev),
                                   torch.from_numpy(sd.ingest_lengths).to(dev), num_tokens=self.n)
                self.ring.ingest(self.o_tok, sd.finished, sd.ingest_starts, sd.ingest_lengths,
                                 num_tokens=self.o_n)
                self.ingested_since_build += int(sd.ingest_lengths.sum())
            for i, b in enumerate(sd.finished):
                self.o_tok[b] = sd.reset_tokens[i]
                self.o_n[b] = sd.reset_n[i]
            idx = torch.from_numpy(sd.finished.astype(np.int64)).to(dev)
            self.tok[idx] = torch.from_numpy(sd.reset_tokens).to(dev)
            self.n[idx] = torch.from_numpy(sd.reset_n).to(dev)
            if self.row_index:  # new requests in these rows
                self.dr.reset_rows(self.tok, self.n, idx.to(torch.int32))
            if (self.ring is not None and not self.build_pending
                    and self.ingested_since_build >= self.cfg.rebuild_tokens):
                self.start_build()
        return sd

    def close(self):
        if self.build_pending:
            self.dr.poll(wait=True)
        self.dr.close()
