"""Python face of libsgd: torch tensors in, torch tensors out.

Every method marshals pointers and sizes and calls one C entry point of
include/sgd.h; all work runs in the library's CUDA kernels on the given
stream.  PyTorch only provides device memory and streams.

Mirrors the drafter surface described on the "SuffixGPU" PyPI page
(Quickstart): a constructor with k, enable_global (here: corpus_capacity > 0),
max_spec_factor and min_token_prob; propose_with_update, propose with a mask,
harvest_finished (here: ingest) and poll.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from fractions import Fraction
from typing import Optional, Tuple, Union

import torch

from . import _lib as L

Rational = Union[float, Tuple[int, int]]


def _rational(x: Rational, denom: int = 10 ** 6) -> Tuple[int, int]:
    if isinstance(x, tuple):
        return int(x[0]), int(x[1])
    f = Fraction(int(round(float(x) * denom)), denom)
    return f.numerator, f.denominator


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class Proposal:
    drafts: torch.Tensor       # [B, k] int32, -1 padded
    num_valid: torch.Tensor    # [B] int32
    score: torch.Tensor        # [B] float32
    probs: torch.Tensor        # [B, k] float32
    match_info: torch.Tensor   # [B, 2] int32: {match length, source (0 none, 1 self, 2 corpus)}


class SuffixDrafter:
    """One libsgd context on one GPU.

    The knobs are those of sgd_config in include/sgd.h, where each is
    documented; the ones that change what is drafted: max_spec_factor,
    max_spec_offset, min_token_prob, depth_sum_cap, delta_capacity (docs not
    yet indexed are matched too), draft_mode (1: Model Runner V2 fixed-length
    drafts), select_by_score (1: the better score wins between the row's and
    the corpus's candidates) and num_backoff (2..8: multi-length backoff).
    The others choose between equivalent forms of the same computation.
    """

    def __init__(self, max_batch: int, seq_capacity: int, vocab_size: int, k: int = 16,
                 max_tree_depth: int = 24, max_occurrences: int = 64, max_sampled: Optional[int] = None,
                 max_spec_factor: Rational = 1.0, max_spec_offset: int = 0,
                 min_token_prob: Rational = 0.1, depth_sum_cap: bool = False,
                 corpus_capacity: int = 0, max_docs: int = 65536, max_ingest_docs: int = 4096,
                 corpus_cand_cap: int = 2048, self_warps: int = 0, corpus_records: int = 1,
                 corpus_gram_index: int = 1, propose_mode: int = 0, delta_capacity: int = 0,
                 draft_mode: int = 0, select_by_score: int = 0, num_backoff: int = 1,
                 row_index: int = 0, gram_drafts: int = 1, device: int = 0):
        self._lib = L.load()
        cfg = L.SgdConfig()
        self._check(self._lib.sgd_config_default(ctypes.byref(cfg)), "sgd_config_default")
        cfg.max_batch = max_batch
        cfg.seq_capacity = seq_capacity
        cfg.vocab_size = vocab_size
        cfg.k = k
        cfg.max_tree_depth = max_tree_depth
        cfg.max_occurrences = max_occurrences
        cfg.max_sampled = max_sampled if max_sampled is not None else k + 1
        cfg.spec_factor_num, cfg.spec_factor_den = _rational(max_spec_factor)
        cfg.spec_offset = max_spec_offset
        cfg.min_prob_num, cfg.min_prob_den = _rational(min_token_prob)
        cfg.depth_sum_cap = int(bool(depth_sum_cap))
        cfg.corpus_capacity = corpus_capacity
        cfg.max_docs = max_docs
        cfg.max_ingest_docs = max_ingest_docs
        cfg.corpus_cand_cap = corpus_cand_cap
        cfg.self_warps = self_warps
        cfg.corpus_records = corpus_records
        cfg.corpus_gram_index = corpus_gram_index
        cfg.propose_mode = propose_mode
        cfg.delta_capacity = delta_capacity
        cfg.draft_mode = draft_mode
        cfg.select_by_score = select_by_score
        cfg.num_backoff = num_backoff
        cfg.row_index = row_index
        cfg.gram_drafts = gram_drafts
        self.cfg = cfg
        self.device = torch.device("cuda", device)
        torch.cuda.init()
        with torch.cuda.device(self.device):
            torch.zeros(1, device=self.device)  # make the primary context current
            h = ctypes.c_void_p()
            self._check(self._lib.sgd_create(ctypes.byref(cfg), device, ctypes.byref(h)), "sgd_create")
        self._h = h
        self.k = k
        self.S = seq_capacity
        self.V = vocab_size
        self.max_batch = max_batch

    # -- helpers ------------------------------------------------------------
    @staticmethod
    def _check(status: int, where: str) -> int:
        if status < 0:
            raise L.SgdError(status, where)
        return status

    def _t(self, t: Optional[torch.Tensor], dtype=torch.int32, name="tensor") -> ctypes.c_void_p:
        if t is None:
            return ctypes.c_void_p(0)
        if t.device != self.device:
            raise ValueError("%s must be on %s" % (name, self.device))
        if t.dtype != dtype or not t.is_contiguous():
            raise ValueError("%s must be a contiguous %s tensor" % (name, dtype))
        return ctypes.c_void_p(t.data_ptr())

    @staticmethod
    def _host(t: Optional[torch.Tensor], dtype=torch.int32, name="tensor") -> ctypes.c_void_p:
        """A host (CPU) tensor's address; pinned memory keeps the copies asynchronous."""
        if t is None:
            return ctypes.c_void_p(0)
        if t.is_cuda:
            raise ValueError("%s must be a host (CPU) tensor" % name)
        if t.dtype != dtype or not t.is_contiguous():
            raise ValueError("%s must be a contiguous %s tensor" % (name, dtype))
        return ctypes.c_void_p(t.data_ptr())

    def new_outputs(self, B: int) -> Proposal:
        d = self.device
        return Proposal(torch.empty((B, self.k), dtype=torch.int32, device=d),
                        torch.empty(B, dtype=torch.int32, device=d),
                        torch.empty(B, dtype=torch.float32, device=d),
                        torch.empty((B, self.k), dtype=torch.float32, device=d),
                        torch.empty((B, 2), dtype=torch.int32, device=d))

    # -- drafting -----------------------------------------------------------
    def update_state(self, token_ids: torch.Tensor, num_tokens: torch.Tensor, sampled: torch.Tensor,
                     stream=None) -> None:
        B, T = sampled.shape
        self._check(self._lib.sgd_update_state(self._h, self._t(token_ids, name="token_ids"),
                                               self._t(num_tokens, name="num_tokens"),
                                               self._t(sampled, name="sampled"), B, T,
                                               _stream_handle(stream)), "sgd_update_state")

    def propose(self, token_ids: torch.Tensor, num_tokens: torch.Tensor,
                active: Optional[torch.Tensor] = None, out: Optional[Proposal] = None,
                stream=None) -> Proposal:
        B = num_tokens.shape[0]
        out = out or self.new_outputs(B)
        self._check(self._lib.sgd_propose(
            self._h, self._t(token_ids, name="token_ids"), self._t(num_tokens, name="num_tokens"),
            self._t(active, torch.uint8, "active"), B, self._t(out.drafts), self._t(out.num_valid),
            self._t(out.score, torch.float32), self._t(out.probs, torch.float32),
            self._t(out.match_info), _stream_handle(stream)), "sgd_propose")
        return out

    def propose_with_update(self, token_ids: torch.Tensor, num_tokens: torch.Tensor,
                            sampled: torch.Tensor, active: Optional[torch.Tensor] = None,
                            out: Optional[Proposal] = None, stream=None) -> Proposal:
        B, T = sampled.shape
        out = out or self.new_outputs(B)
        self._check(self._lib.sgd_propose_with_update(
            self._h, self._t(token_ids, name="token_ids"), self._t(num_tokens, name="num_tokens"),
            self._t(sampled, name="sampled"), T, self._t(active, torch.uint8, "active"), B,
            self._t(out.drafts), self._t(out.num_valid), self._t(out.score, torch.float32),
            self._t(out.probs, torch.float32), self._t(out.match_info), _stream_handle(stream)),
            "sgd_propose_with_update")
        return out

    def step(self, token_ids: torch.Tensor, num_tokens: torch.Tensor, sampled: torch.Tensor,
             rows: torch.Tensor, starts: torch.Tensor, lengths: torch.Tensor,
             active: Optional[torch.Tensor] = None, out: Optional[Proposal] = None,
             stream=None) -> Proposal:
        """propose_with_update, then ingest of the docs (rows, starts, lengths)
        read after the update: one kernel launch for up to 64 docs."""
        B, T = sampled.shape
        m = rows.shape[0]
        out = out or self.new_outputs(B)
        self._check(self._lib.sgd_step(
            self._h, self._t(token_ids, name="token_ids"), self._t(num_tokens, name="num_tokens"),
            self._t(sampled, name="sampled"), T, self._t(active, torch.uint8, "active"), B,
            self._t(out.drafts), self._t(out.num_valid), self._t(out.score, torch.float32),
            self._t(out.probs, torch.float32), self._t(out.match_info),
            self._t(rows, name="rows"), self._t(starts, name="starts"),
            self._t(lengths, name="lengths"), m, _stream_handle(stream)), "sgd_step")
        return out

    def step_host(self, token_ids: torch.Tensor, num_tokens: torch.Tensor, h_sampled: torch.Tensor,
                  h_rows: torch.Tensor, h_starts: torch.Tensor, h_lengths: torch.Tensor,
                  h_drafts: torch.Tensor, h_num_valid: torch.Tensor,
                  h_score: Optional[torch.Tensor] = None, h_probs: Optional[torch.Tensor] = None,
                  h_match_info: Optional[torch.Tensor] = None, stream=None) -> None:
        """step() with the step's inputs and outputs in host memory (pinned CPU
        tensors): the copies, the fused launch and the read-back are queued on
        `stream`; the host outputs are valid once that stream is synchronised."""
        B, T = h_sampled.shape
        m = h_rows.shape[0]
        H = self._host
        self._check(self._lib.sgd_step_host(
            self._h, self._t(token_ids, name="token_ids"), self._t(num_tokens, name="num_tokens"),
            H(h_sampled, name="h_sampled"), T, B, H(h_rows, name="h_rows"),
            H(h_starts, name="h_starts"), H(h_lengths, name="h_lengths"), m,
            H(h_drafts, name="h_drafts"), H(h_num_valid, name="h_num_valid"),
            H(h_score, torch.float32, "h_score"), H(h_probs, torch.float32, "h_probs"),
            H(h_match_info, name="h_match_info"), _stream_handle(stream)), "sgd_step_host")

    def bind_step_host(self, token_ids: torch.Tensor, num_tokens: torch.Tensor,
                       h_sampled: torch.Tensor, h_rows: torch.Tensor, h_starts: torch.Tensor,
                       h_lengths: torch.Tensor, h_drafts: torch.Tensor, h_num_valid: torch.Tensor,
                       h_score: Optional[torch.Tensor] = None, h_probs: Optional[torch.Tensor] = None,
                       h_match_info: Optional[torch.Tensor] = None, stream=None):
        """step_host on fixed buffers, with its arguments checked and marshalled
        once: the returned function queues one step per call (new inputs are
        written into the same host buffers between calls)."""
        B, T = h_sampled.shape
        H = self._host
        fn = self._lib.sgd_step_host
        args = (self._h, self._t(token_ids, name="token_ids"), self._t(num_tokens, name="num_tokens"),
                H(h_sampled, name="h_sampled"), T, B, H(h_rows, name="h_rows"),
                H(h_starts, name="h_starts"), H(h_lengths, name="h_lengths"), h_rows.shape[0],
                H(h_drafts, name="h_drafts"), H(h_num_valid, name="h_num_valid"),
                H(h_score, torch.float32, "h_score"), H(h_probs, torch.float32, "h_probs"),
                H(h_match_info, name="h_match_info"), _stream_handle(stream))
        keep = (token_ids, num_tokens, h_sampled, h_rows, h_starts, h_lengths, h_drafts, h_num_valid,
                h_score, h_probs, h_match_info)  # the buffers outlive the bound call

        def step_bound(_fn=fn, _args=args, _keep=keep):
            st = _fn(*_args)
            if st < 0:
                raise L.SgdError(st, "sgd_step_host")

        return step_bound

    # -- corpus ---------------------------------------------------------------
    def ingest(self, token_ids: torch.Tensor, rows: torch.Tensor, starts: torch.Tensor,
               lengths: torch.Tensor, num_tokens: Optional[torch.Tensor] = None, stream=None) -> None:
        B = token_ids.shape[0]
        m = rows.shape[0]
        self._check(self._lib.sgd_ingest(
            self._h, self._t(token_ids, name="token_ids"), self._t(num_tokens, name="num_tokens"), B,
            self._t(rows, name="rows"), self._t(starts, name="starts"), self._t(lengths, name="lengths"),
            m, _stream_handle(stream)), "sgd_ingest")

    harvest_finished = ingest

    def build_sa(self, side_stream, stream=None) -> int:
        return self._check(self._lib.sgd_build_sa(self._h, _stream_handle(stream),
                                                  _stream_handle(side_stream)), "sgd_build_sa")

    def try_build_sa(self, side_stream, stream=None) -> int:
        """Like build_sa but returns SGD_EBUSY instead of raising."""
        st = self._lib.sgd_build_sa(self._h, _stream_handle(stream), _stream_handle(side_stream))
        if st < 0 and st != L.SGD_EBUSY:
            raise L.SgdError(st, "sgd_build_sa")
        return st

    def poll(self, wait: bool = False, timeout_us: int = -1, stream=None,
             raise_on_error: bool = True) -> Tuple[int, int]:
        gen = ctypes.c_uint64()
        st = self._lib.sgd_poll(self._h, int(bool(wait)), int(timeout_us), _stream_handle(stream),
                                ctypes.byref(gen))
        if st < 0 and raise_on_error and st not in (L.SGD_ETIMEDOUT, L.SGD_EBUILD):
            raise L.SgdError(st, "sgd_poll")
        return st, int(gen.value)

    def suffix_array(self, text: torch.Tensor, out: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
        n = text.shape[0]
        out = out if out is not None else torch.empty(n, dtype=torch.int32, device=self.device)
        self._check(self._lib.sgd_suffix_array(self._h, self._t(text, name="text"), n,
                                               self._t(out, name="sa"), _stream_handle(stream)),
                    "sgd_suffix_array")
        return out

    def export_snapshot(self) -> Tuple[torch.Tensor, torch.Tensor, int]:
        n = ctypes.c_int64()
        gen = ctypes.c_uint64()
        cap = int(self.cfg.corpus_capacity)
        text = torch.empty(max(cap, 1), dtype=torch.int32, device=self.device)
        sa = torch.empty(max(cap, 1), dtype=torch.int32, device=self.device)
        self._check(self._lib.sgd_export_snapshot(self._h, self._t(text), self._t(sa), cap,
                                                  ctypes.byref(n), ctypes.byref(gen)),
                    "sgd_export_snapshot")
        return text[:n.value].clone(), sa[:n.value].clone(), int(gen.value)

    def corpus_stats(self) -> Tuple[int, int]:
        live = ctypes.c_int64()
        nd = ctypes.c_int32()
        self._check(self._lib.sgd_corpus_stats(self._h, ctypes.byref(live), ctypes.byref(nd)),
                    "sgd_corpus_stats")
        return int(live.value), int(nd.value)

    def save(self, path: str, stream=None) -> None:
        """Writes the corpus (ring, document FIFO, current snapshot) to `path`
        once the work queued on `stream` is done."""
        self._check(self._lib.sgd_save(self._h, os.fsencode(path), _stream_handle(stream)),
                    "sgd_save")

    def load(self, path: str, stream=None) -> None:
        """Replaces the corpus with a saved one and rebuilds its index (on
        `stream`, waited for): the context then drafts as the saved one did."""
        self._check(self._lib.sgd_load(self._h, os.fsencode(path), _stream_handle(stream)),
                    "sgd_load")

    def build_stats(self) -> dict:
        info = L.SgdBuildInfo()
        self._check(self._lib.sgd_build_stats(self._h, ctypes.byref(info)), "sgd_build_stats")
        return {f: getattr(info, f) for f, _ in L.SgdBuildInfo._fields_}

    # -- diagnostics ------------------------------------------------------------
    def get_error(self, clear: bool = False) -> int:
        f = ctypes.c_uint32()
        self._check(self._lib.sgd_get_error(self._h, ctypes.byref(f), int(bool(clear))), "sgd_get_error")
        return int(f.value)

    def debug_inject(self, what: int) -> None:
        self._check(self._lib.sgd_debug_inject(self._h, int(what)), "sgd_debug_inject")

    def reset_rows(self, token_ids: torch.Tensor, num_tokens: torch.Tensor, rows: torch.Tensor,
                   stream=None) -> None:
        """Rebuilds the bigram position index of the listed rows from their
        current contents (row_index=1; no-op otherwise).  Call it for every
        row written other than through the library's updates."""
        self._check(self._lib.sgd_reset_rows(self._h, self._t(token_ids), self._t(num_tokens),
                                             self._t(rows, name="rows"), rows.shape[0],
                                             _stream_handle(stream)),
                    "sgd_reset_rows")

    def set_row_stats(self, row_stats: Optional[torch.Tensor]) -> None:
        """Per-row statistics of later drafting launches into `row_stats`
        (int32 [max_batch, 4] on the device: hits scanned, c0, cap, source),
        or None to stop.  The tensor must outlive the launches (and graphs)
        that write it."""
        if row_stats is not None:
            assert row_stats.dtype == torch.int32 and row_stats.is_cuda and row_stats.is_contiguous()
            assert row_stats.numel() >= 4 * self.cfg.max_batch
        self._row_stats = row_stats
        self._check(self._lib.sgd_set_row_stats(
            self._h, ctypes.c_void_p(row_stats.data_ptr() if row_stats is not None else 0)),
            "sgd_set_row_stats")

    def memory(self) -> Tuple[int, int]:
        """(device bytes, page-locked host bytes) the context allocated."""
        d, h = ctypes.c_int64(), ctypes.c_int64()
        self._check(self._lib.sgd_memory(self._h, ctypes.byref(d), ctypes.byref(h)), "sgd_memory")
        return int(d.value), int(h.value)

    def launch_count(self) -> int:
        c = ctypes.c_uint64()
        self._check(self._lib.sgd_launch_count(self._h, ctypes.byref(c)), "sgd_launch_count")
        return int(c.value)

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.sgd_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
