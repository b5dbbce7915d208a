"""Diagnostics the benchmark reads: per-row statistics and context memory.

sgd_set_row_stats makes the drafting kernel write, per row, the suffix-array
hits its corpus probe scanned, the occurrences that voted (c0), the draft cap
and the source.  They are checked against what the oracle fixes: the source
is the oracle's, the draft never exceeds the cap, c0 is at most R and the
score is an integer count sum over c0 (so score * c0 is an integer).
sgd_memory reports what sgd_create allocated.
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


@pytest.mark.parametrize("mode", [0, 2], ids=["one-launch", "two-launch"])
def test_row_stats_agree_with_the_drafts(mode):
    W, O, H = _mods()
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=4096)
    ls = H.Lockstep(cfg, seed=5, B=96, steps=6, corpus=1 << 18, drafter_over=dict(propose_mode=mode))
    ls.prefill(seed=5)
    stats = torch.full((96 * 4,), -9, dtype=torch.int32, device=ls.dr.device)
    ls.dr.set_row_stats(stats)
    seen_corpus = seen_gd = 0
    for _ in range(6):
        ls.step()  # (compares the drafts with the oracle's)
        st = stats.view(96, 4).cpu().numpy()
        mi = H.to_np(ls.out.match_info)
        nv = H.to_np(ls.out.num_valid)
        sc = H.to_np(ls.out.score).astype(np.float64)
        scanned, c0, cap, src = st[:, 0], st[:, 1], st[:, 2], st[:, 3] & 255
        gd = (st[:, 3] >> 12) & 1  # the corpus draft came from a gram draft (nothing scanned)
        assert ((st[:, 3] >> 8) & 15 == 0).all()  # (no row index: every row scanned)
        assert (gd[src != 2] == 0).all()
        assert np.array_equal(src, mi[:, 1])
        assert (nv <= cap).all() and (scanned >= 0).all()
        assert ((c0 >= 1) & (c0 <= cfg.R))[src > 0].all() and (c0[src == 0] == 0).all()
        assert (scanned >= c0)[(src == 2) & (gd == 0)].all()
        seen_gd += int(gd.sum())
        prod = sc * c0
        assert (np.abs(prod - np.round(prod)) < 1e-3).all()
        seen_corpus += int((src == 2).sum())
    assert seen_corpus > 0
    assert seen_gd > 0 or mode == 2  # (gram drafts serve the one-launch kernel)
    ls.dr.set_row_stats(None)
    ls.close()


def test_memory_reports_the_allocations():
    W, O, H = _mods()
    from model_free_suffix_gb300 import SuffixDrafter
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    C = 1 << 20
    dr = SuffixDrafter(max_batch=64, seq_capacity=1024, vocab_size=1000, corpus_capacity=C)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    dev, pinned = dr.memory()
    # ring + two snapshots of text, suffix array and 16-byte keys at least
    assert dev >= C * 4 * (1 + 2 * 6) and pinned > 0
    assert free0 - free1 >= 0.9 * dev
    dr.close()
