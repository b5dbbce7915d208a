"""Gram drafts (gram_drafts = 1, the default) against the oracle.

A row whose corpus match is a 2- or 3-gram with a large suffix-array
interval takes its corpus draft from a block built with the snapshot: the
vote over the gram's R most recent continuing ends to depth k, cut at the
row's cap.  The drafts must equal the oracle's whatever cuts them: the
factor and offset cap, the context room, the depth-sum cap, a higher
probability floor, and Model Runner V2 fixed-length drafts (no floor).
Row statistics show the blocks are used.
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
    # (name, drafter knobs, oracle knobs)
    ("default", {}, {}),
    ("off", dict(gram_drafts=0), {}),
    ("factor-offset", dict(max_spec_factor=(1, 2), max_spec_offset=1), dict(factor=(1, 2), offset=1)),
    ("min-prob", dict(min_token_prob=(3, 10)), dict(min_prob=(3, 10))),
    ("depth-sum-cap", dict(depth_sum_cap=True), dict(depth_sum_cap=True)),
    ("fixed-length", dict(draft_mode=1), dict(fixed_length=True)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_gram_drafts_lockstep(case):
    W, O, H = _mods()
    name, dover, pover = case
    cfg = dataclasses.replace(W.CONFIGS["c3"], rebuild_tokens=8192)
    ls = H.Lockstep(cfg, seed=21, B=128, steps=8, finish_frac=0.05, corpus=1 << 18, fused=True,
                    drafter_over=dover, param_over=pover)
    ls.prefill(seed=21)
    stats = torch.zeros(128 * 4, dtype=torch.int32, device=ls.dr.device)
    ls.dr.set_row_stats(stats)
    used = 0
    for _ in range(8):
        ls.step(check_state=True)
        used += int(((stats.view(128, 4)[:, 3].cpu().numpy() >> 12) & 1).sum())
    if name == "off":
        assert used == 0
    else:
        assert used > 0, "no row was drafted from a gram draft"
    assert ls.dr.get_error() == 0
    ls.close()
