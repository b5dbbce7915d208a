"""The allocation-free suffix array entry point against the context one.

sgd_suffix_array_noalloc serves callers that cannot call cudaMalloc where
they need a suffix array (their own allocator owns the device memory, or an
allocation could fail or synchronise the device mid-work): it works in a
fixed device array of the library.  Its results must equal those of
sgd_suffix_array, which sorts in scratch the context allocated, on
consecutive calls (the fixed array keeps the previous call's contents).
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from model_free_suffix_gb300 import build
    build.build()
    from model_free_suffix_gb300 import SuffixDrafter, _lib
    from model_free_suffix_gb300 import workload as W
    return SuffixDrafter, _lib, W


def _noalloc(L, text, out):
    stream = torch.cuda.current_stream().cuda_stream
    return L.load().sgd_suffix_array_noalloc(ctypes.c_void_p(text.data_ptr()), text.shape[0],
                                            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_matches_context_suffix_array(env):
    SuffixDrafter, L, W = env
    cap = L.NOALLOC_MAX_TOKENS
    dr = SuffixDrafter(max_batch=1, seq_capacity=8, vocab_size=151936, corpus_capacity=cap)
    rng = np.random.default_rng(7)
    texts = [
        W.sa_corpus(cap, seed=3),                                          # full size
        np.concatenate([rng.integers(0, 3, 40000), [151936]]).astype(np.int32),  # long repeats
    ]
    for i, x in enumerate(texts):  # two calls in a row on the same fixed array
        t = torch.from_numpy(x).cuda()
        want = dr.suffix_array(t)
        got = torch.full_like(want, -7)
        assert _noalloc(L, t, got) == L.SGD_OK, "call %d" % i
        torch.cuda.synchronize()
        assert torch.equal(got, want), "call %d differs from sgd_suffix_array" % i
    dr.close()


def test_noalloc_rejects_too_long_and_handles_tiny(env):
    SuffixDrafter, L, W = env
    big = torch.zeros(L.NOALLOC_MAX_TOKENS + 1, dtype=torch.int32, device="cuda")
    out = torch.full_like(big, -7)
    assert _noalloc(L, big, out) == L.SGD_ETOOLARGE
    assert int((out == -7).sum()) == out.numel()  # nothing written
    one = torch.tensor([5], dtype=torch.int32, device="cuda")
    o1 = torch.full_like(one, -7)
    assert _noalloc(L, one, o1) == L.SGD_OK and o1.tolist() == [0]
