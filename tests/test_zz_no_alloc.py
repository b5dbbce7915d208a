"""The allocation-free suffix array entry point.

sgd_suffix_array_noalloc serves callers that cannot call cudaMalloc where
they need a suffix array: a server whose own caching allocator owns the
device memory, code inside another framework's memory budget, or code for
which an allocation could fail or synchronise the device mid-work.  It sorts
in a fixed device array of the library instead of context scratch.

Its result must equal the CPU oracle's suffix array (a comparison sort of
every suffix) and the context entry point sgd_suffix_array, on consecutive
calls: the fixed array keeps the previous call's contents, so the second call
shows that nothing stale leaks into a result.  Suffix arrays are integer
permutations, so the comparison is exact.
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
    from oracle import oracle as O
    O.build()
    from model_free_suffix_gb300 import SuffixDrafter, _lib
    from model_free_suffix_gb300 import workload as W
    return SuffixDrafter, _lib, W, O


def _noalloc(L, text, out):
    stream = torch.cuda.current_stream().cuda_stream
    return L.load().sgd_suffix_array_noalloc(ctypes.c_void_p(text.data_ptr()), text.shape[0],
                                            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_matches_oracle_and_context_suffix_array(env):
    SuffixDrafter, L, W, O = env
    cap = L.NOALLOC_MAX_TOKENS
    dr = SuffixDrafter(max_batch=1, seq_capacity=8, vocab_size=151936, corpus_capacity=cap)
    rng = np.random.default_rng(7)
    texts = [
        W.sa_corpus(cap, seed=3),                                                # full size
        np.concatenate([rng.integers(0, 3, 40000), [151936]]).astype(np.int32),  # long repeats
    ]
    for i, x in enumerate(texts):  # two calls in a row on the same fixed array
        t = torch.from_numpy(x).cuda()
        got = torch.full_like(t, -7)
        assert _noalloc(L, t, got) == L.SGD_OK, "call %d" % i
        torch.cuda.synchronize()
        sa = got.cpu().numpy()
        assert np.array_equal(sa, O.suffix_array(x)), "call %d differs from the oracle" % i
        want = dr.suffix_array(t)
        assert torch.equal(got, want), "call %d differs from sgd_suffix_array" % i
    dr.close()


def test_noalloc_rejects_too_long_and_handles_tiny(env):
    SuffixDrafter, L, W, O = env
    big = torch.zeros(L.NOALLOC_MAX_TOKENS + 1, dtype=torch.int32, device="cuda")
    out = torch.full_like(big, -7)
    assert _noalloc(L, big, out) == L.SGD_ETOOLARGE
    assert int((out == -7).sum()) == out.numel()  # nothing written
    one = torch.tensor([5], dtype=torch.int32, device="cuda")
    o1 = torch.full_like(one, -7)
    assert _noalloc(L, one, o1) == L.SGD_OK and o1.tolist() == [0]
