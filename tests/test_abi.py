"""The C-ABI library builds, loads and exports every symbol include/sgd.h declares.

No compute call is made here (there may be no GPU).
"""
import ctypes

import pytest


@pytest.fixture(scope="module")
def lib():
    from model_free_suffix_gb300 import build as B
    B.build()
    from model_free_suffix_gb300 import _lib as L
    return L


def test_exports_every_declared_function(lib):
    L = lib.load()
    names = lib.header_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_config_defaults(lib):
    L = lib.load()
    c = lib.SgdConfig()
    assert L.sgd_config_default(ctypes.byref(c)) == 0
    assert (c.k, c.max_tree_depth, c.max_occurrences) == (16, 24, 64)
    assert (c.spec_factor_num, c.spec_factor_den) == (1, 1)
    assert (c.min_prob_num, c.min_prob_den) == (1, 10)
    assert c.corpus_capacity == 1 << 20
    assert c.delta_capacity == 0  # newly ingested docs wait for the next swap
    assert c.draft_mode == 0      # drafts stop at the probability floor and the factor cap
    assert c.num_backoff == 1     # one candidate length per path: the longest match
    assert c.row_index == 0       # rows scanned each step unless the caller opts in
    assert c.gram_drafts == 1     # frequent 2/3-gram votes built with each snapshot


def test_config_set_float_rationals(lib):
    L = lib.load()
    c = lib.SgdConfig()
    L.sgd_config_default(ctypes.byref(c))
    assert L.sgd_config_set_float(ctypes.byref(c), 2.0, 0.1) == 0
    assert (c.spec_factor_num, c.spec_factor_den) == (2, 1)
    assert (c.min_prob_num, c.min_prob_den) == (1, 10)
    assert L.sgd_config_set_float(ctypes.byref(c), 1.5, 0.25) == 0
    assert (c.spec_factor_num, c.spec_factor_den) == (3, 2)
    assert (c.min_prob_num, c.min_prob_den) == (1, 4)
    assert L.sgd_config_set_float(ctypes.byref(c), -1.0, 0.1) == lib.SGD_EINVAL
    assert L.sgd_config_set_float(ctypes.byref(c), 1.0, 1.5) == lib.SGD_EINVAL


def test_strerror_and_null_args(lib):
    L = lib.load()
    assert L.sgd_strerror(lib.SGD_EBUSY).decode().startswith("a suffix-array build")
    assert L.sgd_destroy(None) == lib.SGD_EINVAL
    assert L.sgd_propose(None, None, None, None, 0, None, None, None, None, None, None) == lib.SGD_EINVAL
    h = ctypes.c_void_p()
    assert L.sgd_create(None, 0, ctypes.byref(h)) == lib.SGD_EINVAL


def test_create_rejects_bad_knobs_before_touching_the_gpu(lib):
    L = lib.load()
    bad = [("seq_capacity", 4098), ("k", 0), ("k", 65), ("max_tree_depth", 129),
           ("max_occurrences", 0), ("corpus_cand_cap", 100), ("corpus_cand_cap", 32),
           ("min_prob_den", 0), ("self_warps", 17), ("draft_mode", 2), ("draft_mode", -1),
           ("select_by_score", 2), ("num_backoff", 0), ("num_backoff", 9), ("row_index", 2),
           ("row_index", -1), ("gram_drafts", 2), ("gram_drafts", -1)]
    for field, val in bad:
        c = lib.SgdConfig()
        L.sgd_config_default(ctypes.byref(c))
        setattr(c, field, val)
        h = ctypes.c_void_p()
        assert L.sgd_create(ctypes.byref(c), 0, ctypes.byref(h)) == lib.SGD_EINVAL, field
    # row indexes: not with the two-launch mode, a delta, score-ranked selection,
    # backoff (they need every end's length) or ids of 2^24 and more
    for over in [dict(propose_mode=2), dict(delta_capacity=1024), dict(select_by_score=1),
                 dict(num_backoff=2), dict(vocab_size=(1 << 24) + 1)]:
        c = lib.SgdConfig()
        L.sgd_config_default(ctypes.byref(c))
        c.row_index = 1
        for f, v in over.items():
            setattr(c, f, v)
        h = ctypes.c_void_p()
        assert L.sgd_create(ctypes.byref(c), 0, ctypes.byref(h)) == lib.SGD_EINVAL, over
    # the delta: within the ring, and the ring a whole number of 128-token windows
    for cap, dcap in [(1 << 20, -1), (1 << 20, (1 << 20) + 1), (1000, 64), (0, 128)]:
        c = lib.SgdConfig()
        L.sgd_config_default(ctypes.byref(c))
        c.corpus_capacity, c.delta_capacity = cap, dcap
        h = ctypes.c_void_p()
        assert L.sgd_create(ctypes.byref(c), 0, ctypes.byref(h)) == lib.SGD_EINVAL, (cap, dcap)


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from model_free_suffix_gb300 import _lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        L.load()
