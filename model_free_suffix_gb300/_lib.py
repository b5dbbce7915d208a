"""ctypes view of libsgd's C ABI (include/sgd.h).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsgd.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sgd.h")

SGD_OK = 0
SGD_OK_SWAPPED = 1
SGD_PENDING = 2
SGD_EINVAL = -1
SGD_ECUDA = -2
SGD_ENOMEM = -3
SGD_ETIMEDOUT = -4
SGD_EBUSY = -5
SGD_EBUILD = -6
SGD_ENOCORPUS = -7
SGD_ETOOLARGE = -8
SGD_EIO = -9
NOALLOC_MAX_TOKENS = 65536

ERR_SAMPLED_TOKEN = 0x1
ERR_NUM_TOKENS = 0x2
ERR_DOC_ARGS = 0x4
ERR_DOC_TOKEN = 0x8
ERR_DOC_TOO_LONG = 0x10
ERR_LOOKBACK = 0x20
ERR_INGEST_WAIT = 0x40

INJECT_NONE = 0
INJECT_BUILD_FAIL = 1
INJECT_BUILD_HANG = 2
INJECT_STEP_WAIT = 3


class SgdConfig(ctypes.Structure):
    _fields_ = [
        ("max_batch", ctypes.c_int32),
        ("seq_capacity", ctypes.c_int32),
        ("vocab_size", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("max_tree_depth", ctypes.c_int32),
        ("max_occurrences", ctypes.c_int32),
        ("max_sampled", ctypes.c_int32),
        ("spec_factor_num", ctypes.c_uint32),
        ("spec_factor_den", ctypes.c_uint32),
        ("spec_offset", ctypes.c_int32),
        ("min_prob_num", ctypes.c_uint32),
        ("min_prob_den", ctypes.c_uint32),
        ("depth_sum_cap", ctypes.c_int32),
        ("corpus_capacity", ctypes.c_int64),
        ("max_docs", ctypes.c_int32),
        ("max_ingest_docs", ctypes.c_int32),
        ("corpus_cand_cap", ctypes.c_int32),
        ("self_warps", ctypes.c_int32),
        ("corpus_records", ctypes.c_int32),
        ("corpus_gram_index", ctypes.c_int32),
        ("propose_mode", ctypes.c_int32),
        ("delta_capacity", ctypes.c_int64),
        ("draft_mode", ctypes.c_int32),
        ("select_by_score", ctypes.c_int32),
        ("num_backoff", ctypes.c_int32),
        ("row_index", ctypes.c_int32),
        ("gram_drafts", ctypes.c_int32),
    ]


class SgdBuildInfo(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_int64),
        ("rounds", ctypes.c_int32),
        ("passes", ctypes.c_int32),
        ("sorted_elems", ctypes.c_int64),
        ("pass_elems", ctypes.c_int64),
        ("model_bytes", ctypes.c_int64),
        ("ms", ctypes.c_double),
        ("pass_ms", ctypes.c_double),
        ("status", ctypes.c_int32),
    ]


class SgdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, strerror(status), status))


_lib = None


def load() -> ctypes.CDLL:
    """The in-tree libsgd.so; raises if it was not built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libsgd.so is missing: run `python -m model_free_suffix_gb300.build` "
                           "(the CUDA library is required; there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint64)
    sig = {
        "sgd_version": (ctypes.c_int, []),
        "sgd_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "sgd_config_default": (ctypes.c_int, [ctypes.POINTER(SgdConfig)]),
        "sgd_config_set_float": (ctypes.c_int, [ctypes.POINTER(SgdConfig), ctypes.c_double,
                                                ctypes.c_double]),
        "sgd_create": (ctypes.c_int, [ctypes.POINTER(SgdConfig), ctypes.c_int, ctypes.POINTER(P)]),
        "sgd_destroy": (ctypes.c_int, [P]),
        "sgd_update_state": (ctypes.c_int, [P, P, P, P, i32, i32, P]),
        "sgd_propose": (ctypes.c_int, [P, P, P, P, i32, P, P, P, P, P, P]),
        "sgd_propose_with_update": (ctypes.c_int, [P, P, P, P, i32, P, i32, P, P, P, P, P, P]),
        "sgd_ingest": (ctypes.c_int, [P, P, P, i32, P, P, P, i32, P]),
        "sgd_step": (ctypes.c_int, [P, P, P, P, i32, P, i32, P, P, P, P, P, P, P, P, i32, P]),
        "sgd_step_host": (ctypes.c_int, [P, P, P, P, i32, i32, P, P, P, i32, P, P, P, P, P, P]),
        "sgd_build_sa": (ctypes.c_int, [P, P, P]),
        "sgd_poll": (ctypes.c_int, [P, ctypes.c_int, i64, P, u64p]),
        "sgd_suffix_array": (ctypes.c_int, [P, P, i64, P, P]),
        "sgd_suffix_array_noalloc": (ctypes.c_int, [P, i64, P, P]),
        "sgd_get_error": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
        "sgd_export_snapshot": (ctypes.c_int, [P, P, P, i64, ctypes.POINTER(ctypes.c_int64), u64p]),
        "sgd_save": (ctypes.c_int, [P, ctypes.c_char_p, P]),
        "sgd_load": (ctypes.c_int, [P, ctypes.c_char_p, P]),
        "sgd_corpus_stats": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_int64),
                                            ctypes.POINTER(ctypes.c_int32)]),
        "sgd_build_stats": (ctypes.c_int, [P, ctypes.POINTER(SgdBuildInfo)]),
        "sgd_debug_inject": (ctypes.c_int, [P, ctypes.c_int]),
        "sgd_launch_count": (ctypes.c_int, [P, u64p]),
        "sgd_set_row_stats": (ctypes.c_int, [P, P]),
        "sgd_reset_rows": (ctypes.c_int, [P, P, P, P, i32, P]),
        "sgd_memory": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def strerror(status: int) -> str:
    try:
        return load().sgd_strerror(int(status)).decode()
    except Exception:  # library missing: still describe the code
        return "status %d" % status


def header_functions(path: str = HEADER):
    """Names of the functions declared in include/sgd.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgd_[a-z_0-9]+)\s*\(", text)))
