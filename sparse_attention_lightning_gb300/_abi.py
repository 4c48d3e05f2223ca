"""ctypes declarations of libdsa.so (include/dsa.h).  Loading fails loudly."""
from __future__ import annotations

import contextlib
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")
CHECKED_LIB_PATH = os.path.join(_PKG, "libdsa_checked.so")  # -DDSA_CHECKED build

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_WORKSPACE, \
    DSA_ERR_TIMEOUT = range(6)
DSA_F32, DSA_BF16, DSA_FP8_E4M3, DSA_MXFP8_E4M3 = 0, 1, 2, 3
DSA_FLAG_BAD_INDEX, DSA_FLAG_BAD_SEQS, DSA_FLAG_TIMEOUT, DSA_FLAG_CHECK = 0x1, 0x2, 0x4, 0x8
OP_INDEXER_SCORES, OP_TOPK, OP_FUSED_INDEXER, OP_SPARSE_MLA_ATTN, OP_FUSED_FORWARD = 1, 2, 3, 4, 5

# Every symbol include/dsa.h declares.
EXPORTS = ("dsa_workspace_size", "dsa_indexer_scores", "dsa_topk", "dsa_fused_indexer",
           "dsa_sparse_mla_attn", "dsa_fused_forward", "dsa_clear_status", "dsa_read_status",
           "dsa_status_str", "dsa_last_error", "dsa_abi_version", "dsa_trace_begin",
           "dsa_trace_end", "dsa_trace_count", "dsa_trace_get", "dsa_fused_indexer_static",
           "dsa_selftest_wait_timeout", "dsa_indexer_prolog")


class DsaProblem(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("total_k", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("max_k_len", ctypes.c_int32), ("h_idx", ctypes.c_int32),
                ("d_idx", ctypes.c_int32), ("h", ctypes.c_int32), ("d_c", ctypes.c_int32),
                ("d_rope", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("idx_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("cu_q", ctypes.c_void_p), ("cu_k", ctypes.c_void_p),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("block_table", ctypes.c_void_p)]


ABI_VERSION = 4  # DSA_ABI_VERSION this binding is written for
STATUS_BYTES = 16384  # the workspace status block


class DsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dsa error {code}: {msg}")
        self.code = code


_lib = None
_path = LIB_PATH


@contextlib.contextmanager
def using(path: str):
    """Route every call of the binding through the library at ``path`` (e.g. the checked
    build) inside the ``with`` block."""
    global _lib, _path
    saved = (_lib, _path)
    _lib, _path = None, path
    try:
        yield lib()
    finally:
        _lib, _path = saved


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_path):
        raise ImportError(f"{_path} is missing: build it with "
                          "`python -m sparse_attention_lightning_gb300.build`")
    L = ctypes.CDLL(_path)
    P = ctypes.POINTER(DsaProblem)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "dsa_workspace_size": [P, ctypes.c_int, ctypes.POINTER(sz)],
        "dsa_indexer_scores": [P, vp, vp, vp, vp, vp, vp, i64, vp, sz, vp],
        "dsa_topk": [P, vp, i64, vp, vp, vp, sz, vp],
        "dsa_fused_indexer": [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "dsa_sparse_mla_attn": [P, vp, vp, vp, vp, vp, vp, sz, vp],
        "dsa_fused_forward": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
        "dsa_fused_indexer_static": [P, vp, vp, vp, vp, vp, vp, vp, vp, vp],
        "dsa_clear_status": [vp, vp],
        "dsa_selftest_wait_timeout": [vp, ctypes.c_uint64, vp],
        "dsa_indexer_prolog": [ctypes.c_int32] * 4 + [vp] * 7,
        "dsa_read_status": [vp, vp, ctypes.POINTER(ctypes.c_uint32)],
        "dsa_abi_version": [],
        "dsa_trace_begin": [ctypes.c_int],
        "dsa_trace_end": [],
        "dsa_trace_count": [],
        "dsa_trace_get": [ctypes.c_int, ctypes.c_char_p, ctypes.c_int,
                          ctypes.POINTER(ctypes.c_float)],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    for name in ("dsa_status_str", "dsa_last_error"):
        getattr(L, name).restype = ctypes.c_char_p
    L.dsa_status_str.argtypes = [ctypes.c_int]
    L.dsa_last_error.argtypes = []
    if L.dsa_abi_version() != ABI_VERSION:
        raise ImportError(f"{_path} has ABI version {L.dsa_abi_version()}, the binding "
                          f"expects {ABI_VERSION}: rebuild it")
    _lib = L
    return L


def check(code: int) -> None:
    if code != DSA_OK:
        raise DsaError(code, lib().dsa_last_error().decode() or lib().dsa_status_str(code).decode())
