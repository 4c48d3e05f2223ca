"""GB300 (sm_103a) DSA hot path: Lightning Indexer → Top-K → sparse MLA attention.

A thin binding over libdsa.so (include/dsa.h).  Functions take CUDA tensors,
check their dtypes and shapes, and pass raw pointers plus the current CUDA
stream to the library; every step of the computation runs in the library's
kernels.  There is no CPU or framework fallback: if the library is missing,
calls raise.

Names follow the C ABI: indexer_scores, topk, fused_indexer, sparse_mla_attn,
fused_forward.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence, Tuple

import torch

from . import _abi
from ._abi import STATUS_BYTES, DsaError, lib  # noqa: F401

__all__ = ["Problem", "Workspace", "indexer_scores", "topk", "fused_indexer", "sparse_mla_attn",
           "fused_forward", "indexer_prolog", "DsaError", "lib", "trace"]

_DT = {torch.float32: _abi.DSA_F32, torch.bfloat16: _abi.DSA_BF16,
       torch.uint8: _abi.DSA_FP8_E4M3, torch.float8_e4m3fn: _abi.DSA_FP8_E4M3}
_NAME_DT = {"f32": _abi.DSA_F32, "bf16": _abi.DSA_BF16, "e4m3": _abi.DSA_FP8_E4M3,
            "mxfp8": _abi.DSA_MXFP8_E4M3}
_TORCH_OUT = {_abi.DSA_F32: torch.float32, _abi.DSA_BF16: torch.bfloat16}


def _dt(x) -> int:
    if isinstance(x, str):
        return _NAME_DT[x]
    if isinstance(x, int):
        return x
    return _DT[x]


class Problem:
    """Sizes, dtypes and device sequence offsets of one DSA problem (dsa_problem)."""

    def __init__(self, cu_q: torch.Tensor, cu_k: torch.Tensor, *, q_lens: Sequence[int],
                 k_lens: Sequence[int], h_idx: int, d_idx: int, h: int, d_c: int, d_rope: int,
                 top_k: int, idx_dtype, kv_dtype, out_dtype=None, sm_scale: float = 0.0,
                 block_table: Optional[torch.Tensor] = None, page_size: int = 0,
                 num_pages: int = 0):
        """block_table [B, max_pages] int32 (CUDA) with page_size > 0 and num_pages: the key
        caches (k_idx, kv, k_scale) are paged, num_pages * page_size rows; key position s of
        sequence b is row block_table[b, s // page_size] * page_size + s % page_size."""
        if not (cu_q.is_cuda and cu_k.is_cuda) or cu_q.dtype != torch.int32 \
                or cu_k.dtype != torch.int32:
            raise ValueError("cu_q/cu_k must be int32 CUDA tensors")
        self.cu_q, self.cu_k = cu_q.contiguous(), cu_k.contiguous()
        self.page_size, self.num_pages = int(page_size), int(num_pages)
        self.block_table = None
        if self.page_size:
            if block_table is None or not block_table.is_cuda or block_table.dtype != torch.int32 \
                    or block_table.dim() != 2 or block_table.shape[0] != len(q_lens):
                raise ValueError("paged caches need an int32 CUDA block_table [B, max_pages]")
            self.block_table = block_table.contiguous()
        self.q_lens, self.k_lens = list(q_lens), list(k_lens)
        self.h_idx, self.d_idx, self.h, self.d_c, self.d_rope = h_idx, d_idx, h, d_c, d_rope
        self.top_k = top_k
        self.idx_dtype, self.kv_dtype = _dt(idx_dtype), _dt(kv_dtype)
        self.out_dtype = _dt(out_dtype) if out_dtype is not None else self.kv_dtype
        self.sm_scale = float(sm_scale)
        self.c = _abi.DsaProblem(
            len(self.q_lens), sum(self.q_lens), sum(self.k_lens), max(self.q_lens, default=0),
            max(self.k_lens), h_idx, d_idx, h, d_c, d_rope, top_k, self.idx_dtype, self.kv_dtype,
            self.out_dtype, self.sm_scale, self.cu_q.data_ptr(), self.cu_k.data_ptr(),
            self.page_size, self.block_table.shape[1] if self.page_size else 0, self.num_pages,
            self.block_table.data_ptr() if self.page_size else None)

    @classmethod
    def from_config(cls, cfg, cu_q: torch.Tensor, cu_k: torch.Tensor, sm_scale: float = 0.0,
                    block_table: Optional[torch.Tensor] = None, page_size: int = 0,
                    num_pages: int = 0):
        return cls(cu_q, cu_k, q_lens=cfg.q_lens, k_lens=cfg.k_lens, h_idx=cfg.h_idx,
                   d_idx=cfg.d_idx, h=cfg.h, d_c=cfg.d_c, d_rope=cfg.d_rope, top_k=cfg.top_k,
                   idx_dtype=cfg.idx_dtype, kv_dtype=cfg.kv_dtype, out_dtype=cfg.out_dtype,
                   sm_scale=sm_scale, block_table=block_table, page_size=page_size,
                   num_pages=num_pages)

    @property
    def cache_rows(self) -> int:
        """Rows of the key caches (k_idx, kv, k_scale)."""
        return self.num_pages * self.page_size if self.page_size else self.total_k

    @property
    def total_q(self) -> int:
        return self.c.total_q

    @property
    def total_k(self) -> int:
        return self.c.total_k

    @property
    def max_k_len(self) -> int:
        return self.c.max_k_len

    @property
    def d(self) -> int:
        return self.d_c + self.d_rope

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale > 0 else 1.0 / math.sqrt(self.d)

    def workspace_size(self, op: int) -> int:
        n = ctypes.c_size_t(0)
        _abi.check(lib().dsa_workspace_size(ctypes.byref(self.c), op, ctypes.byref(n)))
        return n.value


class Workspace:
    """Caller-owned device scratch; its first 16384 bytes are the status block (the status
    word and the kernels' synchronisation counters, zero between calls)."""

    def __init__(self, device=None, nbytes: int = STATUS_BYTES):
        self.device = torch.device(device or "cuda")
        self.buf = torch.zeros(max(STATUS_BYTES, nbytes), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> "Workspace":
        if self.buf.numel() < nbytes:
            flags = self.buf[:STATUS_BYTES].clone()
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
            self.buf[:STATUS_BYTES].copy_(flags)
        return self

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    def clear_status(self) -> None:
        _abi.check(lib().dsa_clear_status(self.ptr, _stream(self.device)))

    def selftest_wait_timeout(self, limit_ns: int = 1_000_000) -> None:
        """Run the bounded-wait self-test: a wait on an mbarrier nothing arrives at gives up
        after limit_ns and sets DSA_FLAG_TIMEOUT in this workspace's status word."""
        _abi.check(lib().dsa_selftest_wait_timeout(self.ptr, int(limit_ns), _stream(self.device)))

    def status(self) -> int:
        """Synchronise the current stream and return the device status flags."""
        f = ctypes.c_uint32(0)
        rc = lib().dsa_read_status(self.ptr, _stream(self.device), ctypes.byref(f))
        if rc not in (_abi.DSA_OK, _abi.DSA_ERR_TIMEOUT):
            _abi.check(rc)
        return f.value


_default_ws = {}


def _workspace(ws: Optional[Workspace], device, nbytes: int) -> Workspace:
    if ws is None:
        key = torch.device(device).index
        ws = _default_ws.get(key)
        if ws is None:
            ws = _default_ws[key] = Workspace(device, nbytes)
    return ws.ensure(nbytes)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: Optional[torch.Tensor], name: str, dtype_code: Optional[int], shape: Tuple[int, ...],
          optional: bool = False) -> None:
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype_code is not None and _DT.get(t.dtype) != dtype_code:
        raise ValueError(f"{name} has dtype {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check_indexer(P: Problem, q_idx, k_idx, w, q_scale, k_scale):
    mx = P.idx_dtype == _abi.DSA_MXFP8_E4M3
    codes = _abi.DSA_FP8_E4M3 if mx else P.idx_dtype  # MXFP8 codes are E4M3 bytes
    _need(q_idx, "q_idx", codes, (P.total_q, P.h_idx, P.d_idx))
    _need(k_idx, "k_idx", codes, (P.cache_rows, P.d_idx))
    _need(w, "w", _abi.DSA_F32, (P.total_q, P.h_idx))
    if mx:  # E8M0 bytes, one per 32 elements
        _need(q_scale, "q_scale", _abi.DSA_FP8_E4M3, (P.total_q, P.h_idx, P.d_idx // 32))
        _need(k_scale, "k_scale", _abi.DSA_FP8_E4M3, (P.cache_rows, P.d_idx // 32))
        return
    fp8 = P.idx_dtype == _abi.DSA_FP8_E4M3
    _need(q_scale, "q_scale", _abi.DSA_F32, (P.total_q, P.h_idx), optional=not fp8)
    _need(k_scale, "k_scale", _abi.DSA_F32, (P.cache_rows,), optional=not fp8)


def _idx_out(P: Problem, idx, vals, device, want_vals: bool):
    if idx is None:
        idx = torch.empty(P.total_q, P.top_k, dtype=torch.int32, device=device)
    _need(idx, "idx", None, (P.total_q, P.top_k))
    if vals is None and want_vals:
        vals = torch.empty(P.total_q, P.top_k, dtype=torch.float32, device=device)
    _need(vals, "vals", _abi.DSA_F32, (P.total_q, P.top_k), optional=True)
    return idx, vals


def indexer_scores(P: Problem, q_idx, k_idx, w, q_scale=None, k_scale=None, scores=None,
                   ws: Optional[Workspace] = None) -> torch.Tensor:
    """scores[ΣT, max_k_len] (fp32, -inf past each query's position)."""
    _check_indexer(P, q_idx, k_idx, w, q_scale, k_scale)
    dev = k_idx.device
    if scores is None:
        scores = torch.empty(P.total_q, P.max_k_len, dtype=torch.float32, device=dev)
    _need(scores, "scores", _abi.DSA_F32, (P.total_q, scores.shape[1]))
    ws = _workspace(ws, dev, P.workspace_size(_abi.OP_INDEXER_SCORES))
    _abi.check(lib().dsa_indexer_scores(
        ctypes.byref(P.c), q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), _ptr(q_scale),
        _ptr(k_scale), scores.data_ptr(), scores.shape[1], ws.ptr, ws.nbytes, _stream(dev)))
    return scores


def topk(P: Problem, scores: torch.Tensor, idx=None, vals=None, want_vals: bool = False,
         ws: Optional[Workspace] = None):
    """(idx[ΣT, top_k] int32 ascending positions, -1 padded; vals or None)."""
    _need(scores, "scores", _abi.DSA_F32, (P.total_q, scores.shape[1]))
    dev = scores.device
    idx, vals = _idx_out(P, idx, vals, dev, want_vals)
    ws = _workspace(ws, dev, P.workspace_size(_abi.OP_TOPK))
    _abi.check(lib().dsa_topk(ctypes.byref(P.c), scores.data_ptr(), scores.shape[1],
                              idx.data_ptr(), _ptr(vals), ws.ptr, ws.nbytes, _stream(dev)))
    return idx, vals


def fused_indexer(P: Problem, q_idx, k_idx, w, q_scale=None, k_scale=None, idx=None, vals=None,
                  want_vals: bool = False, ws: Optional[Workspace] = None):
    """Scoring + head weighting + Top-K in one call: (idx, vals or None)."""
    _check_indexer(P, q_idx, k_idx, w, q_scale, k_scale)
    dev = k_idx.device
    idx, vals = _idx_out(P, idx, vals, dev, want_vals)
    ws = _workspace(ws, dev, P.workspace_size(_abi.OP_FUSED_INDEXER))
    _abi.check(lib().dsa_fused_indexer(
        ctypes.byref(P.c), q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), _ptr(q_scale),
        _ptr(k_scale), idx.data_ptr(), _ptr(vals), ws.ptr, ws.nbytes, _stream(dev)))
    return idx, vals


def indexer_prolog(q_proj=None, x=None, w_h=None, q_codes=None, q_scale=None, w=None):
    """Q quantisation and head-weight projection in one launch (dsa_indexer_prolog).

    q_proj [T, H_I, d_I] bf16 -> (q_codes [T, H_I, d_I] uint8 E4M3, q_scale [T, H_I] f32);
    x [T, d_model] bf16, w_h [H_I, d_model] bf16 -> w [T, H_I] f32.  Either part may be
    left out (None inputs).  Returns (q_codes, q_scale, w), None for a part not computed.
    """
    if q_proj is None and x is None:
        raise ValueError("indexer_prolog needs q_proj or (x, w_h)")
    if q_proj is not None:
        T, h, d = q_proj.shape
    else:
        T, h = x.shape[0], w_h.shape[0]
        d = 8
    dev = (q_proj if q_proj is not None else x).device
    d_model = 0
    if q_proj is not None:
        _need(q_proj, "q_proj", _abi.DSA_BF16, (T, h, d))
        if q_codes is None:
            q_codes = torch.empty((T, h, d), dtype=torch.uint8, device=dev)
        if q_scale is None:
            q_scale = torch.empty((T, h), dtype=torch.float32, device=dev)
        _need(q_codes, "q_codes", _abi.DSA_FP8_E4M3, (T, h, d))
        _need(q_scale, "q_scale", _abi.DSA_F32, (T, h))
    else:
        q_codes = q_scale = None
    if x is not None or w_h is not None:
        if x is None or w_h is None:
            raise ValueError("x and w_h go together")
        d_model = x.shape[1]
        _need(x, "x", _abi.DSA_BF16, (T, d_model))
        _need(w_h, "w_h", _abi.DSA_BF16, (h, d_model))
        if w is None:
            w = torch.empty((T, h), dtype=torch.float32, device=dev)
        _need(w, "w", _abi.DSA_F32, (T, h))
    else:
        w = None
    _abi.check(lib().dsa_indexer_prolog(T, h, d, d_model, _ptr(q_proj), _ptr(x), _ptr(w_h),
                                        _ptr(q_codes), _ptr(q_scale), _ptr(w), _stream(dev)))
    return q_codes, q_scale, w


def _attn_out(P: Problem, out, lse, device, want_lse: bool):
    if out is None:
        out = torch.empty(P.total_q, P.h, P.d_c, dtype=_TORCH_OUT[P.out_dtype], device=device)
    _need(out, "out", P.out_dtype, (P.total_q, P.h, P.d_c))
    if lse is None and want_lse:
        lse = torch.empty(P.total_q, P.h, dtype=torch.float32, device=device)
    _need(lse, "lse", _abi.DSA_F32, (P.total_q, P.h), optional=True)
    return out, lse


def sparse_mla_attn(P: Problem, q, kv, idx, out=None, lse=None, want_lse: bool = True,
                    ws: Optional[Workspace] = None):
    """Sparse attention over the latent rows idx selects: (out[ΣT, H, d_c], lse or None)."""
    _need(q, "q", P.kv_dtype, (P.total_q, P.h, P.d))
    _need(kv, "kv", P.kv_dtype, (P.cache_rows, P.d))
    _need(idx, "idx", None, (P.total_q, P.top_k))
    dev = kv.device
    out, lse = _attn_out(P, out, lse, dev, want_lse)
    ws = _workspace(ws, dev, P.workspace_size(_abi.OP_SPARSE_MLA_ATTN))
    _abi.check(lib().dsa_sparse_mla_attn(ctypes.byref(P.c), q.data_ptr(), kv.data_ptr(),
                                         idx.data_ptr(), out.data_ptr(), _ptr(lse), ws.ptr,
                                         ws.nbytes, _stream(dev)))
    return out, lse


def fused_forward(P: Problem, q_idx, k_idx, w, q, kv, q_scale=None, k_scale=None, out=None,
                  lse=None, idx=None, vals=None, want_lse: bool = True, want_idx: bool = True,
                  want_vals: bool = False, ws: Optional[Workspace] = None):
    """The DSA layer: fused indexer then sparse attention → (out, lse, idx, vals)."""
    _check_indexer(P, q_idx, k_idx, w, q_scale, k_scale)
    _need(q, "q", P.kv_dtype, (P.total_q, P.h, P.d))
    _need(kv, "kv", P.kv_dtype, (P.cache_rows, P.d))
    dev = kv.device
    out, lse = _attn_out(P, out, lse, dev, want_lse)
    if want_idx or idx is not None:
        idx, vals = _idx_out(P, idx, vals, dev, want_vals)
    elif want_vals or vals is not None:
        raise ValueError("vals needs idx")
    ws = _workspace(ws, dev, P.workspace_size(_abi.OP_FUSED_FORWARD))
    _abi.check(lib().dsa_fused_forward(
        ctypes.byref(P.c), q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), _ptr(q_scale),
        _ptr(k_scale), q.data_ptr(), kv.data_ptr(), out.data_ptr(), _ptr(lse), _ptr(idx),
        _ptr(vals), ws.ptr, ws.nbytes, _stream(dev)))
    return out, lse, idx, vals


class trace:
    """Context manager recording per-launch CUDA-event times of the library's kernels."""

    def __init__(self, capacity: int = 4096):
        self.capacity = capacity
        self.records = []

    def __enter__(self):
        _abi.check(lib().dsa_trace_begin(self.capacity))
        return self

    def __exit__(self, *exc):
        _abi.check(lib().dsa_trace_end())
        n = lib().dsa_trace_count()
        name = ctypes.create_string_buffer(128)
        ms = ctypes.c_float(0)
        self.records = []
        for i in range(n):
            _abi.check(lib().dsa_trace_get(i, name, 128, ctypes.byref(ms)))
            self.records.append((name.value.decode(), ms.value))
        return False
