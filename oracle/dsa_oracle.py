"""fp64 CPU oracle of the DSA hot path.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the bench's CPU-baseline leg may
import this module.  The CUDA library never calls it and shares no code with it.

It restates, in plain numpy fp64 and one query row at a time, what the DSA
layer computes:

1. Lightning-Indexer relevance scoring and head-weighted summation
   ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
   LLMs", §4.1 Indexer Fusion: batched dot of the indexer query with the K cache,
   then a weighted sum over heads; §2.2: the indexer scores each historical
   position).  The score is
       I[t, s] = Σ_j w[t, j] · ReLU(q_I[t, j, :] · k_I[s, :]),   0 <= s <= pos(t)
   (ReLU and the weight form are the DSA indexer definition; the pages give the
   dot → weighted-sum order.)  FP8 inputs are dequantised exactly first:
   q_I[t, j, :] = code · q_scale[t, j], k_I[s, :] = code · k_scale[s].
   MXFP8 inputs ("… New-Architecture LLMs" §5.1 Index Path: Fully Quantized with
   MXFP8 Per-Group; "Optimizing LLM Inference for New Architectures", §4: one
   scale per 32 elements) carry one E8M0 scale (2^(e − 127)) per 32 consecutive
   elements of a query head or a key:
   q_I[t, j, c] = code · 2^(q_scale[t, j, c/32] − 127),
   k_I[s, c] = code · 2^(k_scale[s, c/32] − 127).
2. Causal Top-K ("… New-Architecture LLMs" §4.1 and §6.2: index computation is
   causal, later positions see a longer history): the min(k, pos+1) positions
   with the largest I, ties broken toward the smaller position.
3. Sparse Flash Attention over the MLA latent cache at the selected positions
   ("… New-Architecture LLMs" §2.2 and §4.1; "Day0 Inference Adaptation … on
   Ascend" §4: SFA reads the KV cache at the position set the indexer outputs):
       S_i = scale · q[t, h, :] · kv[sel_i, :]          (all D = d_c + d_rope columns)
       out[t, h, :] = Σ_i softmax(S)_i · kv[sel_i, :d_c] (value = latent columns)
       lse[t, h] = log Σ_i exp(S_i)
   with scale = 1/sqrt(D) unless given.

Positions are local to a sequence: the queries of sequence b are its last T_b
tokens, so query i of sequence b sits at pos = L_b − T_b + i.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# Exact decoding of the stored element types into fp64.


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32: widen the bits, then to fp64."""
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 (the 'fn' variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.

    exponent 0 is subnormal (m/8 · 2^-6); S.1111.111 is NaN; no infinities.
    """
    c = np.ascontiguousarray(codes).view(np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def e8m0_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP E8M0 scale (the MX formats' shared scale): 2^(code − 127); 255 is NaN."""
    c = np.ascontiguousarray(codes).view(np.uint8).astype(np.float64)
    return np.where(c == 255, np.nan, np.exp2(c - 127.0))


def mx_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 codes [..., n] with one E8M0 scale per 32 consecutive elements [..., n/32]."""
    v = e4m3_to_f64(codes)
    s = e8m0_to_f64(scales)
    return v * np.repeat(s, 32, axis=-1)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Decode an array stored as 'f32' (float32), 'bf16' (uint16/int16 bits) or 'e4m3' (uint8 codes)."""
    if dtype == "f32":
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_to_f64(arr)
    if dtype in ("e4m3", "mxfp8"):
        return e4m3_to_f64(arr)
    if dtype == "f64":
        return np.asarray(arr, dtype=np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Positions.


def query_rows(cu_q: Sequence[int], cu_k: Sequence[int]) -> List[Tuple[int, int, int]]:
    """(packed row t, sequence b, position pos(t)) for every query row."""
    rows = []
    for b in range(len(cu_q) - 1):
        T = int(cu_q[b + 1]) - int(cu_q[b])
        L = int(cu_k[b + 1]) - int(cu_k[b])
        for i in range(T):
            rows.append((int(cu_q[b]) + i, b, L - T + i))
    return rows


# ---------------------------------------------------------------------------
# The three steps, one query row at a time.


def indexer_row(q_idx_t: np.ndarray, k_idx_b: np.ndarray, w_t: np.ndarray, pos: int) -> np.ndarray:
    """I[s] for s = 0..pos: Σ_j w[j] · max(0, q_I[j]·k_I[s]).

    q_idx_t [H_I, d_I], k_idx_b [L_b, d_I], w_t [H_I], all fp64 (dequantised).
    """
    keys = k_idx_b[: pos + 1]                 # the visible history (causal)
    z = q_idx_t @ keys.T                      # [H_I, pos+1]: per-head relevance
    return w_t @ np.maximum(z, 0.0)           # weighted sum over heads


def topk_row(scores: np.ndarray, top_k: int) -> np.ndarray:
    """Positions of the min(top_k, len) largest scores; ties go to the smaller position."""
    n = min(int(top_k), scores.shape[0])
    order = np.argsort(-scores, kind="stable")  # stable: equal scores keep ascending position
    return order[:n].astype(np.int64)


def sfa_row(q_t: np.ndarray, kv_b: np.ndarray, sel: Sequence[int], d_c: int,
            sm_scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of every head of one query over the selected latent rows.

    q_t [H, D], kv_b [L_b, D]; returns out [H, d_c] and lse [H].
    An empty selection gives out = 0 and lse = -inf.
    """
    sel = np.asarray(sel, dtype=np.int64)
    H = q_t.shape[0]
    if sel.size == 0:
        return np.zeros((H, d_c)), np.full(H, -np.inf)
    rows = kv_b[sel]                          # gathered latent rows [n, D]
    S = sm_scale * (q_t @ rows.T)             # [H, n]
    m = S.max(axis=1, keepdims=True)
    e = np.exp(S - m)
    l = e.sum(axis=1)
    out = (e @ rows[:, :d_c]) / l[:, None]    # value = the latent columns
    lse = m[:, 0] + np.log(l)
    return out, lse


# ---------------------------------------------------------------------------
# Whole-problem driver over a set of query rows.


class Problem:
    """Inputs of one DSA problem, decoded to fp64 lazily per sequence / row.

    ``arrays`` maps names to numpy arrays as stored ('bf16' as uint16 bits,
    'e4m3' and 'mxfp8' as uint8 codes): cu_q, cu_k, q_idx, k_idx, w, q, kv and, for
    FP8, q_scale [ΣT, H_I] and k_scale [ΣL] (fp32); for MXFP8, q_scale
    [ΣT, H_I, d_I/32] and k_scale [ΣL, d_I/32] (E8M0 bytes).
    """

    def __init__(self, arrays: Dict[str, np.ndarray], *, idx_dtype: str, kv_dtype: str,
                 d_c: int, top_k: int, sm_scale: float = 0.0):
        self.a = arrays
        self.idx_dtype = idx_dtype
        self.kv_dtype = kv_dtype
        self.d_c = int(d_c)
        self.top_k = int(top_k)
        self.cu_q = [int(v) for v in arrays["cu_q"]]
        self.cu_k = [int(v) for v in arrays["cu_k"]]
        D = arrays["kv"].shape[1]
        self.sm_scale = float(sm_scale) if sm_scale else 1.0 / math.sqrt(D)
        self.rows = query_rows(self.cu_q, self.cu_k)
        self._k_cache: Dict[int, np.ndarray] = {}
        self._kv_cache: Dict[int, np.ndarray] = {}

    # -- decoded slices ---------------------------------------------------
    def k_idx_seq(self, b: int) -> np.ndarray:
        if b not in self._k_cache:
            lo, hi = self.cu_k[b], self.cu_k[b + 1]
            if self.idx_dtype == "mxfp8":
                k = mx_dequant(self.a["k_idx"][lo:hi], self.a["k_scale"][lo:hi])
            else:
                k = to_f64(self.a["k_idx"][lo:hi], self.idx_dtype)
            if self.idx_dtype == "e4m3":
                k = k * np.asarray(self.a["k_scale"][lo:hi], dtype=np.float64)[:, None]
            self._k_cache = {b: k}            # keep one sequence decoded at a time
        return self._k_cache[b]

    def kv_seq(self, b: int) -> np.ndarray:
        if b not in self._kv_cache:
            lo, hi = self.cu_k[b], self.cu_k[b + 1]
            self._kv_cache = {b: to_f64(self.a["kv"][lo:hi], self.kv_dtype)}
        return self._kv_cache[b]

    def kv_rows(self, b: int, sel: Sequence[int]) -> np.ndarray:
        """Latent rows ``sel`` of sequence b, decoded (only the rows asked for)."""
        sel = np.asarray(sel, dtype=np.int64)
        return to_f64(self.a["kv"][self.cu_k[b] + sel], self.kv_dtype)

    def q_idx_row(self, t: int) -> np.ndarray:
        if self.idx_dtype == "mxfp8":
            return mx_dequant(self.a["q_idx"][t], self.a["q_scale"][t])
        q = to_f64(self.a["q_idx"][t], self.idx_dtype)
        if self.idx_dtype == "e4m3":
            q = q * np.asarray(self.a["q_scale"][t], dtype=np.float64)[:, None]
        return q

    def q_row(self, t: int) -> np.ndarray:
        return to_f64(self.a["q"][t], self.kv_dtype)

    def w_row(self, t: int) -> np.ndarray:
        return np.asarray(self.a["w"][t], dtype=np.float64)

    # -- steps ------------------------------------------------------------
    def scores(self, t: int) -> np.ndarray:
        _, b, pos = self.rows[t]
        return indexer_row(self.q_idx_row(t), self.k_idx_seq(b), self.w_row(t), pos)

    def sfa(self, t: int, sel: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
        _, b, _ = self.rows[t]
        sel = np.asarray(sel, dtype=np.int64)
        # decode just the selected rows, then attend over all of them
        return sfa_row(self.q_row(t), self.kv_rows(b, sel), np.arange(sel.size), self.d_c,
                       self.sm_scale)

    def forward_row(self, t: int) -> Dict[str, np.ndarray]:
        """Scores → Top-K → SFA for one query row."""
        I = self.scores(t)
        sel = topk_row(I, self.top_k)
        out, lse = self.sfa(t, sel)
        return {"scores": I, "idx": sel, "out": out, "lse": lse}

    def forward(self, rows: Optional[Iterable[int]] = None) -> Dict[int, Dict[str, np.ndarray]]:
        """forward_row over ``rows`` (all rows by default), grouped by sequence."""
        rows = list(range(len(self.rows))) if rows is None else sorted(int(r) for r in rows)
        return {t: self.forward_row(t) for t in rows}


def torch_case_arrays(case) -> Dict[str, np.ndarray]:
    """Numpy views of a host ``Case``'s tensors in the stored encodings (bf16 → uint16 bits)."""
    import torch  # only to read the host tensors

    out = {}
    for k, v in case.tensors().items():
        v = v.contiguous()
        if v.dtype == torch.bfloat16:
            out[k] = v.view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = v.numpy()
    return out


def problem_from_case(case, sm_scale: float = 0.0) -> Problem:
    cfg = case.cfg
    return Problem(torch_case_arrays(case), idx_dtype=cfg.idx_dtype, kv_dtype=cfg.kv_dtype,
                   d_c=cfg.d_c, top_k=cfg.top_k, sm_scale=sm_scale)
