"""Comparison rules between the CUDA path and the fp64 oracle.

Top-K: the GPU row must hold exactly n = min(k, pos+1) unique causal positions
first, then -1 padding (their order is free); every position in the symmetric difference with
the oracle's set must have an oracle score within 1e-3 (relative) of the
oracle's n-th score.  Scores: max |gpu - oracle| <= 1e-2 · max |oracle| per row.
Attention: compared with the oracle's SFA evaluated on the GPU's own index set:
max abs error <= atol, per-(row, head) relative L2 error <= rel_l2, and lse
within lse_atol.
"""
from __future__ import annotations

import numpy as np
import torch

TOPK_BAND = 1e-3
SCORE_REL = 1e-2

# (atol, rel_l2, lse_atol) per configuration family
TOL = {
    "f32": (1e-5, 1e-5, 1e-5),
    "bf16": (2e-2, 1e-2, 2e-3),
    "e4m3": (6e-2, 1e-2, 2e-3),
}


def tol_for(cfg):
    if cfg.idx_dtype in ("e4m3", "mxfp8"):  # quantised indexer configurations
        return TOL["e4m3"]
    return TOL["f32"] if (cfg.kv_dtype == "f32" and cfg.out_dtype == "f32") else TOL["bf16"]


def check_topk_row(gpu_row: np.ndarray, scores: np.ndarray, k: int, ctx: str = "") -> dict:
    """Check one GPU index row against the oracle's scores of that query."""
    n = min(k, scores.shape[0])
    pos = scores.shape[0] - 1
    valid = gpu_row[:n]
    assert np.all(gpu_row[n:] == -1), f"{ctx}: padding is not -1"
    assert np.all(valid >= 0) and np.all(valid <= pos), f"{ctx}: non-causal index"
    assert np.unique(valid).size == valid.size, f"{ctx}: repeated index"
    order = np.argsort(-scores, kind="stable")
    ref = order[:n]
    s_k = scores[order[n - 1]]
    diff = np.setxor1d(valid, ref)
    band = TOPK_BAND * abs(s_k)
    bad = diff[np.abs(scores[diff] - s_k) > band]
    assert bad.size == 0, (f"{ctx}: {bad.size} selections differ outside the band "
                           f"(s_k={s_k}, e.g. pos {bad[:5]} scores {scores[bad[:5]]})")
    return {"swaps": int(diff.size // 2)}


def check_scores_row(gpu_row: np.ndarray, scores: np.ndarray, ctx: str = "") -> float:
    n = scores.shape[0]
    g = gpu_row[:n].astype(np.float64)
    assert np.all(np.isneginf(gpu_row[n:])), f"{ctx}: masked scores are not -inf"
    m = np.abs(scores).max()
    err = np.abs(g - scores).max()
    assert err <= SCORE_REL * m + 1e-30, f"{ctx}: score error {err} vs row max {m}"
    return float(err / m) if m > 0 else 0.0


def check_attn_row(out_gpu: np.ndarray, lse_gpu, out_ref: np.ndarray, lse_ref: np.ndarray, tol,
                   ctx: str = "") -> dict:
    atol, rel_l2, lse_atol = tol
    o = out_gpu.astype(np.float64)
    err = np.abs(o - out_ref)
    assert np.all(np.isfinite(o)), f"{ctx}: non-finite output"
    assert err.max() <= atol, f"{ctx}: max abs err {err.max()}"
    num = np.linalg.norm(o - out_ref, axis=-1)
    den = np.linalg.norm(out_ref, axis=-1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
    assert rel.max() <= rel_l2, f"{ctx}: rel L2 err {rel.max()}"
    if lse_gpu is not None:
        lg = lse_gpu.astype(np.float64)
        both_inf = np.isneginf(lg) & np.isneginf(lse_ref)
        d = np.where(both_inf, 0.0, np.abs(lg - lse_ref))
        assert d.max() <= lse_atol, f"{ctx}: lse err {d.max()}"
    return {"max_abs": float(err.max()), "rel_l2": float(rel.max())}


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.to(torch.float32)
    return t.numpy()
