"""CPU oracle of the indexer prolog.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the bench's CPU-baseline leg may
import this module.  The CUDA library never calls it and shares no code with it.

Before the fused indexer runs, two independent preparation steps produce its
inputs ("Day0 Inference Adaptation and Performance Optimization for
New-Architecture LLMs", §4.2 Three-Stream Coordination for Indexer
Preprocessing: q_quant = quant(q_proj) and w_proj = W_h @ x on the third
stream; "Optimizing LLM Inference for New Architectures", §3 Three-stream
coordination; "Day0 Inference Optimization for New Architecture LLMs Based on
CANN", §2.2 Indexer Prolog Three-Stream Coordination):

1. Q quantisation.  The indexer query q_proj[t] (all H_I·d_I elements of token
   t) becomes FP8 E4M3 codes with one fp32 scale per token, the format the FP8
   indexer reads (q = code · q_scale[t, j], the same scale for every head j):
       amax  = max |q_proj[t, :]|
       scale = fp32(amax / 448)            (1 for an all-zero token)
       code  = E4M3(fp32(q_proj[t, e] / scale)), round to nearest even,
               saturated to ±448 (the largest finite E4M3 value).
   Floating point decides an integer code here, so both divisions are taken in
   fp32 (IEEE, correctly rounded), the precision the kernel uses; the rounding
   to E4M3 is written out from the format's definition (e4m3_encode).
2. Head-weight projection.  w[t, j] = Σ_c W_h[j, c] · x[t, c] in fp64 over the
   bf16 inputs: one weight per (token, indexer head), no further factor (the
   pages give the plain product).
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

E4M3_MAX = 448.0        # S.1111.110: the largest finite E4M3 ('fn') value
_MIN_NORMAL = 2.0 ** -6  # exponent field 1
_SUB_QUANTUM = 2.0 ** -9  # spacing of the subnormals (and of the first binade)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """fp32 values → OCP E4M3 ('fn') codes: round to nearest, ties to even, saturating.

    Written from the format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 holds the subnormals m·2^-9; S.1111.111 is NaN; there are
    no infinities.  A finite magnitude above 448 saturates to 448 (0x7E); NaN
    encodes as 0x7F with its sign.
    """
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64))
    sign = np.where(np.signbit(y), 0x80, 0x00).astype(np.int64)
    # spacing of representable values around a: 2^(e-3) in binade [2^e, 2^(e+1)),
    # 2^-9 below the smallest normal
    _, E = np.frexp(np.where(a > 0, a, 1.0))  # a = f·2^E, f in [0.5, 1): e = E - 1
    quantum = np.where(a < _MIN_NORMAL, _SUB_QUANTUM, np.exp2((E - 1 - 3).astype(np.float64)))
    r = np.rint(a / quantum) * quantum        # a / quantum is exact; rint rounds half to even
    r = np.minimum(r, E4M3_MAX)
    _, Er = np.frexp(np.where(r > 0, r, 1.0))
    er = (Er - 1).astype(np.int64)
    normal = r >= _MIN_NORMAL
    mant = np.where(normal, r / np.exp2(er.astype(np.float64)) * 8.0 - 8.0, r / _SUB_QUANTUM)
    expf = np.where(normal, er + 7, 0)
    code = (expf << 3) | np.rint(mant).astype(np.int64)
    code = np.where(np.isnan(a), 0x7F, code)
    return (sign | code).astype(np.uint8)


def quantise_tokens(q_proj: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-token E4M3 quantisation of q_proj [T, n] (float32 values; bf16 inputs widened).

    Returns (codes uint8 [T, n], scale float32 [T]).
    """
    x = np.asarray(q_proj, dtype=np.float32)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / scale[:, None]).astype(np.float32)  # float32 / float32: IEEE, rounded to nearest
    return e4m3_encode(y), scale


def head_weights(x: np.ndarray, w_h: np.ndarray) -> np.ndarray:
    """w[t, j] = Σ_c W_h[j, c] · x[t, c] in fp64: x [T, d_model], W_h [H_I, d_model]."""
    return np.asarray(x, np.float64) @ np.asarray(w_h, np.float64).T
