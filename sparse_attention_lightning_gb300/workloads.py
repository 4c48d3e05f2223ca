"""Seeded synthetic inputs for the DSA hot path.

This module only draws random numbers and stores them in the dtypes the path
consumes.  It holds none of the method's arithmetic: no scoring, no selection,
no attention.  Both the CUDA path (through the tests and the bench) and the
fp64 oracle consume the exact tensors made here, so the two sides see the same
bytes.

Workloads (the five DSA configurations: one tiny fp32 prefill, bf16 decode,
bf16 8k prefill, bf16 64k prefill, FP8-indexer decode):

* indexer query ``q_idx[ΣT, H_I, d_I]`` and keys ``k_idx[ΣL, d_I]`` ~ N(0, σ²)
  with σ = d_I^-1/2;
* MLA query ``q[ΣT, H, D]`` and latent cache ``kv[ΣL, D]`` ~ N(0, σ²) with
  σ = D^-1/2, D = d_c + d_rope (latent then rope columns);
* head weights ``w[ΣT, H_I]`` ~ U(0, 1);
* decode context lengths integer-uniform (inclusive) in the stated range;
* FP8 indexer inputs: bf16-valued data quantised per token (one fp32 scale
  per key row, one per query token broadcast over its heads), scale =
  amax/448, codes = E4M3 round-to-nearest-even of x/scale;
* MXFP8 indexer inputs: the same bf16 draws quantised per 32 elements: the
  shared scale 2^e is the smallest power of two with amax / 2^e <= 448 (so no
  element saturates), stored as the E8M0 byte e + 127 (127 for an all-zero
  group), codes = E4M3 round-to-nearest-even of x / 2^e;
* indexer prolog inputs (``prolog_inputs``): the bf16 indexer query before
  quantisation (the same draw the FP8 query codes are made from), a hidden
  state ``x[ΣT, d_model]`` ~ N(0, 1) and a head-weight projection
  ``W_h[H_I, d_model]`` ~ N(0, 1/d_model), both bf16.  The pages give no
  hidden width; 7168 is used for the DSA workloads.

All tensors live on the host (torch CPU); callers move them to the device.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import torch

F32, BF16, FP8, MXFP8 = "f32", "bf16", "e4m3", "mxfp8"

_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}

# Stable ids so each tensor gets its own stream for a given seed.
_STREAM_IDS = {"lens": 1, "q_idx": 2, "k_idx": 3, "w": 4, "q": 5, "kv": 6, "x": 9, "w_h": 10}
# (7 is the page order of paged caches)

_CHUNK = 1 << 24  # values drawn per generator call (bounds host temporaries)


@dataclasses.dataclass(frozen=True)
class Config:
    """Shape of one DSA problem (all sequences share the head/dim sizes)."""

    name: str
    q_lens: Sequence[int]
    k_lens: Sequence[int]
    h_idx: int
    d_idx: int
    h: int
    d_c: int
    d_rope: int
    top_k: int
    idx_dtype: str
    kv_dtype: str
    out_dtype: str

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def total_k(self) -> int:
        return int(sum(self.k_lens))

    @property
    def d(self) -> int:
        return self.d_c + self.d_rope


@dataclasses.dataclass
class Case:
    """Host tensors of one problem.

    FP8 tensors are stored as their raw E4M3 code bytes (``torch.uint8``); MXFP8 scales as
    their E8M0 bytes.
    """

    cfg: Config
    cu_q: torch.Tensor  # int32 [B+1]
    cu_k: torch.Tensor  # int32 [B+1]
    q_idx: torch.Tensor
    k_idx: torch.Tensor
    w: torch.Tensor
    q: torch.Tensor
    kv: torch.Tensor
    q_scale: Optional[torch.Tensor] = None  # f32 [ΣT, H_I] (FP8); uint8 [ΣT, H_I, d_I/32] (MXFP8)
    k_scale: Optional[torch.Tensor] = None  # f32 [ΣL] (FP8 only)

    def tensors(self) -> Dict[str, torch.Tensor]:
        out = {k: getattr(self, k) for k in
               ("cu_q", "cu_k", "q_idx", "k_idx", "w", "q", "kv", "q_scale", "k_scale")}
        return {k: v for k, v in out.items() if v is not None}


def _gen(seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + _STREAM_IDS[name])
    return g


def _normal(shape, std: float, g: torch.Generator, dtype) -> torch.Tensor:
    """N(0, std²) drawn in fp32 chunk by chunk, rounded (RNE) to ``dtype``."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=dtype)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        x = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        x.mul_(std)
        out[lo:hi] = x.to(dtype)
    return out.view(*shape)


def _quantise_e4m3_rows(x: torch.Tensor):
    """Per-row E4M3 codes and fp32 scales of a 2-D tensor (input preparation).

    scale = amax(|row|)/448 (1 for an all-zero row); codes = E4M3 RNE of
    row/scale, saturated to ±448.
    """
    xf = x.to(torch.float32)
    amax = xf.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    y = (xf / scale[:, None]).clamp_(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.contiguous()


def _quantise_mx_rows(x: torch.Tensor):
    """E4M3 codes [R, n] and E8M0 scale bytes [R, n/32] of a 2-D tensor, one scale per 32
    consecutive elements (input preparation)."""
    R, n = x.shape
    xf = x.to(torch.float32).reshape(R, n // 32, 32)
    amax = xf.abs().amax(dim=2)
    m, ex = torch.frexp(amax)                   # amax = m·2^ex, m in [0.5, 1); 448 = 0.875·2^9
    e = ex - 9 + (m > 0.875).to(ex.dtype)       # smallest e with amax <= 448·2^e
    e = torch.where(amax > 0, e, torch.zeros_like(e)).clamp_(-127, 127)
    y = (xf / torch.exp2(e.to(torch.float32))[:, :, None]).clamp_(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, n)
    return codes, (e + 127).to(torch.uint8).contiguous()


def decode_lengths(batch: int, lo: int, hi: int, seed: int) -> List[int]:
    """Context lengths integer-uniform in [lo, hi], inclusive."""
    g = _gen(seed, "lens")
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g)]


def make_case(cfg: Config, seed: int, attention: bool = True) -> Case:
    """Draw every input of ``cfg`` from streams seeded by ``seed`` (``attention=False``: the
    indexer's inputs only, q and kv left empty).  A config holding the first sequences of
    another draws exactly that config's first rows (every stream is drawn in row order)."""
    B = cfg.num_seqs
    for t, l in zip(cfg.q_lens, cfg.k_lens):
        if t > l:
            raise ValueError("each sequence needs q_len <= k_len (queries are its last tokens)")
    cu_q = torch.zeros(B + 1, dtype=torch.int32)
    cu_k = torch.zeros(B + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor(list(cfg.q_lens), dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.tensor(list(cfg.k_lens), dtype=torch.int64), 0).to(torch.int32)
    TQ, TK = cfg.total_q, cfg.total_k
    sd_i = cfg.d_idx ** -0.5
    sd_m = cfg.d ** -0.5
    kvd = _TORCH_DTYPE[cfg.kv_dtype]
    q_scale = k_scale = None
    if cfg.idx_dtype == FP8:
        qf = _normal((TQ, cfg.h_idx * cfg.d_idx), sd_i, _gen(seed, "q_idx"), torch.bfloat16)
        kf = _normal((TK, cfg.d_idx), sd_i, _gen(seed, "k_idx"), torch.bfloat16)
        q_codes, qs = _quantise_e4m3_rows(qf)
        q_idx = q_codes.view(TQ, cfg.h_idx, cfg.d_idx)
        q_scale = qs[:, None].expand(TQ, cfg.h_idx).contiguous()
        k_idx, k_scale = _quantise_e4m3_rows(kf)
    elif cfg.idx_dtype == MXFP8:
        qf = _normal((TQ, cfg.h_idx * cfg.d_idx), sd_i, _gen(seed, "q_idx"), torch.bfloat16)
        kf = _normal((TK, cfg.d_idx), sd_i, _gen(seed, "k_idx"), torch.bfloat16)
        q_codes, qs = _quantise_mx_rows(qf.reshape(TQ * cfg.h_idx, cfg.d_idx))
        q_idx = q_codes.view(TQ, cfg.h_idx, cfg.d_idx)
        q_scale = qs.view(TQ, cfg.h_idx, cfg.d_idx // 32)
        k_idx, k_scale = _quantise_mx_rows(kf)
    else:
        idd = _TORCH_DTYPE[cfg.idx_dtype]
        q_idx = _normal((TQ, cfg.h_idx, cfg.d_idx), sd_i, _gen(seed, "q_idx"), idd)
        k_idx = _normal((TK, cfg.d_idx), sd_i, _gen(seed, "k_idx"), idd)
    w = torch.rand(TQ, cfg.h_idx, generator=_gen(seed, "w"), dtype=torch.float32)
    if attention:
        q = _normal((TQ, cfg.h, cfg.d), sd_m, _gen(seed, "q"), kvd)
        kv = _normal((TK, cfg.d), sd_m, _gen(seed, "kv"), kvd)
    else:
        q = torch.empty(0, dtype=kvd)
        kv = torch.empty(0, dtype=kvd)
    return Case(cfg, cu_q, cu_k, q_idx, k_idx, w, q, kv, q_scale, k_scale)


# ---------------------------------------------------------------------------
# The five workloads.  Sizes are those of the DSA decode/prefill settings; seeds
# are fixed per workload (0 for the tiny one, 1..4 for the others).

def tiny_prefill() -> Config:
    return Config("tiny_prefill_T256_fp32", [256], [256], 4, 32, 8, 64, 16, 32, F32, F32, F32)


def decode(batch: int = 32, lo: int = 8192, hi: int = 32768, seed: int = 1) -> Config:
    lens = decode_lengths(batch, lo, hi, seed)
    return Config(f"decode_B{batch}_L{lo}-{hi}_bf16", [1] * batch, lens, 64, 128, 128, 512, 64,
                  2048, BF16, BF16, BF16)


def prefill(T: int) -> Config:
    return Config(f"prefill_T{T}_bf16", [T], [T], 64, 128, 128, 512, 64, 2048, BF16, BF16, BF16)


def fp8_decode(batch: int = 128, L: int = 131072) -> Config:
    return Config(f"fp8_indexer_decode_B{batch}_L{L}", [1] * batch, [L] * batch, 64, 128, 128, 512,
                  64, 2048, FP8, BF16, BF16)


def mxfp8_decode(batch: int = 128, L: int = 131072) -> Config:
    """The FP8 indexer decode shape with the pages' MXFP8 index format (same bf16 draws)."""
    return Config(f"mxfp8_indexer_decode_B{batch}_L{L}", [1] * batch, [L] * batch, 64, 128, 128,
                  512, 64, 2048, MXFP8, BF16, BF16)


WORKLOAD_SEEDS = {"tiny_prefill": 0, "decode": 1, "prefill_8k": 2, "prefill_64k": 3,
                  "fp8_decode": 4, "mxfp8_decode": 4}


def workload(name: str) -> Config:
    if name == "tiny_prefill":
        return tiny_prefill()
    if name == "decode":
        return decode(seed=WORKLOAD_SEEDS["decode"])
    if name == "prefill_8k":
        return prefill(8192)
    if name == "prefill_64k":
        return prefill(65536)
    if name == "fp8_decode":
        return fp8_decode()
    if name == "mxfp8_decode":
        return mxfp8_decode()
    raise KeyError(name)


def custom(q_lens, k_lens, h_idx=4, d_idx=32, h=8, d_c=64, d_rope=16, top_k=32,
           idx_dtype=F32, kv_dtype=F32, out_dtype=None, name="custom") -> Config:
    return Config(name, list(q_lens), list(k_lens), h_idx, d_idx, h, d_c, d_rope, top_k,
                  idx_dtype, kv_dtype, out_dtype or kv_dtype)


# ---------------------------------------------------------------------------
# Paged key caches: the same key-side rows scattered over pages.

_PAGE_STREAM = 7


@dataclasses.dataclass
class PagedKeys:
    """Key-side tensors of a case laid out in pages, and the block table that maps them."""

    page_size: int
    num_pages: int
    block_table: torch.Tensor   # int32 [B, max_pages]: page of each sequence's page slot, -1 unused
    k_idx: torch.Tensor         # [num_pages * page_size, d_I]
    kv: torch.Tensor            # [num_pages * page_size, D]
    k_scale: Optional[torch.Tensor] = None  # [num_pages * page_size] f32 (FP8), [.., d_I/32] uint8 (MXFP8)

    def tensors(self) -> Dict[str, torch.Tensor]:
        out = {"block_table": self.block_table, "k_idx": self.k_idx, "kv": self.kv}
        if self.k_scale is not None:
            out["k_scale"] = self.k_scale
        return out


def paged_keys(case: Case, page_size: int, seed: int, spare_pages: int = 3) -> PagedKeys:
    """Scatter the key side of ``case`` over pages: sequence b's L_b keys fill
    ceil(L_b / page_size) pages, drawn in a seeded random order from a pool that also holds
    ``spare_pages`` unused pages.  Rows that hold no key (unused pages, page tails) are
    filled with large values, so that reading one shows up in the results."""
    lens = list(case.cfg.k_lens)
    need = [(L + page_size - 1) // page_size for L in lens]
    num_pages = sum(need) + spare_pages
    max_pages = max(max(need), 1)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + _PAGE_STREAM)
    order = torch.randperm(num_pages, generator=g)
    table = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    rows = num_pages * page_size
    src = torch.full((rows,), -1, dtype=torch.int64)  # packed key row held by each cache row
    nxt, k0 = 0, 0
    for b, (L, npg) in enumerate(zip(lens, need)):
        for i in range(npg):
            pg = int(order[nxt])
            nxt += 1
            table[b, i] = pg
            n = min(page_size, L - i * page_size)
            src[pg * page_size: pg * page_size + n] = torch.arange(k0 + i * page_size,
                                                                   k0 + i * page_size + n)
        k0 += L
    used = src >= 0

    def scatter(x: torch.Tensor, fill) -> torch.Tensor:
        out = torch.full((rows,) + tuple(x.shape[1:]), fill, dtype=x.dtype)
        out[used] = x[src[used]]
        return out

    fill_idx = 0x7E if case.k_idx.dtype == torch.uint8 else 100.0  # E4M3 code 0x7E = 448
    if case.k_scale is None:
        k_scale = None
    else:
        k_scale = scatter(case.k_scale, 200 if case.k_scale.dtype == torch.uint8 else 1.0e4)
    return PagedKeys(page_size, num_pages, table, scatter(case.k_idx, fill_idx),
                     scatter(case.kv, 100.0), k_scale)


def first_sequences(cfg: Config, n: int) -> Config:
    """The config of ``cfg``'s first ``n`` sequences (same dims)."""
    return dataclasses.replace(cfg, name=f"{cfg.name}_first{n}", q_lens=list(cfg.q_lens[:n]),
                               k_lens=list(cfg.k_lens[:n]))


D_MODEL = 7168  # hidden width of the prolog's head-weight projection (not given by the pages)


def prolog_inputs(cfg: Config, seed: int, d_model: int = D_MODEL) -> Dict[str, torch.Tensor]:
    """The indexer prolog's inputs for ``cfg``'s query tokens: ``q_proj`` [ΣT, H_I, d_I] bf16
    (drawn from the stream the FP8 query codes are quantised from, so quantising it gives
    exactly ``make_case(cfg).q_idx`` of an FP8 config), ``x`` [ΣT, d_model] bf16 and ``w_h``
    [H_I, d_model] bf16."""
    TQ = cfg.total_q
    q_proj = _normal((TQ, cfg.h_idx * cfg.d_idx), cfg.d_idx ** -0.5, _gen(seed, "q_idx"),
                     torch.bfloat16).view(TQ, cfg.h_idx, cfg.d_idx)
    x = _normal((TQ, d_model), 1.0, _gen(seed, "x"), torch.bfloat16)
    w_h = _normal((cfg.h_idx, d_model), d_model ** -0.5, _gen(seed, "w_h"), torch.bfloat16)
    return {"q_proj": q_proj, "x": x, "w_h": w_h}
