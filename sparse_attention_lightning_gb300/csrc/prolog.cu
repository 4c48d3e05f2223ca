// dsa_indexer_prolog: the indexer's two input-preparation steps that do not
// depend on the K cache, fused into one launch ("Day0 Inference Adaptation and
// Performance Optimization for New-Architecture LLMs", §4.2 Three-Stream
// Coordination for Indexer Preprocessing: Q quantisation and the head-weight
// projection share one stream; "Optimizing LLM Inference for New
// Architectures", §3).
//
//   Q quantisation: one CTA per token.  The token's H_I·d_I query elements
//     (up to 8192) are loaded once into registers, all loads in flight together:
//     first their absolute maximum, then each element divided by scale =
//     amax / 448 and rounded to E4M3 (nearest even, saturating).  Both
//     divisions are IEEE fp32 (__fdiv_rn), so the codes are a function of the
//     inputs alone, not of the compiler's division.  Longer tokens take a
//     two-pass loop.
//   Head-weight projection: w = x · W_hᵀ, one CTA per tile of 4 tokens × 8
//     heads.  Its threads split d_model in 16-byte chunks.  Each chunk's 12 row
//     loads are issued before any is used (rows past the end are clamped to the
//     last one and their sums dropped), so a chunk costs one memory latency,
//     not one per row.  fp32 accumulation, then a transpose-reduce across
//     each warp and a sum over the 16 warps.
//
// Both kinds of CTA run in the same grid (quantisation first), so the prolog
// is one launch on the caller's stream.  The outputs are what the FP8 fused
// indexer reads: codes [T, H_I, d_I], q_scale [T, H_I] (the token's scale
// repeated per head) and w [T, H_I] f32.
#include <cuda_fp8.h>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTB = 4;      // tokens of one projection tile
constexpr int kHB = 8;      // heads of one projection tile
constexpr int kQChunks = 2;  // 16-byte chunks of a token per thread kept in registers

struct PrologParams {
  const uint4* q_proj;  // [T, n8] chunks of 8 bf16
  const uint4* x;       // [T, dm8]
  const uint4* w_h;     // [h, dm8]
  uint2* q_codes;       // [T, n8] chunks of 8 e4m3 codes
  float* q_scale;       // [T, h]
  float* w;             // [T, h]
  int T, h, n8, dm8;
  int quant_blocks, head_tiles;
};

// 8 bf16 (one 16-byte chunk) widened exactly to fp32: a bf16 is the upper half of a binary32.
__device__ __forceinline__ void widen8(const uint4& v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float absmax8(const uint4& v, float m) {
  float f[8];
  widen8(v, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

__device__ __forceinline__ uint2 codes8(const uint4& v, float scale) {
  float f[8];
  widen8(v, f);
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    b[i] = __nv_cvt_float_to_fp8(__fdiv_rn(f[i], scale), __NV_SATFINITE, __NV_E4M3);
  return make_uint2(b[0] | b[1] << 8 | b[2] << 16 | b[3] << 24,
                    b[4] | b[5] << 8 | b[6] << 16 | b[7] << 24);
}

__device__ void quantise_token(const PrologParams& p, int t, float* red) {
  const uint4* src = p.q_proj + (size_t)t * p.n8;
  uint2* dst = p.q_codes + (size_t)t * p.n8;
  const bool resident = p.n8 <= kThreads * kQChunks;
  uint4 v[kQChunks];
  float m = 0.f;
  if (resident) {
#pragma unroll
    for (int i = 0; i < kQChunks; ++i) {
      const int c = threadIdx.x + i * kThreads;
      v[i] = c < p.n8 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kQChunks; ++i) m = absmax8(v[i], m);
  } else {
    for (int c = threadIdx.x; c < p.n8; c += kThreads) m = absmax8(__ldg(src + c), m);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) m = fmaxf(m, red[i]);
  const float scale = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;

  if (resident) {
#pragma unroll
    for (int i = 0; i < kQChunks; ++i) {
      const int c = threadIdx.x + i * kThreads;
      if (c < p.n8) dst[c] = codes8(v[i], scale);
    }
  } else {
    for (int c = threadIdx.x; c < p.n8; c += kThreads) dst[c] = codes8(__ldg(src + c), scale);
  }
  for (int j = threadIdx.x; j < p.h; j += kThreads) p.q_scale[(size_t)t * p.h + j] = scale;
}

__device__ void project_tile(const PrologParams& p, int tile, float* red) {
  const int t0 = (tile / p.head_tiles) * kTB, j0 = (tile % p.head_tiles) * kHB;
  const int nt = min(kTB, p.T - t0), nh = min(kHB, p.h - j0);
  // rows past the end repeat the last row: their loads stay in bounds, their sums are dropped
  const uint4* xrow[kTB];
  const uint4* wrow[kHB];
#pragma unroll
  for (int tt = 0; tt < kTB; ++tt) xrow[tt] = p.x + (size_t)(t0 + min(tt, nt - 1)) * p.dm8;
#pragma unroll
  for (int j = 0; j < kHB; ++j) wrow[j] = p.w_h + (size_t)(j0 + min(j, nh - 1)) * p.dm8;
  float acc[kTB][kHB];
#pragma unroll
  for (int a = 0; a < kTB; ++a)
#pragma unroll
    for (int b = 0; b < kHB; ++b) acc[a][b] = 0.f;

  for (int c = threadIdx.x; c < p.dm8; c += kThreads) {
    uint4 xr[kTB], wr[kHB];
#pragma unroll
    for (int tt = 0; tt < kTB; ++tt) xr[tt] = __ldg(xrow[tt] + c);
#pragma unroll
    for (int j = 0; j < kHB; ++j) wr[j] = __ldg(wrow[j] + c);
    float xf[kTB][8];
#pragma unroll
    for (int tt = 0; tt < kTB; ++tt) widen8(xr[tt], xf[tt]);
#pragma unroll
    for (int j = 0; j < kHB; ++j) {
      float wf[8];
      widen8(wr[j], wf);
#pragma unroll
      for (int tt = 0; tt < kTB; ++tt)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[tt][j] = fmaf(wf[e], xf[tt][e], acc[tt][j]);
    }
  }
  // Transpose-reduce the warp's 32 sums (one per (token, head) of the tile) in 31 shuffles:
  // at each halving step a lane keeps the half of its values its lane bit selects and adds the
  // partner's copy of that half; afterwards lane l holds value l summed over the warp.
  static_assert(kTB * kHB == 32, "one value per lane after the transpose-reduce");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float v[32];
#pragma unroll
  for (int tt = 0; tt < kTB; ++tt)
#pragma unroll
    for (int j = 0; j < kHB; ++j) v[tt * kHB + j] = acc[tt][j];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  red[warp * kTB * kHB + lane] = v[0];
  __syncthreads();
  if (threadIdx.x < kTB * kHB) {
    const int tt = threadIdx.x / kHB, j = threadIdx.x % kHB;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w * kTB * kHB + threadIdx.x];
    if (tt < nt && j < nh) p.w[(size_t)(t0 + tt) * p.h + j0 + j] = s;
  }
}

__global__ void __launch_bounds__(kThreads) indexer_prolog_kernel(PrologParams p) {
  __shared__ float red[kWarps * kTB * kHB];
  if ((int)blockIdx.x < p.quant_blocks)
    quantise_token(p, blockIdx.x, red);
  else
    project_tile(p, blockIdx.x - p.quant_blocks, red);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace dsa

extern "C" int dsa_indexer_prolog(int32_t total_q, int32_t h_idx, int32_t d_idx, int32_t d_model,
                                  const void* q_proj, const void* x, const void* w_h,
                                  uint8_t* q_codes, float* q_scale, float* w, void* stream) {
  using namespace dsa;
  if (total_q < 0 || h_idx < 1 || d_idx < 1)
    return set_error(DSA_ERR_INVALID_ARG, "total_q = %d, h_idx = %d, d_idx = %d", total_q, h_idx,
                     d_idx);
  if (total_q == 0) return DSA_OK;  // nothing to do; the pointers may be NULL
  const bool quant = q_proj != nullptr, proj = x != nullptr || w_h != nullptr;
  if (!quant && !proj) return set_error(DSA_ERR_INVALID_ARG, "q_proj, x and w_h are all NULL");
  if (quant) {
    if (!q_codes || !q_scale) return set_error(DSA_ERR_INVALID_ARG, "q_codes/q_scale is NULL");
    if (d_idx % 8) return set_error(DSA_ERR_UNSUPPORTED, "d_idx = %d (a multiple of 8)", d_idx);
    if (!al16(q_proj) || !al16(q_codes) || !al4(q_scale))
      return set_error(DSA_ERR_INVALID_ARG, "q_proj/q_codes not 16-byte or q_scale not 4-byte aligned");
  }
  if (proj) {
    if (!x || !w_h || !w) return set_error(DSA_ERR_INVALID_ARG, "x, w_h and w go together");
    if (d_model < 8 || d_model % 8)
      return set_error(DSA_ERR_UNSUPPORTED, "d_model = %d (a positive multiple of 8)", d_model);
    if (!al16(x) || !al16(w_h) || !al4(w))
      return set_error(DSA_ERR_INVALID_ARG, "x/w_h not 16-byte or w not 4-byte aligned");
  }
  if ((int64_t)h_idx * d_idx > (1 << 24) || (int64_t)total_q * h_idx >= (int64_t(1) << 31))
    return set_error(DSA_ERR_UNSUPPORTED, "total_q = %d, h_idx = %d, d_idx = %d too large",
                     total_q, h_idx, d_idx);

  PrologParams prm{};
  prm.q_proj = static_cast<const uint4*>(q_proj);
  prm.x = static_cast<const uint4*>(x);
  prm.w_h = static_cast<const uint4*>(w_h);
  prm.q_codes = reinterpret_cast<uint2*>(q_codes);
  prm.q_scale = q_scale;
  prm.w = w;
  prm.T = total_q;
  prm.h = h_idx;
  prm.n8 = h_idx * d_idx / 8;
  prm.dm8 = d_model / 8;
  prm.quant_blocks = quant ? total_q : 0;
  prm.head_tiles = (h_idx + kHB - 1) / kHB;
  const int64_t tiles = proj ? (int64_t)((total_q + kTB - 1) / kTB) * prm.head_tiles : 0;
  const int64_t blocks = prm.quant_blocks + tiles;
  if (blocks > 0x7fffffff) return set_error(DSA_ERR_UNSUPPORTED, "grid too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DSA_LAUNCH("indexer_prolog", s,
             indexer_prolog_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(prm));
  return check_launch("indexer_prolog");
}
