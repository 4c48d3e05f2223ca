// Lightning-Indexer scores on the CUDA cores (any dtype, any supported shape).
//
//   scores[t, s] = Σ_j w[t,j] · ReLU(q_idx[t,j,:] · k_idx[s,:])   s <= pos(t)
//
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
// LLMs", §4.1: batched dot of the indexer query against the K cache, then a
// weighted sum over the heads.)  This is the materialising variant behind
// dsa_indexer_scores and the fp32 path; it computes in fp32 with FMA.
//
// One CTA = one query row × one tile of 64 keys.  The query row (H_I × d_I) and
// the key tile sit in shared memory as fp32 (FP8 dequantised on load); each of
// the 256 threads takes one key and a quarter of the heads, and the four
// partial head sums are added in a fixed order.  MXFP8 inputs are dequantised
// with their E8M0 group scale (one per 32 elements of a query head or a key).
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kKeysPerCta = 64;
constexpr int kThreads = 256;
constexpr int kHeadGroups = kThreads / kKeysPerCta;  // 4

template <typename TI>
__global__ void __launch_bounds__(kThreads)
indexer_scores_simt_kernel(IndexerArgs a, float* __restrict__ scores, int64_t ld) {
  extern __shared__ float smem[];
  const int HI = a.h_idx, DI = a.d_idx;
  float* qs = smem;                         // [HI][DI]
  float* wsm = qs + HI * DI;                // [HI]
  float* ks = wsm + HI;                     // [64][DI + 1]
  float* red = ks + kKeysPerCta * (DI + 1); // [4][64]

  const int t = a.row0 + blockIdx.x;
  const int tid = threadIdx.x;
  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;
  const TI* qg = static_cast<const TI*>(a.q_idx) + (int64_t)t * HI * DI;
  const TI* kg = static_cast<const TI*>(a.k_idx);
  const bool fp8 = a.q_scale != nullptr;
  const bool mx = a.idx_dtype == DSA_MXFP8_E4M3;
  const int G = DI / 32;  // MXFP8 scale groups per head / key
  const uint8_t* qsb = reinterpret_cast<const uint8_t*>(a.q_scale);
  const uint8_t* ksb = reinterpret_cast<const uint8_t*>(a.k_scale);

  // the query row and its head weights
  for (int i = tid; i < HI * DI; i += kThreads) {
    float v = to_f32(qg[i]);
    if (mx) v *= e8m0_to_f32(__ldg(qsb + ((int64_t)t * HI + i / DI) * G + (i % DI) / 32));
    else if (fp8) v *= __ldg(a.q_scale + (int64_t)t * HI + i / DI);
    qs[i] = v;
  }
  for (int j = tid; j < HI; j += kThreads) wsm[j] = __ldg(a.w + (int64_t)t * HI + j);

  for (int64_t s0 = (int64_t)blockIdx.y * kKeysPerCta; s0 < ld;
       s0 += (int64_t)gridDim.y * kKeysPerCta) {
    float* out = scores + (int64_t)blockIdx.x * ld + s0;
    if (s0 > r.pos) {  // whole tile in the future: masked
      for (int i = tid; i < kKeysPerCta && s0 + i < ld; i += kThreads) out[i] = -INFINITY;
      continue;
    }
    __syncthreads();
    for (int i = tid; i < kKeysPerCta * DI; i += kThreads) {
      const int kr = i / DI, c = i - kr * DI;
      const int64_t s = s0 + kr;
      float v = 0.f;
      if (s <= r.pos) {
        const int64_t row = (int64_t)key_row(a.seqs, r.b, r.k0, (int)s);  // -1: page outside the cache
        if (row >= 0) {
          v = to_f32(kg[row * DI + c]);
          if (mx) v *= e8m0_to_f32(__ldg(ksb + row * G + c / 32));
          else if (fp8) v *= __ldg(a.k_scale + row);
        } else if (c == 0) {
          atomicOr(a.status, DSA_FLAG_BAD_SEQS);
        }
      }
      ks[kr * (DI + 1) + c] = v;
    }
    __syncthreads();

    const int kr = tid % kKeysPerCta, g = tid / kKeysPerCta;
    const float* krow = ks + kr * (DI + 1);
    float acc = 0.f;
    for (int j = g; j < HI; j += kHeadGroups) {
      const float* qrow = qs + j * DI;
      float dot = 0.f;
      for (int c = 0; c < DI; ++c) dot = fmaf(qrow[c], krow[c], dot);
      acc = fmaf(wsm[j], fmaxf(dot, 0.f), acc);
    }
    red[g * kKeysPerCta + kr] = acc;
    __syncthreads();
    if (g == 0) {
      const int64_t s = s0 + kr;
      float v = red[kr];
      for (int gg = 1; gg < kHeadGroups; ++gg) v += red[gg * kKeysPerCta + kr];
      if (s < ld) out[kr] = (s <= r.pos) ? v : -INFINITY;
    }
  }
}

template <typename TI>
int launch_typed(const IndexerArgs& a, float* scores, int64_t ld, cudaStream_t stream) {
  const size_t smem = sizeof(float) * ((size_t)a.h_idx * a.d_idx + a.h_idx +
                                       (size_t)kKeysPerCta * (a.d_idx + 1) +
                                       kHeadGroups * kKeysPerCta);
  auto kern = indexer_scores_simt_kernel<TI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("indexer_scores_simt: smem attribute");
  const int64_t tiles = (ld + kKeysPerCta - 1) / kKeysPerCta;
  const int rows = (a.row1 < a.seqs.total_q ? a.row1 : a.seqs.total_q) - a.row0;
  if (rows <= 0) return DSA_OK;
  dim3 grid((unsigned)rows, (unsigned)(tiles < 65535 ? tiles : 65535));
  DSA_LAUNCH("indexer_scores_simt", stream,
             kern<<<grid, kThreads, smem, stream>>>(a, scores, ld));
  return check_launch("indexer_scores_simt");
}

}  // namespace

int launch_indexer_scores_simt(const IndexerArgs& a, float* scores, int64_t ld,
                               cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  switch (a.idx_dtype) {
    case DSA_F32: return launch_typed<float>(a, scores, ld, stream);
    case DSA_BF16: return launch_typed<__nv_bfloat16>(a, scores, ld, stream);
    case DSA_FP8_E4M3:
    case DSA_MXFP8_E4M3: return launch_typed<__nv_fp8_e4m3>(a, scores, ld, stream);
  }
  return set_error(DSA_ERR_UNSUPPORTED, "indexer: idx_dtype %d", a.idx_dtype);
}

}  // namespace dsa
