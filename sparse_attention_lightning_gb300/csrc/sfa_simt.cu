// Sparse Flash Attention over the MLA latent cache, on the CUDA cores.
//
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
// LLMs", §2.2 and §4.1: the sparse attention core gathers the latent rows at the
// selected positions and attends over that subset, chunk by chunk.)  For query
// row t and head h, over the valid entries of idx[t, :]:
//   S_i = scale · q[t,h,:]·kv[row_i, :],  out = Σ softmax(S)_i · kv[row_i, :d_c]
// with a running (online) max and sum so the selected rows are read once.
//
// One CTA = one query row × up to 16 heads; the heads of a CTA share each
// gathered latent row (MLA: every head attends over the same latent).  This is
// the generic fp32/bf16 path; it computes in fp32.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxHeads = 16;   // heads per CTA
constexpr int kChunk = 32;      // gathered rows per step

template <typename TK, typename TO>
__global__ void __launch_bounds__(kThreads) sfa_simt_kernel(SfaArgs a) {
  extern __shared__ float smem[];
  const int D = a.d_c + a.d_rope, DP = D + 1, dc = a.d_c;
  const int t = blockIdx.x, h0 = blockIdx.y * kMaxHeads;
  const int HG = min(kMaxHeads, a.h - h0);
  const int tid = threadIdx.x;

  float* qs = smem;                          // [HG][D]
  float* kvs = qs + kMaxHeads * D;           // [kChunk][D+1]
  float* acc = kvs + kChunk * DP;            // [HG][dc]
  float* P = acc + kMaxHeads * dc;           // [HG][kChunk]
  float* m_s = P + kMaxHeads * kChunk;       // [HG] running max
  float* l_s = m_s + kMaxHeads;              // [HG] running sum
  float* al_s = l_s + kMaxHeads;             // [HG] rescale factor of this step
  int* sel = reinterpret_cast<int*>(al_s + kMaxHeads);  // [top_k] valid key rows
  __shared__ uint32_t warp_cnt[kThreads / 32];
  __shared__ int s_nvalid;

  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;

  // --- compact the valid indices (ascending slot order) -----------------------
  const int32_t* irow = a.idx + (int64_t)t * a.top_k;
  if (tid == 0) s_nvalid = 0;
  __syncthreads();
  for (int base = 0; base < a.top_k; base += kThreads) {
    const int i = base + tid;
    int v = -1;
    bool ok = false;
    int64_t row = -1;
    if (i < a.top_k) {
      v = irow[i];
      ok = (v >= 0 && v <= r.pos);
      if (ok) {
        row = key_row(a.seqs, r.b, r.k0, v);  // -1: page outside the cache
        ok = row >= 0;
      }
      if (!ok && v != -1) atomicOr(a.status, DSA_FLAG_BAD_INDEX);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    const int lane = tid & 31, warp = tid >> 5;
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int off = s_nvalid;
    for (int w = 0; w < warp; ++w) off += warp_cnt[w];
    if (ok) sel[off + __popc(bal & ((1u << lane) - 1u))] = (int32_t)row;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < kThreads / 32; ++w) tot += warp_cnt[w];
      s_nvalid += tot;
    }
    __syncthreads();
  }
  const int nvalid = s_nvalid;

  // --- query rows, accumulators ----------------------------------------------------
  const TK* qg = static_cast<const TK*>(a.q) + ((int64_t)t * a.h + h0) * D;
  for (int i = tid; i < HG * D; i += kThreads) qs[i] = to_f32(qg[i]);
  for (int i = tid; i < HG * dc; i += kThreads) acc[i] = 0.f;
  if (tid < kMaxHeads) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }
  const TK* kvg = static_cast<const TK*>(a.kv);

  for (int c0 = 0; c0 < nvalid; c0 += kChunk) {
    const int cn = min(kChunk, nvalid - c0);
    __syncthreads();
    for (int i = tid; i < kChunk * D; i += kThreads) {
      const int rr = i / D, c = i - rr * D;
      kvs[rr * DP + c] = rr < cn ? to_f32(kvg[(int64_t)sel[c0 + rr] * D + c]) : 0.f;
    }
    __syncthreads();
    // logits: (head, row) pairs; a warp shares a head, lanes take rows
    for (int p = tid; p < HG * kChunk; p += kThreads) {
      const int hh = p / kChunk, rr = p - hh * kChunk;
      const float* qrow = qs + hh * D;
      const float* krow = kvs + rr * DP;
      float dot = 0.f;
      for (int c = 0; c < D; ++c) dot = fmaf(qrow[c], krow[c], dot);
      P[hh * kChunk + rr] = rr < cn ? dot * a.scale : -INFINITY;
    }
    __syncthreads();
    // online softmax update, one warp per head
    for (int hh = tid >> 5; hh < HG; hh += kThreads / 32) {
      const int lane = tid & 31;
      float s = P[hh * kChunk + lane];  // kChunk == 32
      float mx = s;
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = m_s[hh];
      const float m_new = fmaxf(m_old, mx);
      const float e = (lane < cn) ? expf(s - m_new) : 0.f;
      P[hh * kChunk + lane] = e;
      float sum = e;
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      __syncwarp();
      if (lane == 0) {
        const float alpha = expf(m_old - m_new);  // 0 on the first chunk (m_old = -inf)
        al_s[hh] = alpha;
        l_s[hh] = l_s[hh] * alpha + sum;
        m_s[hh] = m_new;
      }
    }
    __syncthreads();
    // acc[h, c] = alpha·acc + Σ_r P[h, r]·kv[r, c]
    for (int i = tid; i < HG * dc; i += kThreads) {
      const int hh = i / dc, c = i - hh * dc;
      const float* ph = P + hh * kChunk;
      float v = acc[i] * al_s[hh];
      for (int rr = 0; rr < cn; ++rr) v = fmaf(ph[rr], kvs[rr * DP + c], v);
      acc[i] = v;
    }
  }
  __syncthreads();

  TO* og = static_cast<TO*>(a.out) + ((int64_t)t * a.h + h0) * dc;
  for (int i = tid; i < HG * dc; i += kThreads) {
    const int hh = i / dc;
    store_f32(og + i, nvalid ? acc[i] / l_s[hh] : 0.f);
  }
  if (a.lse && tid < HG)
    a.lse[(int64_t)t * a.h + h0 + tid] = nvalid ? m_s[tid] + logf(l_s[tid]) : -INFINITY;
}

template <typename TK, typename TO>
int launch_typed(const SfaArgs& a, cudaStream_t stream) {
  const int D = a.d_c + a.d_rope;
  const size_t smem = sizeof(float) * ((size_t)kMaxHeads * D + (size_t)kChunk * (D + 1) +
                                       (size_t)kMaxHeads * a.d_c + kMaxHeads * kChunk +
                                       3 * kMaxHeads) +
                      sizeof(int) * (size_t)a.top_k;
  auto kern = sfa_simt_kernel<TK, TO>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("sfa_simt: smem attribute");
  dim3 grid(a.seqs.total_q, (a.h + kMaxHeads - 1) / kMaxHeads);
  DSA_LAUNCH("sfa_simt", stream, kern<<<grid, kThreads, smem, stream>>>(a));
  return check_launch("sfa_simt");
}

}  // namespace

int launch_sfa_simt(const SfaArgs& a, cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  if (a.kv_dtype == DSA_F32 && a.out_dtype == DSA_F32) return launch_typed<float, float>(a, stream);
  if (a.kv_dtype == DSA_F32 && a.out_dtype == DSA_BF16)
    return launch_typed<float, __nv_bfloat16>(a, stream);
  if (a.kv_dtype == DSA_BF16 && a.out_dtype == DSA_F32)
    return launch_typed<__nv_bfloat16, float>(a, stream);
  if (a.kv_dtype == DSA_BF16 && a.out_dtype == DSA_BF16)
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream);
  return set_error(DSA_ERR_UNSUPPORTED, "sfa: kv_dtype %d out_dtype %d", a.kv_dtype, a.out_dtype);
}

}  // namespace dsa
