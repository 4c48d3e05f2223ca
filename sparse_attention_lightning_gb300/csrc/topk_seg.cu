// Causal Top-K of materialised score rows, spread over many CTAs per row, for
// rows whose score histogram (top 12 bits of the order-preserving key) was
// built by the tensor-core indexer's epilogue.
//
// Top-K selection of the Lightning Indexer ("Day0 Inference Adaptation and
// Performance Optimization for New-Architecture LLMs", §4.1): row t keeps the
// n = min(top_k, pos+1) largest of scores[t, 0..pos]; equal scores go to the
// smaller position.
//
// Phase 1, one CTA per 8192-key segment of a row: the histogram gives the bin
// B* that holds the n-th largest key and the count of keys above it.  The CTA
// reads its keys once and, in position order (block-wide prefix sums, no
// atomics), writes the positions of keys in bins above B* ("definite") and of
// keys in B* ("candidates") into the segment's slot of a per-row buffer.
// Phase 2, the last segment CTA of the row to finish (arrival counter): it
// refines only the candidates (exact radix select on the low 20 key bits, ties
// by position) and writes the row: all definite positions, ascending, then the
// selected candidates, ascending.  The result is deterministic.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kT = 1024;
constexpr int kW = kT / 32;
constexpr int kSeg = 8 * kT;       // keys per segment CTA
constexpr int kCandCap = 6144;     // candidates refined from shared memory
constexpr int kMaxSegs = 512;      // segments per row (rows up to 4M keys; grid y <= 65535)

struct Shared {
  uint32_t warp_a[kW], warp_b[kW];
  uint32_t seg_def[kMaxSegs + 1], seg_cnd[kMaxSegs + 1];  // exclusive prefix over segments
  uint32_t hist[2048];
  uint32_t ckey[kCandCap];
  int32_t cpos[kCandCap];
  uint32_t s_bin, s_above, s_cnt, s_last, s_digit;
};

// Block-wide exclusive prefix sum of a packed pair (low / high 16 bits).
__device__ __forceinline__ uint32_t scan_pair(uint32_t v, uint32_t* warp_a, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_a[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = warp_a[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_a[lane] = s;
  }
  __syncthreads();
  const uint32_t before = (warp ? warp_a[warp - 1] : 0u) + x - v;
  *total = warp_a[kW - 1];
  __syncthreads();
  return before;
}

// Bin of the n-th largest key and the number of keys in higher bins.
__device__ __forceinline__ void threshold_bin(const uint32_t* hrow, uint32_t k, Shared& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint4 c4 = __ldcg(reinterpret_cast<const uint4*>(hrow) + tid);  // bins 4tid..4tid+3
  const uint32_t mine = c4.x + c4.y + c4.z + c4.w;
  uint32_t x = mine;  // suffix sum over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) S.warp_b[warp] = x;
  __syncthreads();
  uint32_t above = x - mine;
  for (int w = warp + 1; w < kW; ++w) above += S.warp_b[w];
  if (above < k && above + mine >= k) {
    const uint32_t c[4] = {c4.w, c4.z, c4.y, c4.x};
    uint32_t run = above;
    for (int i = 0; i < 4; ++i) {
      if (run + c[i] >= k) {
        S.s_bin = 4 * tid + 3 - i;
        S.s_above = run;
        S.s_cnt = c[i];
        break;
      }
      run += c[i];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kT, 1) topk_seg_kernel(TopkArgs a, int32_t* buf, int64_t buf_ld,
                                                         uint32_t* seg_counts, int seg_ld,
                                                         uint32_t* done) {
  extern __shared__ uint8_t smem_raw[];
  Shared& S = *reinterpret_cast<Shared*>(smem_raw);
  const int t = blockIdx.x, seg = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;
  const int n = r.pos + 1;
  const int s0 = seg * kSeg;
  if (s0 >= n) return;
  const int nseg = (n + kSeg - 1) / kSeg;
  const int k = min(a.top_k, n);
  griddep_wait();                          // the scores and histograms are complete
  if (tid == 0) griddep_launch();          // the attention kernel may be scheduled (it waits)
  const float* row = a.scores + (int64_t)t * a.ld;
  int32_t* irow = a.idx + (int64_t)t * a.top_k;
  float* vrow = a.vals ? a.vals + (int64_t)t * a.top_k : nullptr;

  if (k == n) {  // the whole history is kept
    for (int i = s0 + tid; i < min(n, s0 + kSeg); i += kT) {
      irow[i] = i;
      if (vrow) vrow[i] = row[i];
    }
    if (seg == 0)
      for (int j = n + tid; j < a.top_k; j += kT) {
        irow[j] = -1;
        if (vrow) vrow[j] = -INFINITY;
      }
    return;
  }

  // ---- phase 1: this segment's definite positions and candidates ----
  threshold_bin(a.hist + (int64_t)t * kHistBins, (uint32_t)k, S);
  const uint32_t bstar = S.s_bin;
  const int i0 = s0 + 8 * tid;  // this thread's 8 consecutive keys
  uint32_t key[8];
  {
    float f[8];
    if (i0 + 7 < n) {
      const float4 a4 = __ldcg(reinterpret_cast<const float4*>(row + i0));
      const float4 b4 = __ldcg(reinterpret_cast<const float4*>(row + i0 + 4));
      f[0] = a4.x; f[1] = a4.y; f[2] = a4.z; f[3] = a4.w;
      f[4] = b4.x; f[5] = b4.y; f[6] = b4.z; f[7] = b4.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = i0 + j < n ? row[i0 + j] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) key[j] = order_key(f[j]);
  }
  uint32_t dm = 0, cm = 0;  // 8-bit masks
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (i0 + j < n) {
      const uint32_t b = key[j] >> 20;
      if (b > bstar) dm |= 1u << j;
      else if (b == bstar) cm |= 1u << j;
    }
  }
  uint32_t tot;
  const uint32_t pre = scan_pair((uint32_t)__popc(dm) | ((uint32_t)__popc(cm) << 16), S.warp_a, &tot);
  const uint32_t td = tot & 0xffffu, tcn = tot >> 16;
  int32_t* sbuf = buf + (int64_t)t * buf_ld + s0;
  {
    uint32_t pd = pre & 0xffffu, pc = (pre >> 16) + (kSeg - tcn);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (dm >> j & 1u) sbuf[pd++] = i0 + j;
      if (cm >> j & 1u) sbuf[pc++] = i0 + j;
    }
  }
  if (tid == 0) {
    seg_counts[((int64_t)t * seg_ld + seg) * 2] = td;
    seg_counts[((int64_t)t * seg_ld + seg) * 2 + 1] = tcn;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) S.s_last = atomicAdd(done + t, 1u) == (uint32_t)(nseg - 1);
  __syncthreads();
  if (!S.s_last) return;
  __threadfence();

  // ---- phase 2 (last segment of the row): refine the candidates, write the row ----
  if (tid == 0) done[t] = 0u;  // ready for the next call
  const uint32_t above = S.s_above;
  for (int s = tid; s < nseg; s += kT) {
    S.seg_def[s + 1] = __ldcg(seg_counts + ((int64_t)t * seg_ld + s) * 2);
    S.seg_cnd[s + 1] = __ldcg(seg_counts + ((int64_t)t * seg_ld + s) * 2 + 1);
  }
  if (tid == 0) { S.seg_def[0] = 0u; S.seg_cnd[0] = 0u; }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < nseg; ++s) { S.seg_def[s + 1] += S.seg_def[s]; S.seg_cnd[s + 1] += S.seg_cnd[s]; }
  __syncthreads();
  const uint32_t nc = S.seg_cnd[nseg];
  const int32_t* rbuf = buf + (int64_t)t * buf_ld;
  // definite positions, segment by segment (ascending)
  for (int s = 0; s < nseg; ++s) {
    const uint32_t base = S.seg_def[s], cnt = S.seg_def[s + 1] - base;
    for (uint32_t j = tid; j < cnt; j += kT) {
      const int32_t p = __ldcg(rbuf + (int64_t)s * kSeg + j);
      irow[base + j] = p;
      if (vrow) vrow[base + j] = row[p];
    }
  }
  // candidates in position order: (key, position)
  const bool in_smem = nc <= (uint32_t)kCandCap;
  for (int s = 0; s < nseg; ++s) {
    const uint32_t base = S.seg_cnd[s], cnt = S.seg_cnd[s + 1] - base;
    const int32_t* cb = rbuf + (int64_t)s * kSeg + (kSeg - cnt);
    if (in_smem)
      for (uint32_t j = tid; j < cnt; j += kT) {
        const int32_t p = __ldcg(cb + j);
        S.cpos[base + j] = p;
        S.ckey[base + j] = order_key(row[p]);
      }
  }
  __syncthreads();
  // position and key of candidate c (shared memory, or through the segment buffers)
  auto cand_pos = [&](uint32_t c) -> int32_t {
    if (in_smem) return S.cpos[c];
    int s = 0;
    while (S.seg_cnd[s + 1] <= c) ++s;
    const uint32_t cnt = S.seg_cnd[s + 1] - S.seg_cnd[s];
    return __ldcg(rbuf + (int64_t)s * kSeg + (kSeg - cnt) + (c - S.seg_cnd[s]));
  };
  auto cand_key = [&](uint32_t c) -> uint32_t {
    return in_smem ? S.ckey[c] : order_key(row[cand_pos(c)]);
  };

  // exact radix select among the candidates on the low 20 bits (11 + 9)
  uint32_t prefix = bstar << 20, need = (uint32_t)k - above;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 9 : 0;
    const uint32_t bits = pass == 0 ? 11u : 9u;
    const uint32_t dmask = (1u << bits) - 1u;
    const uint32_t pmask = pass == 0 ? 0xfff00000u : 0xfffffe00u;
    for (int i = tid; i < 2048; i += kT) S.hist[i] = 0u;
    __syncthreads();
    for (uint32_t c = tid; c < nc; c += kT) {
      const uint32_t kk = cand_key(c);
      if ((kk & pmask) == prefix) atomicAdd(&S.hist[(kk >> shift) & dmask], 1u);
    }
    __syncthreads();
    // digit d (descending) where the need-th key falls: thread tid owns bins 2tid+1, 2tid
    {
      const uint32_t h1 = tid * 2 + 1 < 2048 ? S.hist[tid * 2 + 1] : 0u;
      const uint32_t h0 = S.hist[tid * 2];
      const uint32_t mine = h0 + h1;
      uint32_t x = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      if (lane == 0) S.warp_b[tid >> 5] = x;
      __syncthreads();
      uint32_t ab = x - mine;
      for (int w = (tid >> 5) + 1; w < kW; ++w) ab += S.warp_b[w];
      if (ab < need && ab + mine >= need) {
        if (ab + h1 >= need) { S.s_digit = tid * 2 + 1; S.s_cnt = ab; }
        else { S.s_digit = tid * 2; S.s_cnt = ab + h1; }
      }
      __syncthreads();
    }
    need -= S.s_cnt;
    prefix |= S.s_digit << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // exact key of the n-th largest; `need` of the ties are kept

  // selected candidates, in position order, after the definite ones
  uint32_t G = 0, E = 0;
  for (uint32_t c0 = 0; c0 < nc; c0 += kT) {
    const uint32_t c = c0 + tid;
    uint32_t kk = 0;
    if (c < nc) kk = cand_key(c);
    const uint32_t gt = (c < nc && kk > T) ? 1u : 0u, eq = (c < nc && kk == T) ? 1u : 0u;
    uint32_t ttot;
    const uint32_t pr = scan_pair(gt | (eq << 16), S.warp_a, &ttot);
    const uint32_t gb = G + (pr & 0xffffu), eb = E + (pr >> 16);
    int slot = -1;
    if (gt) slot = (int)(above + gb + min(eb, need));
    else if (eq && eb < need) slot = (int)(above + gb + eb);
    if (slot >= 0) {
      irow[slot] = cand_pos(c);
      if (vrow) vrow[slot] = key_to_float(kk);
    }
    G += ttot & 0xffffu;
    E += ttot >> 16;
  }
}

}  // namespace

int topk_seg_segments(int max_k_len) { return (max_k_len + kSeg - 1) / kSeg; }
int topk_seg_max_keys() { return kMaxSegs * kSeg; }

int launch_topk_seg(const TopkArgs& a, int32_t* buf, int64_t buf_ld, uint32_t* seg_counts,
                    uint32_t* done, cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  const int nseg = topk_seg_segments(a.seqs.max_k_len);
  const size_t smem = sizeof(Shared);
  if (cudaFuncSetAttribute(topk_seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return check_launch("topk_seg: smem attribute");
  dim3 grid(a.seqs.total_q, nseg);  // rows on x (up to 2^31 - 1), segments on y
  cudaError_t e = cudaSuccess;
  DSA_LAUNCH("topk_seg", stream,
             e = launch_pdl(topk_seg_kernel, grid, dim3(kT), smem, stream, a, buf, buf_ld,
                            seg_counts, nseg, done));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "topk_seg: %s", cudaGetErrorString(e));
  return check_launch("topk_seg");
}

}  // namespace dsa
