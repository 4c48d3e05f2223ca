// Causal Top-K of materialised score rows: one CTA per query row.
//
// Top-K selection of the Lightning Indexer ("Day0 Inference Adaptation and
// Performance Optimization for New-Architecture LLMs", §4.1).  Row t keeps the
// n = min(top_k, pos+1) largest of scores[t, 0..pos]; equal scores go to the
// smaller position.  Output is in ascending position order, padded with -1.
//
// Method: MSB-first radix select on order-preserving uint32 keys, 8 bits per
// pass with a 256-bin shared-memory histogram, fixes the exact n-th key T and
// how many keys equal to T are kept.  One ordered pass then writes every key
// > T and the first `need` keys == T, slots given by a block-wide prefix sum.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Block-wide exclusive prefix sum; returns the block total in *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = (warp ? warp_sums[warp - 1] : 0u) + x - v;
  *total = warp_sums[kWarps - 1];
  __syncthreads();  // warp_sums may be reused right after
  return before;
}

__global__ void __launch_bounds__(kThreads) topk_rows_kernel(TopkArgs a) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[kWarps];
  __shared__ uint32_t s_digit, s_above;

  const int t = a.row0 + blockIdx.x, tid = threadIdx.x;  // scores: row blockIdx.x
  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;
  const float* row = a.scores + (int64_t)blockIdx.x * a.ld;
  const int n = r.pos + 1;
  const int k = min(a.top_k, n);
  int32_t* idx = a.idx + (int64_t)t * a.top_k;
  float* vals = a.vals ? a.vals + (int64_t)t * a.top_k : nullptr;

  for (int j = k + tid; j < a.top_k; j += kThreads) {  // padding
    idx[j] = -1;
    if (vals) vals[j] = -INFINITY;
  }
  if (k == n) {  // the whole history is kept
    for (int i = tid; i < n; i += kThreads) {
      idx[i] = i;
      if (vals) vals[i] = row[i];
    }
    return;
  }

  // --- radix select of the k-th largest key ---------------------------------
  uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = order_key(row[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending order of digit)
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { c[i] = hist[255 - 8 * tid - i]; sum += c[i]; }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need && excl < need);
      if (hit) {
        const int owner = __ffs(hit) - 1;
        if (tid == owner) {
          uint32_t run = excl;
          for (int i = 0; i < 8; ++i) {
            if (run + c[i] >= need) { s_digit = 255 - 8 * tid - i; s_above = run; break; }
            run += c[i];
          }
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    need -= s_above;
    __syncthreads();
  }
  const uint32_t T = prefix;  // exact k-th largest key; `need` keys equal to it are kept

  // --- ordered write -----------------------------------------------------------
  uint32_t G = 0, E = 0;  // keys > T and keys == T before the current chunk
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + tid;
    uint32_t key = 0;
    if (i < n) key = order_key(row[i]);
    const uint32_t gt = (i < n && key > T) ? 1u : 0u;
    const uint32_t eq = (i < n && key == T) ? 1u : 0u;
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan(gt | (eq << 16), warp_sums, &tot);
    const uint32_t g_before = G + (pre & 0xffffu), e_before = E + (pre >> 16);
    int slot = -1;
    if (gt) slot = (int)(g_before + min(e_before, need));
    else if (eq && e_before < need) slot = (int)(g_before + e_before);
    if (slot >= 0) {
      idx[slot] = i;
      if (vals) vals[slot] = row[i];
    }
    G += tot & 0xffffu;
    E += tot >> 16;
  }
}

}  // namespace

int launch_topk_rows(const TopkArgs& a, cudaStream_t stream) {
  if (a.rows() <= 0) return DSA_OK;
  DSA_LAUNCH("topk_rows", stream,
             topk_rows_kernel<<<a.rows(), kThreads, 0, stream>>>(a));
  return check_launch("topk_rows");
}

}  // namespace dsa
