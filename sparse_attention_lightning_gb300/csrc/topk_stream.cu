// Causal Top-K of materialised score rows, one 256-thread CTA per row streaming the row,
// for batches of many rows (prefill) whose score histogram (top 12 bits of the
// order-preserving key) was built by the tensor-core indexer's epilogue.
//
// Top-K selection of the Lightning Indexer ("Day0 Inference Adaptation and
// Performance Optimization for New-Architecture LLMs", §4.1): row t keeps the
// n = min(top_k, pos+1) largest of scores[t, 0..pos]; equal scores go to the
// smaller position.
//
// The histogram gives the bin B* that holds the n-th largest key, the count of keys
// above it and the count in it.  The CTA then reads the row once, 8192 keys at a time
// (bulk copies into a double-buffered tile in shared memory, the next tile in flight
// while this one is processed; 32 consecutive keys per thread): keys above B* ("definite") go straight to the
// output row at a running offset (block prefix sums keep position order), keys in B*
// ("candidates") are collected with their positions in shared memory (or, for a row
// whose histogram says they will not fit, just their positions in the row's slot of the
// workspace buffer, the keys read again from the scores).
// The candidates are refined by exact radix select on the low 20 key bits (ties by
// position) and written after the definite ones: all definite positions ascending,
// then the selected candidates ascending, as the other Top-K kernels write them.  No
// CTA waits for another, so many rows are in flight on every SM.
#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kT = 256;
constexpr int kW = kT / 32;
constexpr int kKPT = 32;               // keys per thread per tile
constexpr int kTile = kT * kKPT;       // 8192
constexpr int kCap = 4096;             // candidates refined from shared memory

struct ShS {
  float tile[2][kTile];                // the row, two 8192-key tiles at a time
  uint64_t tbar[2];
  uint32_t warp_a[kW], warp_b[kW];
  uint64_t warp_s[kW];
  uint32_t hist[2048];
  uint2 cand[kCap];                    // (key, position), position order
  uint32_t s_bin, s_above, s_cnt, s_digit;
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
  cta_sync();
  if (warp == 0) {
    const uint32_t v0 = lane < kW ? warp_a[lane] : 0u;
    uint32_t s = v0;
#pragma unroll
    for (int o = 1; o < kW; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    __syncwarp();
    if (lane < kW) warp_a[lane] = s;
  }
  cta_sync();
  const uint32_t before = (warp ? warp_a[warp - 1] : 0u) + x - v;
  *total = warp_a[kW - 1];
  cta_sync();
  return before;
}

// The same for a pair of 32-bit counts.
__device__ __forceinline__ uint64_t scan_pair64(uint64_t v, uint64_t* warp_s, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_s[warp] = x;
  cta_sync();
  if (warp == 0) {
    const uint64_t v0 = lane < kW ? warp_s[lane] : 0ull;
    uint64_t z = v0;
#pragma unroll
    for (int o = 1; o < kW; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    __syncwarp();
    if (lane < kW) warp_s[lane] = z;
  }
  cta_sync();
  const uint64_t before = (warp ? warp_s[warp - 1] : 0ull) + x - v;
  *total = warp_s[kW - 1];
  cta_sync();
  return before;
}

// Block-wide count held by all higher threads (exclusive suffix sum).
__device__ __forceinline__ uint32_t suffix_above(uint32_t mine, uint32_t* warp_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) warp_b[warp] = x;
  cta_sync();
  if (warp == 0) {
    const uint32_t v = lane < kW ? warp_b[lane] : 0u;
    uint32_t z = v;
#pragma unroll
    for (int o = 1; o < kW; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, z, o);
      if (lane + o < kW) z += y;
    }
    __syncwarp();
    if (lane < kW) warp_b[lane] = z - v;
  }
  cta_sync();
  const uint32_t r = warp_b[warp] + x - mine;
  cta_sync();
  return r;
}

__global__ void __launch_bounds__(kT, 2) topk_stream_kernel(TopkArgs a, int32_t* spill,
                                                         int64_t spill_ld) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ShS& S = *reinterpret_cast<ShS*>(smem_raw);
  const int tid = threadIdx.x;
  const int t = a.row0 + blockIdx.x;  // query row; its scores are row blockIdx.x
  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;
  const int n = r.pos + 1;
  const int k = min(a.top_k, n);
  griddep_wait();                  // the scores and histograms are complete
  if (tid == 0) griddep_launch();  // the attention kernel may be scheduled (it waits)
  const float* row = a.scores + (int64_t)blockIdx.x * a.ld;
  int32_t* irow = a.idx + (int64_t)t * a.top_k;
  float* vrow = a.vals ? a.vals + (int64_t)t * a.top_k : nullptr;

  if (k == n) {  // the whole history is kept
    for (int i = tid; i < n; i += kT) {
      irow[i] = i;
      if (vrow) vrow[i] = row[i];
    }
    for (int j = n + tid; j < a.top_k; j += kT) {
      irow[j] = -1;
      if (vrow) vrow[j] = -INFINITY;
    }
    return;
  }

  // ---- threshold bin: thread tid owns bins 16 tid .. 16 tid + 15 ----
  {
    const uint4* h4 = reinterpret_cast<const uint4*>(a.hist + (int64_t)blockIdx.x * kHistBins) + 4 * tid;
    uint32_t c[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldcg(h4 + q);
      c[4 * q] = v.x; c[4 * q + 1] = v.y; c[4 * q + 2] = v.z; c[4 * q + 3] = v.w;
    }
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) mine += c[i];
    const uint32_t above = suffix_above(mine, S.warp_b);
    if (above < (uint32_t)k && above + mine >= (uint32_t)k) {
      uint32_t run = above;
      for (int i = 15; i >= 0; --i) {
        if (run + c[i] >= (uint32_t)k) {
          S.s_bin = 16 * tid + i;
          S.s_above = run;
          S.s_cnt = c[i];
          break;
        }
        run += c[i];
      }
    }
    cta_sync();
  }
  const uint32_t bstar = S.s_bin, above = S.s_above, nc = S.s_cnt;
  const bool in_smem = nc <= (uint32_t)kCap;
  int32_t* gpos = spill + (int64_t)blockIdx.x * spill_ld;
  auto cand = [&](uint32_t c) -> uint2 {  // (key, position) of candidate c
    if (in_smem) return S.cand[c];
    const int32_t p = gpos[c];
    return make_uint2(order_key(row[p]), (uint32_t)p);
  };

  // ---- stream the row: definite positions out, candidates collected ----
  // tile i of the row into buffer i & 1 (16-byte rounded: the row's leading dimension is a
  // multiple of 32 scores, so the copy stays inside the row)
  const int ntile = (n + kTile - 1) / kTile;
  auto fetch = [&](int i) {
    const int base = i * kTile;
    const uint32_t bytes = (uint32_t)((min(kTile, n - base) * 4 + 15) & ~15);
    mbar_arrive_expect_tx(&S.tbar[i & 1], bytes);
    bulk_load(S.tile[i & 1], row + base, bytes, &S.tbar[i & 1]);
  };
  __shared__ int abort_word;
  if (tid == 0) {
    abort_word = 0;
    mbar_init(&S.tbar[0], 1);
    mbar_init(&S.tbar[1], 1);
    fence_barrier_init();
    fetch(0);
    if (ntile > 1) fetch(1);
  }
  cta_sync();
  uint32_t def_base = 0, cand_base = 0;
  int landed = 0;  // tiles consumed
  for (int ti = 0; ti < ntile; ++ti) {
    const int base = ti * kTile;
    const int i0 = base + kKPT * tid;
    // the same outcome in every thread, so that no thread is left at a barrier
    const bool ok = mbar_wait(&S.tbar[ti & 1], (ti >> 1) & 1, &abort_word, a.status,
                              DSA_FLAG_TIMEOUT);
    __syncwarp();  // the lanes left their waits apart; the barrier below is warp-aligned
    if (__syncthreads_or(!ok)) break;
    landed = ti + 1;
    const float* tl = S.tile[ti & 1] + kKPT * tid;
    float f[kKPT];
#pragma unroll
    for (int q = 0; q < kKPT / 4; ++q) {
      const float4 v = reinterpret_cast<const float4*>(tl)[q];
      f[4 * q] = v.x; f[4 * q + 1] = v.y; f[4 * q + 2] = v.z; f[4 * q + 3] = v.w;
    }
    uint32_t dm = 0, cm = 0;
#pragma unroll
    for (int j = 0; j < kKPT; ++j) {
      const uint32_t bin = order_key(f[j]) >> 20;
      dm |= (uint32_t)(bin > bstar) << j;
      cm |= (uint32_t)(bin == bstar) << j;
    }
    if (base + kTile > n) {  // the row's last tile: keys past the row do not count
      const int valid = n - i0;
      const uint32_t vm = valid >= kKPT ? 0xffffffffu : (valid <= 0 ? 0u : (1u << valid) - 1u);
      dm &= vm;
      cm &= vm;
    }
    uint32_t tot;
    const uint32_t pre = scan_pair((uint32_t)__popc(dm) | ((uint32_t)__popc(cm) << 16), S.warp_a,
                                   &tot);
    uint32_t pd = def_base + (pre & 0xffffu), pc = cand_base + (pre >> 16);
    // only the (few) set bits: one iteration per selected key
    for (uint32_t m = dm; m; m &= m - 1u, ++pd) {
      const int j = __ffs(m) - 1;
      // a definite key always has a slot (checked builds flag it; every build guards it)
      if (dsa_check(pd < (uint32_t)k, a.status) && pd < (uint32_t)k) {
        irow[pd] = i0 + j;
        if (vrow) vrow[pd] = tl[j];
      }
    }
    for (uint32_t m = cm; m; m &= m - 1u, ++pc) {
      const int j = __ffs(m) - 1;
      if (pc < nc) {
        if (in_smem) S.cand[pc] = make_uint2(order_key(tl[j]), (uint32_t)(i0 + j));
        else gpos[pc] = i0 + j;
      }
    }
    def_base += tot & 0xffffu;
    cand_base += tot >> 16;
    cta_sync();  // everyone is done with this buffer
    if (tid == 0 && ti + 2 < ntile) fetch(ti + 2);
  }
  if (landed < ntile) {
    // a copy that never landed (timed out): wait, bounded, for the ones still in flight,
    // then give up on the row
    if (tid == 0)
      for (int i = landed; i < min(ntile, landed + 2); ++i)
        mbar_wait_drain(&S.tbar[i & 1], (i >> 1) & 1);
    return;
  }
  if (tid == 0 && (def_base != above || cand_base != nc)) atomicOr(a.status, DSA_FLAG_BAD_SEQS);
  if (!in_smem) __threadfence_block();
  cta_sync();

  // ---- exact radix select among the candidates on the low 20 bits (11 + 9); thread tid
  // takes the candidates [tid * cpt, (tid + 1) * cpt) ----
  const uint32_t cpt = (nc + kT - 1) / kT;
  const uint32_t c_lo = min(nc, tid * cpt), c_hi = min(nc, c_lo + cpt);
  uint32_t prefix = bstar << 20, need = (uint32_t)k - above;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 9 : 0;
    const uint32_t bits = pass == 0 ? 11u : 9u;
    const uint32_t dmask = (1u << bits) - 1u;
    const uint32_t pmask = pass == 0 ? 0xfff00000u : 0xfffffe00u;
#pragma unroll
    for (int i = 0; i < 8; ++i) S.hist[8 * tid + i] = 0u;
    cta_sync();
    for (uint32_t c = c_lo; c < c_hi; ++c) {
      const uint32_t kk = cand(c).x;
      if ((kk & pmask) == prefix) atomicAdd(&S.hist[(kk >> shift) & dmask], 1u);
    }
    cta_sync();
    // digit (descending) where the need-th key falls: thread tid owns bins 8 tid .. 8 tid + 7
    uint32_t h[8], mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) { h[i] = S.hist[8 * tid + i]; mine += h[i]; }
    const uint32_t ab = suffix_above(mine, S.warp_b);
    if (ab < need && ab + mine >= need) {
      uint32_t run = ab;
      for (int i = 7; i >= 0; --i) {
        if (run + h[i] >= need) { S.s_digit = 8 * tid + i; S.s_cnt = run; break; }
        run += h[i];
      }
    }
    cta_sync();
    need -= S.s_cnt;
    prefix |= S.s_digit << shift;
    cta_sync();
  }
  const uint32_t T = prefix;  // exact key of the n-th largest; `need` of the ties are kept

  // ---- selected candidates, in position order, after the definite ones ----
  uint32_t ng = 0, ne = 0;
  for (uint32_t c = c_lo; c < c_hi; ++c) {
    const uint32_t kk = cand(c).x;
    ng += kk > T;
    ne += kk == T;
  }
  uint64_t ttot;
  const uint64_t pr = scan_pair64((uint64_t)ng | ((uint64_t)ne << 32), S.warp_s, &ttot);
  uint32_t gb = (uint32_t)pr, eb = (uint32_t)(pr >> 32);
  for (uint32_t c = c_lo; c < c_hi; ++c) {
    const uint2 ck = cand(c);
    int slot = -1;
    if (ck.x > T) {
      slot = (int)(above + gb + min(eb, need));
      ++gb;
      dsa_check(slot < k, a.status);  // every candidate above the threshold has a slot
    }
    else if (ck.x == T) { if (eb < need) slot = (int)(above + gb + eb); ++eb; }
    if (slot >= 0 && slot < k) {
      irow[slot] = (int32_t)ck.y;
      if (vrow) vrow[slot] = key_to_float(ck.x);
    }
  }
}

}  // namespace

int launch_topk_stream(const TopkArgs& a, int32_t* buf, int64_t buf_ld, cudaStream_t stream) {
  if (a.rows() <= 0) return DSA_OK;
  const size_t smem = sizeof(ShS);
  if (cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return check_launch("topk_stream: smem attribute");
  cudaError_t e = cudaSuccess;
  // candidates of a row that does not fit in shared memory: their positions in the row's
  // slot of the workspace buffer (buf_ld >= max_k_len entries)
  DSA_LAUNCH("topk_stream", stream,
             e = launch_pdl(topk_stream_kernel, dim3((unsigned)a.rows()), dim3(kT), smem,
                            stream, a, buf, buf_ld));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "topk_stream: %s", cudaGetErrorString(e));
  return check_launch("topk_stream");
}

}  // namespace dsa
