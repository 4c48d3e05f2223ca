// Lightning-Indexer scores on the 5th-generation tensor cores (tcgen05), for
// H_I = 64 heads of width d_I = 128 in bf16 or FP8 E4M3.
//
//   I[t, s] = Σ_j w[t,j] · ReLU(q_I[t,j,:] · k_I[s,:])      s <= pos(t)
//
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
// LLMs", §4.1: batched dot product of the indexer query with the K cache, then
// the weighted sum over heads, read straight from the K cache.)
//
// Work unit: one query row t × one tile of 128 keys.  The tile is the MMA's
// M = 128 (one key per TMEM lane), the row's 64 heads are N = 64, K = d_I.
// The per-head logits z[t, j, s] exist only in tensor memory: the epilogue
// reads its key's 64 columns and reduces them to one score (ReLU, · w, Σ_j)
// without any cross-thread reduction.  For FP8 the scales fold in as
// I = k_scale[s] · Σ_j (w·q_scale)[t,j] · ReLU(z8) (all scales are positive).
//
// Schedule: the tiles of all rows are laid end to end; each persistent CTA
// takes one contiguous, equal share, so a long-history row is simply spread
// over more CTAs than a short one.  Warp roles: warp 0 issues TMA loads
// (a 4-8 stage ring of key tiles, a 2-slot ring of query blocks), warp 1 owns
// TMEM and issues the MMAs, warps 2..5 run the epilogue on a double-buffered
// TMEM accumulator.  Every wait is bounded (DSA_FLAG_TIMEOUT).
#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {
namespace {

using namespace tc;

template <bool FP8>
struct Cfg {
  static constexpr int BM = 128;   // keys per tile (MMA M)
  static constexpr int HI = 64;    // heads (MMA N)
  static constexpr int DI = 128;   // head width (MMA K total)
  static constexpr int ES = FP8 ? 1 : 2;
  static constexpr int ROWB = DI * ES;             // bytes per key row (128 or 256)
  static constexpr int ATOMS = ROWB / 128;         // 128-byte swizzle atoms per row
  static constexpr int KTILE = BM * ROWB;          // 32 KB bf16, 16 KB fp8
  static constexpr int QTILE = HI * ROWB;          // 16 KB bf16, 8 KB fp8
  static constexpr int NS = FP8 ? 8 : 4;           // key-tile stages
  static constexpr int KSTEPS = FP8 ? 4 : 8;       // MMAs per tile (32 B of K each)
  static constexpr int ACC_COLS = HI;              // fp32 accumulator columns
  static constexpr int TMEM_COLS = 2 * ACC_COLS;   // double buffered
  static constexpr int SMEM = NS * KTILE + 2 * QTILE + 2048 /*bars etc*/ + 1024 /*align*/;
};

struct Params {
  Seqs seqs;
  const float* w;
  const float* q_scale;
  const float* k_scale;
  float* scores;
  int64_t ld;
  const int32_t* tile_start;  // [total_q + 1]: first tile of each row, then the total
  uint32_t* status;
};

// Row info without flagging (the tile-count pass has flagged bad rows already).
__device__ __forceinline__ void row_of(const Seqs& s, int t, int& pos, int& k0) {
  int lo = 0, hi = s.B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(s.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int q1 = __ldg(s.cu_q + lo + 1);
  k0 = __ldg(s.cu_k + lo);
  const int L = __ldg(s.cu_k + lo + 1) - k0;
  pos = L - (q1 - t);
}

// First row whose tile range contains g (tile_start is non-decreasing).
__device__ __forceinline__ int row_of_tile(const int32_t* ts, int nrows, int g) {
  int lo = 0, hi = nrows - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(ts + mid) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <bool FP8>
__global__ void __launch_bounds__(192, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  Params p) {
  using C = Cfg<FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ks = smem;                                  // NS key tiles
  uint8_t* qs = ks + C::NS * C::KTILE;                 // 2 query blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(qs + 2 * C::QTILE);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* q_full = k_empty + C::NS;
  uint64_t* q_empty = q_full + 2;
  uint64_t* acc_full = q_empty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  float* wsm = reinterpret_cast<float*>(drain + 2);  // [4 epilogue warps][64]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wsm + 4 * 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = p.seqs.total_q;
  const int total = __ldg(p.tile_start + nrows);
  const int g0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int g1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  if (g0 >= g1) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1);
      mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int t = row_of_tile(p.tile_start, nrows, g0), cur = -1, rows_seen = 0, pos = 0, k0 = 0;
      int issued = 0;
      for (int g = g0, it = 0; g < g1; ++g, ++it) {
        while (__ldg(p.tile_start + t + 1) <= g) ++t;
        if (t != cur) {
          cur = t;
          row_of(p.seqs, t, pos, k0);
          const int slot = rows_seen & 1;
          if (!mbar_wait(&q_empty[slot], ((rows_seen >> 1) & 1) ^ 1, abort_flag, p.status,
                         DSA_FLAG_TIMEOUT)) break;
          mbar_arrive_expect_tx(&q_full[slot], C::QTILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_2d(qs + slot * C::QTILE + a * (C::HI * 128), &qmap, &q_full[slot],
                        a * (128 / C::ES), t * C::HI);
          ++rows_seen;
        }
        const int j = g - __ldg(p.tile_start + t);
        const int s = it % C::NS;
        if (!mbar_wait(&k_empty[s], ((it / C::NS) & 1) ^ 1, abort_flag, p.status,
                       DSA_FLAG_TIMEOUT)) break;
        mbar_arrive_expect_tx(&k_full[s], C::KTILE);
        for (int a = 0; a < C::ATOMS; ++a)
          tma_load_2d_hint(ks + s * C::KTILE + a * (C::BM * 128), &kmap, &k_full[s],
                           a * (128 / C::ES), k0 + j * C::BM, pol);
        issued = it + 1;
      }
      // every key-tile copy issued has landed before the CTA may exit
      for (int i = (issued > C::NS ? issued - C::NS : 0); i < issued; ++i)
        mbar_wait_drain(&k_full[i % C::NS], (i / C::NS) & 1);
      if (rows_seen > 0) mbar_wait_drain(&q_full[(rows_seen - 1) & 1], ((rows_seen - 1) >> 1) & 1);
      if (rows_seen > 1) mbar_wait_drain(&q_full[(rows_seen - 2) & 1], ((rows_seen - 2) >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = FP8 ? idesc_e4m3(128, C::HI) : idesc_bf16(128, C::HI);
      int t = row_of_tile(p.tile_start, nrows, g0), cur = -1, rows_seen = 0;
      for (int g = g0, it = 0; g < g1; ++g, ++it) {
        while (__ldg(p.tile_start + t + 1) <= g) ++t;
        if (t != cur) {
          cur = t;
          if (!mbar_wait(&q_full[rows_seen & 1], (rows_seen >> 1) & 1, abort_flag, p.status,
                         DSA_FLAG_TIMEOUT)) break;
          tc_fence_after();
          ++rows_seen;
        }
        const int slot = (rows_seen - 1) & 1;
        const int s = it % C::NS, acc = it & 1;
        if (!mbar_wait(&acc_empty[acc], ((it >> 1) & 1) ^ 1, abort_flag, p.status,
                       DSA_FLAG_TIMEOUT)) break;
        if (!mbar_wait(&k_full[s], (it / C::NS) & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT))
          break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(ks + s * C::KTILE), b0 = smem_u32(qs + slot * C::QTILE);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          const int atom = (kk * 32) / 128, off = (kk * 32) % 128;
          const uint64_t ad = sdesc_sw128(a0 + atom * (C::BM * 128) + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(b0 + atom * (C::HI * 128) + off, 16, 1024);
          if (FP8) mma_e4m3(tmem + acc * C::ACC_COLS, ad, bd, idesc, kk > 0);
          else mma_bf16(tmem + acc * C::ACC_COLS, ad, bd, idesc, kk > 0);
        }
        mma_commit(&k_empty[s]);
        mma_commit(&acc_full[acc]);
        const bool last_of_row = (g + 1 == g1) || (__ldg(p.tile_start + t + 1) == g + 1);
        if (last_of_row) mma_commit(&q_empty[slot]);
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lane quarter warp % 4 ----------------
    const int quarter = warp & 3;
    float* wq = wsm + (warp - 2) * 64;
    int t = row_of_tile(p.tile_start, nrows, g0), cur = -1, pos = 0, k0 = 0;
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
      while (__ldg(p.tile_start + t + 1) <= g) ++t;
      if (t != cur) {
        cur = t;
        row_of(p.seqs, t, pos, k0);
        __syncwarp();
        float w0 = __ldg(p.w + (int64_t)t * C::HI + lane);
        float w1 = __ldg(p.w + (int64_t)t * C::HI + lane + 32);
        if (FP8) {
          w0 *= __ldg(p.q_scale + (int64_t)t * C::HI + lane);
          w1 *= __ldg(p.q_scale + (int64_t)t * C::HI + lane + 32);
        }
        wq[lane] = w0;
        wq[lane + 32] = w1;
        __syncwarp();
      }
      const int acc = it & 1;
      if (!mbar_wait(&acc_full[acc], (it >> 1) & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * C::ACC_COLS;
      uint32_t r[32];
      float sum = 0.f;
      tmem_ld32(taddr, r);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) sum = fmaf(wq[jj], fmaxf(__uint_as_float(r[jj]), 0.f), sum);
      tmem_ld32(taddr + 32, r);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj)
        sum = fmaf(wq[32 + jj], fmaxf(__uint_as_float(r[jj]), 0.f), sum);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      const int j = g - __ldg(p.tile_start + t);
      const int s = j * C::BM + quarter * 32 + lane;
      if (s <= pos) {
        if (FP8) sum *= __ldg(p.k_scale + k0 + s);
        p.scores[(int64_t)t * p.ld + s] = sum;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Tiles per row (ceil((pos+1)/128)) and their running start; 0 for invalid rows.
__global__ void __launch_bounds__(1024) row_tiles_kernel(Seqs seqs, int32_t* tile_start,
                                                          uint32_t* status) {
  __shared__ uint32_t warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t carry = 0;
  for (int base = 0; base < seqs.total_q; base += 1024) {
    const int t = base + tid;
    uint32_t n = 0;
    RowInfo r;
    if (t < seqs.total_q && query_row_info(seqs, t, r, status)) n = (uint32_t)(r.pos / 128 + 1);
    uint32_t x = n;
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
      warp_sums[lane] = s;
    }
    __syncthreads();
    const uint32_t excl = carry + (warp ? warp_sums[warp - 1] : 0u) + x - n;
    if (t < seqs.total_q) tile_start[t] = (int32_t)excl;
    carry += warp_sums[31];
    __syncthreads();
  }
  if (tid == 0) tile_start[seqs.total_q] = (int32_t)carry;
}

template <bool FP8>
int launch_typed(const IndexerArgs& a, float* scores, int64_t ld, int32_t* tile_start,
                 cudaStream_t stream) {
  using C = Cfg<FP8>;
  CUtensorMap kmap, qmap;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int rc = make_tmap_2d(&kmap, dt, a.k_idx, C::DI, (uint64_t)a.seqs.total_k, C::ROWB,
                        128 / C::ES, C::BM);
  if (rc != DSA_OK) return rc;
  rc = make_tmap_2d(&qmap, dt, a.q_idx, C::DI, (uint64_t)a.seqs.total_q * C::HI, C::ROWB,
                    128 / C::ES, C::HI);
  if (rc != DSA_OK) return rc;
  auto kern = indexer_tc_kernel<FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return check_launch("indexer_tc: smem attribute");
  DSA_LAUNCH("row_tiles", stream,
             row_tiles_kernel<<<1, 1024, 0, stream>>>(a.seqs, tile_start, a.status));
  rc = check_launch("row_tiles");
  if (rc != DSA_OK) return rc;
  const int64_t bound = (int64_t)a.seqs.total_q * ((a.seqs.max_k_len + C::BM - 1) / C::BM);
  const int grid = (int)(bound < num_sms() ? bound : num_sms());
  Params p{a.seqs, a.w, a.q_scale, a.k_scale, scores, ld, tile_start, a.status};
  DSA_LAUNCH(FP8 ? "indexer_tc_fp8" : "indexer_tc_bf16", stream,
             kern<<<grid, 192, C::SMEM, stream>>>(kmap, qmap, p));
  return check_launch("indexer_tc");
}

}  // namespace

bool indexer_tc_eligible(const IndexerArgs& a) {
  return (a.idx_dtype == DSA_BF16 || a.idx_dtype == DSA_FP8_E4M3) && a.h_idx == 64 &&
         a.d_idx == 128;
}

size_t indexer_tc_tile_start_bytes(int total_q) { return sizeof(int32_t) * ((size_t)total_q + 1); }

int launch_indexer_tc(const IndexerArgs& a, float* scores, int64_t ld, int32_t* tile_start,
                      cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  if (a.idx_dtype == DSA_FP8_E4M3) return launch_typed<true>(a, scores, ld, tile_start, stream);
  return launch_typed<false>(a, scores, ld, tile_start, stream);
}

}  // namespace dsa
