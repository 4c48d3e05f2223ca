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
// Schedule: the tiles of all rows are laid end to end (a causal row at
// position p has floor(p/128) + 1 of them) and each persistent CTA takes one
// contiguous, equal share, so a long-history row is simply spread over more
// CTAs than a short one.  Each CTA derives the tile layout itself from cu_q /
// cu_k: per sequence the tile count is F(L) - F(L - T) with
// F(n) = Σ_{p<n} (floor(p/128) + 1) = n + 64 q (q - 1) + r q  (q = n / 128, r = n % 128).
// Warp roles: warp 0 issues TMA loads (a 4-8 stage ring of key tiles, a 2-slot
// ring of query blocks), warp 1 owns TMEM and issues the MMAs, warps 2..5 run
// the epilogue on a double-buffered TMEM accumulator.  Every wait is bounded
// (DSA_FLAG_TIMEOUT).
#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kMaxSeqs = 4096;  // sequences per launch on this path (tile table in smem)

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
  static constexpr int SMEM_FIXED = NS * KTILE + 2 * QTILE + kHistBins * 4 + 2048 /*bars etc*/ +
                                    1024 /*align*/;
};

struct Params {
  Seqs seqs;
  const float* w;
  const float* q_scale;
  const float* k_scale;
  float* scores;
  int64_t ld;
  uint32_t* status;
  uint32_t* hist;  // [total_q][kHistBins] or null
};

__device__ __forceinline__ int64_t ftiles(int64_t n) {  // Σ_{p<n} (floor(p/128) + 1)
  const int64_t q = n >> 7, r = n & 127;
  return n + 64 * q * (q - 1) + r * q;
}

// Per-sequence tile table built in shared memory by every CTA.
struct SeqTab {
  const int32_t* st;  // [B+1] first tile of each sequence, then the total
  const int32_t* cq;  // [B+1] cu_q
  const int32_t* ck;  // [B+1] cu_k
  int B;
};

// Walks the CTA's items (row tile by row tile) in order; all roles run one.
struct Cursor {
  int b, i, T, L, q0, k0;  // sequence, query index in it, its sizes and offsets
  int t, pos, j, ntiles;   // packed row, its position, current tile, tiles of the row

  __device__ __forceinline__ void load_seq(const SeqTab& s) {
    q0 = s.cq[b]; T = s.cq[b + 1] - q0;
    k0 = s.ck[b]; L = s.ck[b + 1] - k0;
  }
  __device__ __forceinline__ void set_row() {
    t = q0 + i;
    pos = L - T + i;
    ntiles = pos / 128 + 1;
  }
  __device__ __forceinline__ void locate(const SeqTab& s, int g) {
    int lo = 0, hi = s.B - 1;  // last b with st[b] <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.st[mid] <= g) lo = mid; else hi = mid - 1;
    }
    b = lo;
    load_seq(s);
    const int64_t gl = g - s.st[b], base = ftiles(L - T);
    int ilo = 0, ihi = T - 1;  // last i with F(L - T + i) - base <= gl
    while (ilo < ihi) {
      const int mid = (ilo + ihi + 1) >> 1;
      if (ftiles(L - T + mid) - base <= gl) ilo = mid; else ihi = mid - 1;
    }
    i = ilo;
    set_row();
    j = (int)(gl - (ftiles(L - T + i) - base));
  }
  __device__ __forceinline__ void advance(const SeqTab& s) {
    if (++j < ntiles) return;
    j = 0;
    if (++i == T) {
      i = 0;
      do { ++b; } while (b < s.B - 1 && s.st[b + 1] == s.st[b]);  // skip tile-less sequences
      load_seq(s);
    }
    set_row();
  }
};

__device__ __forceinline__ uint32_t scan192(uint32_t v, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  uint32_t before = 0, tot = 0;
  for (int w = 0; w < 6; ++w) {
    if (w < warp) before += ws[w];
    tot += ws[w];
  }
  *total = tot;
  __syncthreads();
  return before + x - v;
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
  uint32_t* hs = reinterpret_cast<uint32_t*>(qs + 2 * C::QTILE);  // row-segment histogram
  uint64_t* bars = reinterpret_cast<uint64_t*>(hs + kHistBins);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* q_full = k_empty + C::NS;
  uint64_t* q_empty = q_full + 2;
  uint64_t* acc_full = q_empty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* epi_a = drain + 1;     // 128 epilogue threads: row segment scored
  uint64_t* epi_b = drain + 2;     // 128 epilogue threads: histogram flushed
  float* wsm = reinterpret_cast<float*>(drain + 4);  // [4 epilogue warps][64]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wsm + 4 * 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* scan_ws = tmem_slot + 2;                   // [6]
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::SMEM_FIXED - 1024);
  const int B = p.seqs.B;
  int32_t* st = tab;
  int32_t* cq = st + (B + 1);
  int32_t* ck = cq + (B + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile table of the sequences (every CTA builds its own copy) ----
  uint32_t carry = 0;
  for (int base = 0; base < B; base += 192) {
    const int b = base + threadIdx.x;
    uint32_t n = 0;
    if (b < B) {
      const int q0 = __ldg(p.seqs.cu_q + b), q1 = __ldg(p.seqs.cu_q + b + 1);
      const int k0 = __ldg(p.seqs.cu_k + b), k1 = __ldg(p.seqs.cu_k + b + 1);
      const int T = q1 - q0, L = k1 - k0;
      const bool ok = q0 >= 0 && T >= 0 && T <= L && k0 >= 0 && k1 <= p.seqs.total_k &&
                      L <= p.seqs.max_k_len && q1 <= p.seqs.total_q;
      if (ok) n = (uint32_t)(ftiles(L) - ftiles(L - T));
      else if (blockIdx.x == 0) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
      cq[b] = q0;
      ck[b] = k0;
    }
    uint32_t tot;
    const uint32_t excl = scan192(n, scan_ws, &tot);
    if (b < B) st[b] = (int32_t)(carry + excl);
    carry += tot;
  }
  if (p.hist)
    for (int i = threadIdx.x; i < kHistBins; i += 192) hs[i] = 0u;
  if (threadIdx.x == 0) {
    st[B] = (int32_t)carry;
    cq[B] = __ldg(p.seqs.cu_q + B);
    ck[B] = __ldg(p.seqs.cu_k + B);
  }
  __syncthreads();
  const SeqTab tabs{st, cq, ck, B};
  const int total = st[B];
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
    mbar_init(epi_a, 128);
    mbar_init(epi_b, 128);
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
  if (threadIdx.x == 0) griddep_launch();  // the Top-K kernel may be scheduled (it waits)

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      Cursor cur;
      cur.locate(tabs, g0);
      int rows_seen = 0, issued = 0;
      for (int g = g0, it = 0; g < g1; ++g, ++it) {
        if (g > g0) cur.advance(tabs);
        if (g == g0 || cur.j == 0) {
          const int slot = rows_seen & 1;
          if (!mbar_wait(&q_empty[slot], ((rows_seen >> 1) & 1) ^ 1, abort_flag, p.status,
                         DSA_FLAG_TIMEOUT)) break;
          mbar_arrive_expect_tx(&q_full[slot], C::QTILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_2d(qs + slot * C::QTILE + a * (C::HI * 128), &qmap, &q_full[slot],
                        a * (128 / C::ES), cur.t * C::HI);
          ++rows_seen;
        }
        const int s = it % C::NS;
        if (!mbar_wait(&k_empty[s], ((it / C::NS) & 1) ^ 1, abort_flag, p.status,
                       DSA_FLAG_TIMEOUT)) break;
        mbar_arrive_expect_tx(&k_full[s], C::KTILE);
        for (int a = 0; a < C::ATOMS; ++a)
          tma_load_2d_hint(ks + s * C::KTILE + a * (C::BM * 128), &kmap, &k_full[s],
                           a * (128 / C::ES), cur.k0 + cur.j * C::BM, pol);
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
      Cursor cur;
      cur.locate(tabs, g0);
      int rows_seen = 0;
      for (int g = g0, it = 0; g < g1; ++g, ++it) {
        if (g > g0) cur.advance(tabs);
        if (g == g0 || cur.j == 0) {
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
        if (g + 1 == g1 || cur.j + 1 == cur.ntiles) mma_commit(&q_empty[slot]);
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lane quarter warp % 4 ----------------
    const int quarter = warp & 3;
    const int e = threadIdx.x - 64;  // 0..127
    float* wq = wsm + (warp - 2) * 64;
    int nseg = 0;
    Cursor cur;
    cur.locate(tabs, g0);
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
      if (g > g0) cur.advance(tabs);
      if (g == g0 || cur.j == 0) {
        __syncwarp();
        float w0 = __ldg(p.w + (int64_t)cur.t * C::HI + lane);
        float w1 = __ldg(p.w + (int64_t)cur.t * C::HI + lane + 32);
        if (FP8) {
          w0 *= __ldg(p.q_scale + (int64_t)cur.t * C::HI + lane);
          w1 *= __ldg(p.q_scale + (int64_t)cur.t * C::HI + lane + 32);
        }
        wq[lane] = w0;
        wq[lane + 32] = w1;
        __syncwarp();
      }
      const int acc = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (it >> 1) & 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT)))
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
      const int s = cur.j * C::BM + quarter * 32 + lane;
      if (s <= cur.pos) {
        if (FP8) sum *= __ldg(p.k_scale + cur.k0 + s);
        p.scores[(int64_t)cur.t * p.ld + s] = sum;
        if (p.hist) atomicAdd(&hs[order_key(sum) >> 20], 1u);
      }
      if (p.hist && (g + 1 == g1 || cur.j + 1 == cur.ntiles)) {
        // end of this CTA's part of the row: add the segment histogram to the row's
        mbar_arrive(epi_a);
        if (!__all_sync(0xffffffffu, mbar_wait(epi_a, nseg & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) break;
        uint32_t* grow = p.hist + (int64_t)cur.t * kHistBins;
        for (int bin = e; bin < kHistBins; bin += 128) {
          const uint32_t v = hs[bin];
          if (v) { atomicAdd(grow + bin, v); hs[bin] = 0u; }
        }
        mbar_arrive(epi_b);
        if (!__all_sync(0xffffffffu, mbar_wait(epi_b, nseg & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) break;
        ++nseg;
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

template <bool FP8>
int launch_typed(const IndexerArgs& a, float* scores, int64_t ld, cudaStream_t stream) {
  using C = Cfg<FP8>;
  CUtensorMap kmap, qmap;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int rc = make_tmap_2d(&kmap, dt, a.k_idx, C::DI, (uint64_t)a.seqs.total_k, C::ROWB,
                        128 / C::ES, C::BM);
  if (rc != DSA_OK) return rc;
  rc = make_tmap_2d(&qmap, dt, a.q_idx, C::DI, (uint64_t)a.seqs.total_q * C::HI, C::ROWB,
                    128 / C::ES, C::HI);
  if (rc != DSA_OK) return rc;
  const int smem = C::SMEM_FIXED + (int)align_up(3 * sizeof(int32_t) * (a.seqs.B + 1), 16);
  auto kern = indexer_tc_kernel<FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("indexer_tc: smem attribute");
  const int64_t bound = (int64_t)a.seqs.total_q * ((a.seqs.max_k_len + C::BM - 1) / C::BM);
  const int grid = (int)(bound < num_sms() ? bound : num_sms());
  Params p{a.seqs, a.w, a.q_scale, a.k_scale, scores, ld, a.status, a.hist};
  DSA_LAUNCH(FP8 ? "indexer_tc_fp8" : "indexer_tc_bf16", stream,
             kern<<<grid, 192, smem, stream>>>(kmap, qmap, p));
  return check_launch("indexer_tc");
}

}  // namespace

bool indexer_tc_eligible(const IndexerArgs& a) {
  // tiles of the whole problem must stay below 2^31 (int32 item indices)
  const int64_t bound = (int64_t)a.seqs.total_q * ((a.seqs.max_k_len + 127) / 128);
  return (a.idx_dtype == DSA_BF16 || a.idx_dtype == DSA_FP8_E4M3) && a.h_idx == 64 &&
         a.d_idx == 128 && a.seqs.B <= kMaxSeqs && bound < (int64_t(1) << 31);
}

int launch_indexer_tc(const IndexerArgs& a, float* scores, int64_t ld, cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  if (a.idx_dtype == DSA_FP8_E4M3) return launch_typed<true>(a, scores, ld, stream);
  return launch_typed<false>(a, scores, ld, stream);
}

}  // namespace dsa
