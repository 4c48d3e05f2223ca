// The fused Lightning Indexer for rows that carry their own history (decode): relevance
// scoring, head weighting and the causal Top-K in one kernel, with no score ever written
// to global memory.  H_I = 64 heads of width d_I = 128, bf16 or FP8 E4M3.
//
//   I[t, s] = Σ_j w[t,j] · ReLU(q_I[t,j,:] · k_I[s,:])          s <= pos(t)
//   idx[t, :] = the min(top_k, pos+1) positions with the largest I (ties: smaller position)
//
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture LLMs",
// §4.1 Indexer Fusion: batched dot with the K cache, weighted sum over heads and Top-K as
// one operator whose intermediate results never go back to device memory; "Optimizing LLM
// Inference for New Architectures", §3: the scores stay in registers or on-chip memory and
// only the final Top-K indices leave.)
//
// One thread-block cluster of C CTAs per query row (C <= 8).  CTA c scores a contiguous
// run of the row's 128-key tiles on the tensor cores: TMA brings the key tiles two at a
// time into a ring of pair stages, one thread issues tcgen05.mma (M = 128 keys x N = 64
// heads x K = 128) for both tiles of a pair into one of two TMEM accumulator pairs, and
// eight epilogue warps (one per tile of the pair and TMEM lane quarter) reduce each key's
// 64 head logits to its score.  An N = 64 MMA takes ~50 clocks to issue and every barrier
// wait or commit costs about as much, so stages and accumulators come in pairs of tiles:
// one wait and one commit per two tiles.  Each score stays in a column of tensor memory
// (up to 256 tiles, 32,768 keys, per CTA) and is counted in a shared-memory histogram of
// its top 12 order-preserving key bits.
//
// Selection is exact and deterministic.  Round 1: every CTA adds the non-empty bins of its
// histogram into every CTA's copy of the row's histogram (distributed shared memory
// atomics); after a cluster barrier each CTA finds the bin B* of the k-th largest key.  Keys above B* are kept for sure.  The keys in
// B* (the candidates) are few: every CTA writes its own, in position order, into CTA 0's
// shared memory, and CTA 0 resolves the remaining 20 key bits by radix select over them,
// which fixes the exact key T of the k-th largest score and how many keys equal to T are
// kept (those at the smallest positions).  CTA 0 sends each CTA T and the counts of kept
// keys before it; each CTA then writes its kept positions straight to their slots: the
// row's selected positions in ascending order.  (If the candidates do not fit, two more
// histogram rounds over the whole cluster resolve the remaining bits instead.)
// Every mbarrier wait is bounded (DSA_FLAG_TIMEOUT); cluster barriers are hardware
// barriers that every thread of the cluster reaches on every path.
#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kBM = 128;                 // keys per tile (MMA M)
constexpr int kHI = 64;                  // heads (MMA N)
constexpr int kDI = 128;                 // head width (MMA K total)
constexpr int kEpiWarps = 8;             // (tile of the pair) x (TMEM lane quarter)
constexpr int kThreads = 64 + 32 * kEpiWarps;  // + TMA producer warp + MMA warp
constexpr int kWarps = kThreads / 32;
constexpr int kPair = 2;                 // tiles per stage and per accumulator
constexpr int kAccCols = kPair * kHI;    // one accumulator pair (fp32 columns)
constexpr int kScoreCol = 2 * kAccCols;  // first score column
constexpr int kHalfCols = 128;           // score columns of the even / odd tiles
constexpr int kMaxTiles = 2 * kHalfCols;  // tiles a CTA can hold: 256 (32,768 keys)
constexpr int kTmemCols = 512;
constexpr int kMaxCluster = 8;
constexpr int kNB1 = 4096, kNB2 = 2048, kNB3 = 512;  // digits of 12, 11 and 9 bits
static_assert(kScoreCol + kMaxTiles <= kTmemCols, "TMEM layout");

template <bool FP8>
struct Cfg {
  static constexpr int ES = FP8 ? 1 : 2;
  static constexpr int ROWB = kDI * ES;              // bytes per key row
  static constexpr int ATOMS = ROWB / 128;           // 128-byte swizzle atoms per row
  static constexpr int KTILE = kBM * ROWB;           // 32 KB bf16, 16 KB fp8
  static constexpr int STAGE = kPair * KTILE;
  static constexpr int QTILE = kHI * ROWB;           // the row's query heads
  static constexpr int NSS = FP8 ? 4 : 2;            // pair stages (128 KB either way)
  static constexpr int RING = NSS * STAGE;
  static constexpr int KSTEPS = FP8 ? 4 : 8;         // MMAs per tile (32 B of K each)
  // FP8: per-key scales by TMA with their key tile (132 floats from the tile's first key
  // rounded down to a multiple of 4), released by the epilogue; four spare slots
  static constexpr int NSC = FP8 ? kPair * NSS + 4 : 0;
  static constexpr int SC_BOX = kBM + 4;
  static constexpr int SC_BYTES = SC_BOX * 4;
  static constexpr int SC_SLOT = 640;
  // After the scores are in tensor memory the key ring of CTA 0 holds the row's candidates
  // (key, position).
  static constexpr int CAND_CAP = RING / 8;
  static constexpr int OFF_H = RING + QTILE;                  // this CTA's counts of a round
  static constexpr int OFF_A1 = OFF_H + kNB1 * 4;             // the cluster's counts, round 1
  static constexpr int OFF_A2 = OFF_A1 + kNB1 * 4;            // round 2
  static constexpr int OFF_A3 = OFF_A2 + kNB2 * 4;            // round 3
  static constexpr int OFF_CNT = OFF_A3 + kNB3 * 4;           // per (tile, quarter) counts
  static constexpr int OFF_SC = OFF_CNT + kMaxTiles * 4 * 4;  // FP8 scale ring
  static constexpr int OFF_PG = OFF_SC + NSC * SC_SLOT;       // the CTA's pages (paged caches)
  static constexpr int MAX_PG = kMaxTiles * (kBM / 16);       // 16-row pages at most
  static constexpr int OFF_MISC = OFF_PG + MAX_PG * 4;
  static constexpr int MISC = 1024;
  static constexpr int SMEM = OFF_MISC + MISC + 1024 /*alignment*/;
  static_assert(SMEM <= 232448, "shared memory");
};

struct Params {
  Seqs seqs;
  int top_k;
  int csize;  // CTAs per row
  const float* w;
  const float* q_scale;
  const float* k_scale;
  int32_t* idx;
  float* vals;
  uint32_t* status;
};

// Cluster exchange area: every CTA's copy may be written by the others.
struct Xch {
  uint32_t res[4];               // a round's digit, counts above it and in it (local);
                                 // from CTA 0: T, ties kept, kept keys before this CTA
  uint32_t gt[kMaxCluster];      // by CTA: keys above the threshold (bin, then key)
  uint32_t eq[kMaxCluster];      // by CTA: candidates / keys equal to the threshold
  uint32_t sum[2 * kMaxCluster];  // CTA 0: candidates above / equal to T, by source CTA
};

// h[bin] += 1 for every active lane, one shared-memory atomic per distinct bin of the warp
// (the scores of a row crowd into few bins).
__device__ __forceinline__ void warp_count(uint32_t* h, uint32_t bin, bool on) {
  const uint32_t act = __ballot_sync(0xffffffffu, on);
  if (!on) return;
  const uint32_t same = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == (uint32_t)(__ffs(same) - 1)) atomicAdd(&h[bin], (uint32_t)__popc(same));
}

// Exclusive sums over the CTA's threads of `v` held by lower / higher threads, with the
// total (two barriers).
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* ws, uint32_t* total,
                                               bool suffix) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = suffix ? __shfl_down_sync(0xffffffffu, x, o) : __shfl_up_sync(0xffffffffu, x, o);
    if (suffix ? lane + o < 32 : lane >= o) x += y;
  }
  // x: inclusive sum over the warp's lanes on the scanned side (and this lane)
  if (suffix ? lane == 0 : lane == 31) ws[warp] = x;
  __syncthreads();
  uint32_t other = 0, tot = 0;
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = ws[w];
    if (suffix ? w > warp : w < warp) other += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return other + x - v;
}

// The digit holding the need-th largest of the counts A[0..nb) (all threads; the same
// answer everywhere): (digit, count above it, count in it), through X->res.
__device__ uint3 find_digit(const uint32_t* A, int nb, uint32_t need, Xch* X, uint32_t* scan_ws) {
  const int per = (nb + kThreads - 1) / kThreads;
  const int b0 = min(nb, (int)threadIdx.x * per), b1 = min(nb, b0 + per);
  uint32_t mine = 0;
  for (int i = b0; i < b1; ++i) mine += A[i];
  uint32_t total;
  const uint32_t above = block_scan(mine, scan_ws, &total, true);
  if (above < need && above + mine >= need) {  // exactly one thread
    uint32_t run = above;
    for (int i = b1 - 1; i >= b0; --i) {
      if (run + A[i] >= need) {
        X->res[0] = (uint32_t)i;
        X->res[1] = run;
        X->res[2] = A[i];
        break;
      }
      run += A[i];
    }
  }
  __syncthreads();
  const uint3 r = make_uint3(X->res[0], X->res[1], X->res[2]);
  __syncthreads();  // X->res may be written again right after
  return r;
}

// One histogram round over the whole cluster: every CTA has counted its own keys of the
// current bucket into h[0..nb) and every CTA's A[0..nb) is zero.  Each CTA adds its
// non-empty bins into all copies of A; after the cluster barrier each CTA finds the digit.
__device__ uint3 cluster_round(const uint32_t* h, uint32_t* A, int nb, uint32_t need, Xch* X,
                               int C, uint32_t* scan_ws) {
  const uint32_t ab = smem_u32(A);
  for (int i = threadIdx.x; i < nb; i += kThreads) {
    const uint32_t v = h[i];
    if (v)
      for (int r = 0; r < C; ++r) red_cluster_add_u32(mapa(ab + 4u * (uint32_t)i, (uint32_t)r), v);
  }
  cluster_sync();  // every CTA's counts are in every copy (release / acquire, cluster scope)
  return find_digit(A, nb, need, X, scan_ws);
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
indexer_topk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap smap, Params p) {
  using C = Cfg<FP8>;
  constexpr int NSCM = C::NSC > 0 ? C::NSC : 1;
  constexpr int NBAR = 2 * C::NSS + 1 + 4 + 1 + C::NSC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ks = smem;
  uint8_t* qs = ks + C::RING;
  uint2* cand = reinterpret_cast<uint2*>(smem);  // CTA 0, after scoring: [CAND_CAP]
  uint32_t* h = reinterpret_cast<uint32_t*>(smem + C::OFF_H);
  uint32_t* A1 = reinterpret_cast<uint32_t*>(smem + C::OFF_A1);
  uint32_t* A2 = reinterpret_cast<uint32_t*>(smem + C::OFF_A2);
  uint32_t* A3 = reinterpret_cast<uint32_t*>(smem + C::OFF_A3);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + C::OFF_CNT);
  float* scs = reinterpret_cast<float*>(smem + C::OFF_SC);
  int32_t* pages = reinterpret_cast<int32_t*>(smem + C::OFF_PG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  uint64_t* k_full = bars;                   // [NSS]
  uint64_t* k_empty = k_full + C::NSS;       // [NSS]
  uint64_t* q_full = k_empty + C::NSS;
  uint64_t* acc_full = q_full + 1;           // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain = acc_empty + 2;
  uint64_t* sc_empty = drain + 1;            // [NSC]
  Xch* X = reinterpret_cast<Xch*>(smem + C::OFF_MISC + 8 * NBAR);
  uint32_t* scan_ws = reinterpret_cast<uint32_t*>(X + 1);  // [kWarps]
  uint32_t* tmem_slot = scan_ws + kWarps;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert(8 * NBAR + sizeof(Xch) + 4 * (kWarps + 2) <= C::MISC, "misc");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int csize = p.csize;
  const int c = (int)cluster_ctarank();
  const int t = blockIdx.x / csize;

  // ---- the row (the same outcome in every CTA of the cluster) ----
  RowInfo ri;
  if (!query_row_info(p.seqs, t, ri, p.status)) return;
  const int n = ri.pos + 1;                       // keys in the history
  const int k = min(p.top_k, n);
  const bool take_all = k == n;
  const int ntiles = (n + kBM - 1) / kBM;
  const int per = (ntiles + csize - 1) / csize;
  const int j0 = min(ntiles, c * per), j1 = min(ntiles, j0 + per);
  const int mytiles = j1 - j0;                    // this CTA's tiles of the row (may be 0)
  const int npairs = (mytiles + kPair - 1) / kPair;
  const bool stream = mytiles > 0 && !(take_all && p.vals == nullptr);
  int32_t* irow = p.idx + (int64_t)t * p.top_k;
  float* vrow = p.vals ? p.vals + (int64_t)t * p.top_k : nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSS; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], kEpiWarps); }
    mbar_init(drain, 1);
    for (int i = 0; i < C::NSC; ++i) mbar_init(&sc_empty[i], 4);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) X->res[i] = 0u;
    for (int i = 0; i < 2 * kMaxCluster; ++i) X->sum[i] = 0u;
    fence_barrier_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
    if (FP8) prefetch_tmap(&smap);
  }
  for (int i = threadIdx.x; i < kNB1; i += kThreads) { h[i] = 0u; A1[i] = 0u; }
  // paged caches: the block-table entries of this CTA's keys, fetched once (the producer
  // would otherwise wait for each lookup before it can issue the copy)
  const int cr = tile_chunk_rows(p.seqs);
  const int pg0 = p.seqs.paged() ? j0 * kBM / p.seqs.page_size : 0;  // first page of the CTA
  if (p.seqs.paged() && stream) {
    const int npg = min((min(j1 * kBM, n) - 1) / p.seqs.page_size - pg0 + 1, C::MAX_PG);
    for (int i = threadIdx.x; i < npg; i += kThreads)
      pages[i] = __ldg(p.seqs.block_table + (int64_t)ri.b * p.seqs.max_pages + pg0 + i);
  }
  for (int i = threadIdx.x; i < kNB2; i += kThreads) A2[i] = 0u;
  for (int i = threadIdx.x; i < kNB3; i += kThreads) A3[i] = 0u;
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  // every CTA of the cluster has started and cleared what its peers add into
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch();  // the attention kernel may be scheduled (it waits)

  // ================= scoring: this CTA's tiles j0 .. j1-1 of the row =================
  const int quarter = warp & 3;
  const int half = (warp - 2) >> 2;          // epilogue: tile 2p + half of pair p
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  if (stream) {
    if (warp == 0) {
      // ---- TMA producer: pair p = tiles 2p, 2p + 1 into stage p % NSS ----
      if (lane == 0) {
        const int sc_bytes = p.seqs.paged() ? kBM * 4 : C::SC_BYTES;
        const uint64_t pol = l2_policy_evict_first();
        int issued = 0;
        mbar_arrive_expect_tx(q_full, C::QTILE);
        for (int a = 0; a < C::ATOMS; ++a)
          tma_load_2d(qs + a * (kHI * 128), &qmap, q_full, a * (128 / C::ES), t * kHI);
        for (int pp = 0; pp < npairs; ++pp) {
          const int ss = pp % C::NSS;
          if (!mbar_wait(&k_empty[ss], ((pp / C::NSS) & 1) ^ 1, abort_flag, p.status,
                         DSA_FLAG_TIMEOUT)) break;
          const int nt = min(kPair, mytiles - kPair * pp);
          bool ok = true;
          if (FP8)
            for (int j = 0; j < nt && ok; ++j) {
              const int it = kPair * pp + j, sl = it % NSCM;
              ok = mbar_wait(&sc_empty[sl], ((it / NSCM) & 1) ^ 1, abort_flag, p.status,
                             DSA_FLAG_TIMEOUT);
            }
          if (!ok) break;
          mbar_arrive_expect_tx(&k_full[ss], nt * (C::KTILE + (FP8 ? sc_bytes : 0)));
          for (int j = 0; j < nt; ++j) {
            const int it = kPair * pp + j;
            const int s0 = (j0 + it) * kBM;  // the tile's first key position
            uint8_t* kdst = ks + ss * C::STAGE + j * C::KTILE;
            float* sdst = scs + (it % NSCM) * (C::SC_SLOT / 4);
            if (!p.seqs.paged()) {
              const int key0 = ri.k0 + s0;
              if (FP8) tma_load_2d(sdst, &smap, &k_full[ss], key0 & ~3, 0);
              for (int a = 0; a < C::ATOMS; ++a)
                tma_load_2d_hint(kdst + a * (kBM * 128), &kmap, &k_full[ss], a * (128 / C::ES),
                                 key0, pol);
            } else {
              // page by page: chunks of cr rows; a chunk past the history or on a page outside
              // the cache is read out of bounds (zero fill) and never selected
              for (int q = 0; q < kBM / cr; ++q) {
                const int pos = s0 + q * cr;
                int64_t row = -2;
                if (pos < n) {
                  const int pg = pages[pos / p.seqs.page_size - pg0];
                  row = pg >= 0 && pg < p.seqs.num_pages
                            ? (int64_t)pg * p.seqs.page_size + pos % p.seqs.page_size : -1;
                }
                if (row == -1) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
                if (row < 0) row = p.seqs.cache_rows();
                if (FP8) tma_load_2d(sdst + q * cr, &smap, &k_full[ss], (int)row, 0);
                for (int a = 0; a < C::ATOMS; ++a)
                  tma_load_2d_hint(kdst + a * (kBM * 128) + q * cr * 128, &kmap, &k_full[ss],
                                   a * (128 / C::ES), (int)row, pol);
              }
            }
          }
          issued = pp + 1;
        }
        // every copy issued has landed before the CTA goes on
        for (int i = (issued > C::NSS ? issued - C::NSS : 0); i < issued; ++i)
          mbar_wait_drain(&k_full[i % C::NSS], (i / C::NSS) & 1);
        mbar_wait_drain(q_full, 0);
      }
    } else if (warp == 1) {
      // ---- MMA issuer: both tiles of a pair, then one commit each for the stage and the
      // accumulator pair ----
      if (lane == 0) {
        const uint32_t idesc = FP8 ? idesc_e4m3(128, kHI) : idesc_bf16(128, kHI);
        if (mbar_wait(q_full, 0, abort_flag, p.status, DSA_FLAG_TIMEOUT)) {
          tc_fence_after();
          // descriptors of the ring's and of the query block's first K-step; a K-step adds
          // its byte offset / 16 to the start-address field
          const uint64_t bd0 = sdesc_sw128(smem_u32(qs), 16, 1024);
          const uint64_t ad0 = sdesc_sw128(smem_u32(ks), 16, 1024);
          for (int pp = 0; pp < npairs; ++pp) {
            const int ss = pp % C::NSS, acc = pp & 1;
            if (!mbar_wait(&acc_empty[acc], ((pp >> 1) & 1) ^ 1, abort_flag, p.status,
                           DSA_FLAG_TIMEOUT)) break;
            if (!mbar_wait(&k_full[ss], (pp / C::NSS) & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT))
              break;
            tc_fence_after();
            const int nt = min(kPair, mytiles - kPair * pp);
            for (int j = 0; j < nt; ++j) {
              const uint64_t as = ad0 + (uint64_t)((ss * C::STAGE + j * C::KTILE) >> 4);
              const uint32_t d = tmem + acc * kAccCols + j * kHI;
#pragma unroll
              for (int kk = 0; kk < C::KSTEPS; ++kk) {
                const int atom = (kk * 32) / 128, off = (kk * 32) % 128;
                const uint64_t ad = as + (uint64_t)((atom * (kBM * 128) + off) >> 4);
                const uint64_t bd = bd0 + (uint64_t)((atom * (kHI * 128) + off) >> 4);
                if (FP8) mma_e4m3(d, ad, bd, idesc, kk > 0);
                else mma_bf16(d, ad, bd, idesc, kk > 0);
              }
            }
            mma_commit(&k_empty[ss]);
            mma_commit(&acc_full[acc]);
          }
        }
        // every MMA issued has completed before TMEM is read for selection or released
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    } else {
      // ---- epilogue: warp (half, quarter) reduces tile 2p + half of every pair p ----
      float wreg[kHI];  // the row's head weights (FP8: times the query scales)
#pragma unroll
      for (int j = 0; j < kHI; ++j) {
        float wj = __ldg(p.w + (int64_t)t * kHI + j);
        if (FP8) wj *= __ldg(p.q_scale + (int64_t)t * kHI + j);
        wreg[j] = wj;
      }
      for (int pp = 0; pp < npairs; ++pp) {
        const int acc = pp & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (pp >> 1) & 1, abort_flag,
                                               p.status, DSA_FLAG_TIMEOUT)))
          break;
        tc_fence_after();
        const int it = kPair * pp + half;
        if (it < mytiles) {
          float ksc = 1.f;
          if (FP8) {
            // this thread's key scale, landed with the tile; keys past the row read a
            // neighbour's scale or the zero fill and are never selected
            const int sl = it % NSCM;
            const int sh = p.seqs.paged() ? 0 : ((ri.k0 + (j0 + it) * kBM) & 3);
            ksc = scs[sl * (C::SC_SLOT / 4) + sh + quarter * 32 + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sc_empty[sl]);
          }
          float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t r[32];
            tmem_ld32(lane_base + acc * kAccCols + half * kHI + 32 * hh, r);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              part[jj & 3] = fmaf(wreg[32 * hh + jj], fmaxf(__uint_as_float(r[jj]), 0.f), part[jj & 3]);
          }
          float v = (part[0] + part[1]) + (part[2] + part[3]);
          if (FP8) v *= ksc;
          tmem_st1(lane_base + kScoreCol + half * kHalfCols + pp, __float_as_uint(v));
          warp_count(h, order_key(v) >> 20, (j0 + it) * kBM + quarter * 32 + lane < n);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool failed = *abort_flag != 0;

  // Visit this thread's scores (epilogue warps; warp-uniform loop): f(tile, position, score).
  // Column kScoreCol + half * kHalfCols + p holds tile 2p + half.
  auto visit = [&](auto&& f) {
    if (warp < 2) return;
    const int ncol = (mytiles - half + 1) / 2;
    for (int cb = 0; cb < ncol; cb += 16) {
      uint32_t r[16];
      tmem_ld16(lane_base + kScoreCol + half * kHalfCols + cb, r);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int it = kPair * (cb + i) + half;
        if (cb + i < ncol) f(it, (j0 + it) * kBM + quarter * 32 + lane, __uint_as_float(r[i]));
      }
    }
  };
  // Per (tile, lane quarter) entry counts of two predicates of the keys, turned into
  // exclusive prefixes in position order within this CTA (low / high 16 bits); returns
  // the totals in the same packing.
  const uint32_t lt = (1u << lane) - 1u;
  auto count_prefix = [&](auto&& pred_lo, auto&& pred_hi) -> uint32_t {
    visit([&](int it, int s, float v) {
      const uint32_t key = order_key(v);
      const bool ok = s < n;
      const uint32_t lm = __ballot_sync(0xffffffffu, ok && pred_lo(key));
      const uint32_t hm = __ballot_sync(0xffffffffu, ok && pred_hi(key));
      if (lane == 0) cnt[it * 4 + quarter] = (uint32_t)__popc(lm) | ((uint32_t)__popc(hm) << 16);
    });
    __syncthreads();
    const int M = mytiles * 4;
    const int ce = (M + kThreads - 1) / kThreads;
    const int e0 = min(M, (int)threadIdx.x * ce), e1 = min(M, e0 + ce);
    uint32_t my = 0;
    for (int i = e0; i < e1; ++i) my += cnt[i];
    uint32_t tot;
    uint32_t run = block_scan(my, scan_ws, &tot, false);
    for (int i = e0; i < e1; ++i) {
      const uint32_t v = cnt[i];
      cnt[i] = run;
      run += v;
    }
    __syncthreads();
    return tot;
  };

  if (take_all) {
    // every key of the history is kept: position s goes to slot s (no communication)
    if (vrow) {
      if (stream && !failed)
        visit([&](int, int s, float v) {
          if (s < n) { irow[s] = s; vrow[s] = v; }
        });
    } else {
      for (int s = j0 * kBM + threadIdx.x; s < min(n, j1 * kBM); s += kThreads) irow[s] = s;
    }
    if (c == 0)
      for (int j = n + threadIdx.x; j < p.top_k; j += kThreads) {
        irow[j] = -1;
        if (vrow) vrow[j] = -INFINITY;
      }
  } else {
    // ================= exact selection across the cluster =================
    // round 1: top 12 key bits, counted by the epilogue
    const uint3 r1 = cluster_round(h, A1, kNB1, (uint32_t)k, X, csize, scan_ws);
    const uint32_t bstar = r1.x, nc1 = r1.z;
    uint32_t T, need, base_gt, base_eq;
    if (nc1 <= (uint32_t)C::CAND_CAP) {
      // ---- the candidates (keys in bin B*) go to CTA 0, in position order ----
      uint32_t cand_off = 0;  // candidates of the CTAs before this one
      for (int r = 0; r < c; ++r)
        cand_off += ld_cluster_u32(mapa(smem_u32(&h[bstar]), (uint32_t)r));
      const uint32_t tot = count_prefix([&](uint32_t key) { return (key >> 20) == bstar; },
                                        [&](uint32_t key) { return (key >> 20) > bstar; });
      const uint32_t cand0 = mapa(smem_u32(cand), 0u);
      visit([&](int it, int s, float v) {
        const uint32_t key = order_key(v);
        const uint32_t cm = __ballot_sync(0xffffffffu, s < n && (key >> 20) == bstar);
        if (cm >> lane & 1u) {
          const uint32_t rank =
              cand_off + (cnt[it * 4 + quarter] & 0xffffu) + (uint32_t)__popc(cm & lt);
          const uint32_t dst = cand0 + 8u * rank;
          st_cluster_u32(dst, key);
          st_cluster_u32(dst + 4u, (uint32_t)s);
        }
      });
      if (threadIdx.x == 0) {
        const uint32_t x0 = mapa(smem_u32(X), 0u);
        st_cluster_u32(x0 + (uint32_t)offsetof(Xch, gt) + 4u * c, tot >> 16);     // keys above B*
        st_cluster_u32(x0 + (uint32_t)offsetof(Xch, eq) + 4u * c, tot & 0xffffu);  // candidates
      }
      cluster_sync();  // all candidates in CTA 0
      if (c == 0) {
        // exact radix select on the low 20 bits among the candidates (h is free again:
        // the other CTAs read their offsets from it before the barrier)
        uint32_t need0 = (uint32_t)k - r1.y;
        for (int i = threadIdx.x; i < kNB2; i += kThreads) h[i] = 0u;
        __syncthreads();
        for (uint32_t i0 = 0; i0 < nc1; i0 += kThreads) {
          const uint32_t i = i0 + threadIdx.x;
          warp_count(h, i < nc1 ? (cand[i].x >> 9) & (kNB2 - 1) : 0u, i < nc1);
        }
        __syncthreads();
        const uint3 d2 = find_digit(h, kNB2, need0, X, scan_ws);
        need0 -= d2.y;
        const uint32_t prefix = (bstar << 20) | (d2.x << 9);
        for (int i = threadIdx.x; i < kNB3; i += kThreads) h[i] = 0u;
        __syncthreads();
        for (uint32_t i0 = 0; i0 < nc1; i0 += kThreads) {
          const uint32_t i = i0 + threadIdx.x;
          const uint32_t key = i < nc1 ? cand[i].x : 0u;
          warp_count(h, key & (kNB3 - 1), i < nc1 && (key & 0xfffffe00u) == prefix);
        }
        __syncthreads();
        const uint3 d3 = find_digit(h, kNB3, need0, X, scan_ws);
        need0 -= d3.y;
        const uint32_t T0 = prefix | d3.x;
        // candidates above / equal to T of each source CTA (their ranges are consecutive)
        uint32_t lo = 0;
        for (int r = 0; r < csize; ++r) {
          const uint32_t hi = lo + X->eq[r];
          uint32_t g = 0, e = 0;
          for (uint32_t i = lo + threadIdx.x; i < hi; i += kThreads) {
            g += cand[i].x > T0;
            e += cand[i].x == T0;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
          }
          if (lane == 0 && (g | e)) {
            atomicAdd(&X->sum[2 * r], g);
            atomicAdd(&X->sum[2 * r + 1], e);
          }
          lo = hi;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
          uint32_t bg = 0, be = 0;
          for (int r = 0; r < csize; ++r) {
            const uint32_t gr = X->gt[r] + X->sum[2 * r], er = X->sum[2 * r + 1];
            const uint32_t xr = mapa(smem_u32(X), (uint32_t)r);
            st_cluster_u32(xr, T0);
            st_cluster_u32(xr + 4u, need0);
            st_cluster_u32(xr + 8u, bg);
            st_cluster_u32(xr + 12u, be);
            bg += gr;
            be += er;
          }
          if (bg + need0 != (uint32_t)k || be < need0) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
        }
      }
      cluster_sync();  // T and this CTA's offsets from CTA 0
      T = X->res[0];
      need = X->res[1];
      base_gt = X->res[2];
      base_eq = X->res[3];
    } else {
      // ---- too many candidates for one CTA: two more histogram rounds (11 and 9 bits) ----
      need = (uint32_t)k - r1.y;
      uint32_t prefix = bstar << 20;
      for (int i = threadIdx.x; i < kNB2; i += kThreads) h[i] = 0u;
      __syncthreads();
      visit([&](int, int s, float v) {
        const uint32_t key = order_key(v);
        warp_count(h, (key >> 9) & (kNB2 - 1), s < n && (key & 0xfff00000u) == prefix);
      });
      __syncthreads();
      const uint3 r2 = cluster_round(h, A2, kNB2, need, X, csize, scan_ws);
      need -= r2.y;
      prefix |= r2.x << 9;
      for (int i = threadIdx.x; i < kNB3; i += kThreads) h[i] = 0u;
      __syncthreads();
      visit([&](int, int s, float v) {
        const uint32_t key = order_key(v);
        warp_count(h, key & (kNB3 - 1), s < n && (key & 0xfffffe00u) == prefix);
      });
      __syncthreads();
      const uint3 r3 = cluster_round(h, A3, kNB3, need, X, csize, scan_ws);
      need -= r3.y;
      T = prefix | r3.x;
      // keys above / equal to T of every CTA
      const uint32_t Tl = T;
      const uint32_t tot = count_prefix([&](uint32_t key) { return key > Tl; },
                                        [&](uint32_t key) { return key == Tl; });
      if ((int)threadIdx.x < csize) {
        const uint32_t hx = mapa(smem_u32(X), threadIdx.x);
        st_cluster_u32(hx + (uint32_t)offsetof(Xch, gt) + 4u * c, tot & 0xffffu);
        st_cluster_u32(hx + (uint32_t)offsetof(Xch, eq) + 4u * c, tot >> 16);
      }
      cluster_sync();
      base_gt = 0;
      base_eq = 0;
      for (int r = 0; r < c; ++r) { base_gt += X->gt[r]; base_eq += X->eq[r]; }
    }

    // ---- every kept key to its slot: kept keys in position order ----
    // (keys above T, and the first `need` keys equal to T by position)
    const uint32_t Tk = T;
    count_prefix([&](uint32_t key) { return key > Tk; }, [&](uint32_t key) { return key == Tk; });
    if (!failed)
      visit([&](int it, int s, float v) {
        const uint32_t key = order_key(v);
        const bool ok = s < n;
        const uint32_t gm = __ballot_sync(0xffffffffu, ok && key > Tk);
        const uint32_t em = __ballot_sync(0xffffffffu, ok && key == Tk);
        const uint32_t pre = cnt[it * 4 + quarter];
        const uint32_t gb = base_gt + (pre & 0xffffu) + (uint32_t)__popc(gm & lt);
        const uint32_t eb = base_eq + (pre >> 16) + (uint32_t)__popc(em & lt);
        int slot = -1;
        if (ok && key > Tk) slot = (int)(gb + min(eb, need));
        else if (ok && key == Tk && eb < need) slot = (int)(gb + eb);
        if (slot >= 0 && slot < k) {
          irow[slot] = s;
          if (vrow) vrow[slot] = v;
        }
      });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int choose_cluster(const IndexerArgs& a) {
  const int64_t ntiles = ((int64_t)a.seqs.max_k_len + kBM - 1) / kBM;
  const int c_cap = (int)((ntiles + kMaxTiles - 1) / kMaxTiles);
  // one CTA per SM: spread few rows over all SMs in one wave when possible
  const int c_fill = a.seqs.total_q > 0 ? num_sms() / a.seqs.total_q : 1;
  int cs = c_fill > c_cap ? c_fill : c_cap;
  if (cs < 1) cs = 1;
  if (cs > kMaxCluster) cs = kMaxCluster;
  return cs;
}

template <bool FP8>
int launch_typed(const IndexerArgs& a, int top_k, int32_t* idx, float* vals, cudaStream_t stream) {
  using C = Cfg<FP8>;
  CUtensorMap kmap, qmap, smap;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int cr = tile_chunk_rows(a.seqs);  // key rows per copy (a page, for small pages)
  int rc = make_tmap_2d(&kmap, dt, a.k_idx, kDI, (uint64_t)a.seqs.cache_rows(), C::ROWB, 128 / C::ES,
                        (uint32_t)cr);
  if (rc != DSA_OK) return rc;
  rc = make_tmap_2d(&qmap, dt, a.q_idx, kDI, (uint64_t)a.seqs.total_q * kHI, C::ROWB, 128 / C::ES, kHI);
  if (rc != DSA_OK) return rc;
  if (FP8) {
    const uint64_t rows = (uint64_t)a.seqs.cache_rows();
    rc = make_tmap_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.k_scale, rows, 1,
                      align_up((size_t)rows * 4, 16), a.seqs.paged() ? (uint32_t)cr : C::SC_BOX,
                      1, false);
    if (rc != DSA_OK) return rc;
  } else {
    smap = kmap;  // unused
  }
  auto kern = indexer_topk_kernel<FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return check_launch("indexer_topk: smem attribute");
  const int cs = choose_cluster(a);
  Params p{a.seqs, top_k, cs, a.w, a.q_scale, a.k_scale, idx, vals, a.status};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.seqs.total_q * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
  DSA_LAUNCH(FP8 ? "indexer_topk_fp8" : "indexer_topk_bf16", stream,
             e = cudaLaunchKernelEx(&cfg, kern, kmap, qmap, smap, p));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "indexer_topk: %s", cudaGetErrorString(e));
  return check_launch("indexer_topk");
}

}  // namespace

// Rows whose clusters all fit on the GPU at once (one CTA per SM): several waves would each
// end in a selection tail with their SMs idle, and the persistent indexer, which keeps every
// SM streaming to the end, followed by the streaming Top-K is faster there.
bool indexer_topk_eligible(const IndexerArgs& a) {
  const int64_t ntiles = ((int64_t)a.seqs.max_k_len + kBM - 1) / kBM;
  const int64_t c_cap = (ntiles + kMaxTiles - 1) / kMaxTiles;
  return (a.idx_dtype == DSA_BF16 || a.idx_dtype == DSA_FP8_E4M3) && a.h_idx == kHI &&
         a.d_idx == kDI && c_cap <= kMaxCluster &&
         (int64_t)a.seqs.total_q * c_cap <= num_sms() &&
         (a.idx_dtype != DSA_FP8_E4M3 || (reinterpret_cast<uintptr_t>(a.k_scale) & 15) == 0);
}

int launch_indexer_topk(const IndexerArgs& a, int top_k, int32_t* idx, float* vals,
                        cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  return a.idx_dtype == DSA_FP8_E4M3 ? launch_typed<true>(a, top_k, idx, vals, stream)
                                     : launch_typed<false>(a, top_k, idx, vals, stream);
}

}  // namespace dsa
