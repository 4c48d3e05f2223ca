// Lightning-Indexer scores on the 5th-generation tensor cores (tcgen05), for
// H_I = 64 heads of width d_I = 128 in bf16 or FP8 E4M3.
//
//   I[t, s] = Σ_j w[t,j] · ReLU(q_I[t,j,:] · k_I[s,:])      s <= pos(t)
//
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
// LLMs", §4.1: batched dot product of the indexer query with the K cache, then
// the weighted sum over heads, read straight from the K cache.)
//
// Work unit: a block of QB consecutive query rows of one sequence × one tile of 128
// keys.  The tile is the MMA's M = 128 (one key per TMEM lane), the block's QB × 64
// heads are N, K = d_I.  Decode uses QB = 1 (N = 64); prefill uses QB = 4: N = 256
// runs the tensor core at its full rate (an N = 64 MMA takes 46 clocks for a quarter of
// the work an N = 256 one does in 128) and each key tile read from L2 serves four
// query rows instead of one.
// The per-head logits z[t, j, s] exist only in tensor memory: the epilogue
// reads its key's 64 columns and reduces them to one score (ReLU, · w, Σ_j)
// without any cross-thread reduction.  For FP8 the scales fold in as
// I = k_scale[s] · Σ_j (w·q_scale)[t,j] · ReLU(z8) (all scales are positive).
// MXFP8 (one E8M0 scale per 32 elements of a head or key; "… New-Architecture
// LLMs" §5.1) cannot fold a scale past the sum over d_I, so each of a tile's four
// K = 32 MMAs writes its own accumulator (4 × 64 columns, double buffered: all 512)
// and the epilogue forms z_j = Σ_g 2^(ek_g) 2^(eq_jg) z_jg before the ReLU, two heads
// at a time with packed fp32x2 arithmetic (QB = 1 only).
//
// Schedule: the tiles of all blocks are laid end to end (a block whose last row
// sits at position p has floor(p/128) + 1 of them) and each persistent CTA takes
// one contiguous, equal share, so a long-history block is simply spread over more
// CTAs than a short one.  Each CTA derives the tile layout itself from cu_q / cu_k
// in closed form.  QB = 1: per sequence F(L) - F(L - T) with
// F(n) = Σ_{p<n} (floor(p/128) + 1) = n + 64 q (q - 1) + r q  (q = n / 128, r = n % 128).
// QB = 4: the first nb full blocks of a sequence hold nb + G(a + nb) - G(a) tiles,
// a = (L - T + 3) / 4, G(n) = Σ_{x<n} floor(x/32); a partial last block holds
// floor((L-1)/128) + 1.
// Warp roles: warp 0 issues TMA loads (a ring of key tiles, query blocks), warp 1
// owns TMEM and issues the MMAs, the other warps run the epilogue on a
// double-buffered TMEM accumulator (QB = 4: two warps per TMEM lane quarter, each
// taking two of the block's rows).  Every wait is bounded (DSA_FLAG_TIMEOUT).
#include "dsa_internal.cuh"
#include "tc_sm100.cuh"
#include "tile_sched.cuh"

namespace dsa {
namespace {

using namespace tc;
using namespace sched;

constexpr int kMaxSeqs = 4096;  // sequences per launch on this path (tile table in smem)

template <bool FP8, int QB, bool MX = false>
struct Cfg {
  static_assert(!MX || (FP8 && QB == 1), "MXFP8 runs with one query row per block");
  static constexpr int BM = 128;   // keys per tile (MMA M)
  static constexpr int HI = 64;    // heads per query row
  static constexpr int N = HI * QB;  // MMA N: the block's heads
  static constexpr int DI = 128;   // head width (MMA K total)
  static constexpr int ES = FP8 ? 1 : 2;
  static constexpr int ROWB = DI * ES;             // bytes per key row (128 or 256)
  static constexpr int ATOMS = ROWB / 128;         // 128-byte swizzle atoms per row
  static constexpr int KTILE = BM * ROWB;          // 32 KB bf16, 16 KB fp8
  static constexpr int QTILE = N * ROWB;           // one query block
  static constexpr int NQ = QB == 1 ? 2 : 1;       // query-block buffers
  static constexpr int NS = QB == 1 ? (FP8 ? 8 : 4) : (FP8 ? 6 : 3);  // key-tile stages
  static constexpr int KSTEPS = FP8 ? 4 : 8;       // MMAs per tile (32 B of K each)
  static constexpr int ACC_COLS = MX ? 4 * N : N;  // fp32 accumulator columns (MX: per group)
  static constexpr int TMEM_COLS = 2 * ACC_COLS;   // double buffered
  static constexpr int EPI_WARPS = 8;
  // QB = 1: two groups of four warps take alternate tiles (group g owns accumulator g), so
  // a tile's epilogue has two MMA periods; QB = 4: one group, two warps per lane quarter
  static constexpr int GROUPS = QB == 1 ? 2 : 1;
  static constexpr int GROUP_WARPS = EPI_WARPS / GROUPS;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int RPW = QB * 4 / GROUP_WARPS;  // query rows per epilogue warp
  // per-row histograms: 32-bit counters for one row, 16-bit ones (flushed before they
  // can overflow) for a block of four
  static constexpr int HIST_BYTES = QB == 1 ? kHistBins * 4 : QB * kHistBins * 2;
  // FP8: a ring of per-key scales, one slot per key tile: 132 floats from the tile's first
  // key rounded down to a multiple of 4 (a TMA box must start 16-byte aligned), four
  // more slots than key stages (the epilogue reads a tile's scales up to two tiles after
  // its MMA has released the key stage)
  static constexpr int NSC = FP8 ? NS + 4 : 0;
  static constexpr int SC_BOX = BM + 4;
  static constexpr int SC_BYTES = SC_BOX * 4;      // 528 bytes a box
  static constexpr int SC_SLOT = 640;              // slot stride (128-byte aligned copies)
  static constexpr int SQ_FLOATS = MX ? HI * 4 : 0;  // MX: per warp, the row's group scales
  static constexpr int MISC = 512 /*barriers*/ + EPI_WARPS * RPW * HI * 4 /*weights*/ +
                              EPI_WARPS * SQ_FLOATS * 4 + 64;
  static constexpr int SMEM_FIXED =
      NS * KTILE + NQ * QTILE + HIST_BYTES + NSC * SC_SLOT + MISC + 1024 /*align*/;
  static_assert(TMEM_COLS <= 512, "TMEM");
};

constexpr int kQBMaxSeqs = 64;   // sequences per launch of the QB = 4 kernel (table in smem)
constexpr int kFlushItems = 256; // QB = 4: tiles between flushes (a 16-bit bin grows <= 128 a tile)

struct Params {
  Seqs seqs;
  const float* w;
  const float* q_scale;
  const float* k_scale;
  float* scores;    // row t - r0 holds query row t
  int64_t ld;
  uint32_t* status;
  uint32_t* hist;  // [rows][kHistBins] or null (row t - r0)
  int r0, r1;      // the packed query rows scored
};

// Block-wide exclusive prefix sum over NW warps (two barriers).
template <int NW>
__device__ __forceinline__ uint32_t scan_block(uint32_t v, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  cta_sync();
  uint32_t before = 0, tot = 0;
  for (int w = 0; w < NW; ++w) {
    if (w < warp) before += ws[w];
    tot += ws[w];
  }
  *total = tot;
  cta_sync();
  return before + x - v;
}

// Four 16-column TMEM loads of this warp's 32 lanes, `stride` columns apart (the four MXFP8
// group accumulators of 16 heads), then one wait.
__device__ __forceinline__ void tmem_ld16x4(uint32_t taddr, uint32_t stride, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%65];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47}, [%66];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%67];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + stride), "r"(taddr + 2 * stride), "r"(taddr + 3 * stride)
      : "memory");
}

template <bool FP8, int QB, bool MX>
__global__ void __launch_bounds__(Cfg<FP8, QB, MX>::THREADS, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap smap, Params p) {
  using C = Cfg<FP8, QB, MX>;
  static_assert(2 * C::NS + 4 + 4 + 3 + C::NSC <= 64, "barrier area");
  constexpr int NSCM = C::NSC > 0 ? C::NSC : 1;  // scale slots (as a modulus)
  constexpr int EPI_THREADS = 32 * C::EPI_WARPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ks = smem;                                  // NS key tiles
  uint8_t* qs = ks + C::NS * C::KTILE;                 // NQ query blocks
  uint32_t* hs = reinterpret_cast<uint32_t*>(qs + C::NQ * C::QTILE);  // row-segment histograms
  float* scs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(hs) + C::HIST_BYTES);  // NSC slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(scs) + C::NSC * C::SC_SLOT);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* q_full = k_empty + C::NS;
  uint64_t* q_empty = q_full + 2;
  uint64_t* acc_full = q_empty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* epi_a = drain + 1;     // the epilogue threads: row segment scored
  uint64_t* epi_b = drain + 2;     // the epilogue threads: histograms flushed
  uint64_t* sc_empty = drain + 3;  // [NSC] FP8: the tile's epilogue warps have read its scales
  float* wsm = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512);  // [warps][RPW][64]
  // MX: [warps][32 head pairs][4 groups] float2 (heads 2i, 2i+1 of a group side by side)
  float4* sqm = reinterpret_cast<float4*>(wsm + C::EPI_WARPS * C::RPW * C::HI);
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(wsm + C::EPI_WARPS * C::RPW * C::HI + C::EPI_WARPS * C::SQ_FLOATS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* scan_ws = tmem_slot + 2;                   // [THREADS / 32]
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::SMEM_FIXED - 1024);
  const int B = p.seqs.B;
  int32_t* st = tab;
  int32_t* cq = st + (B + 1);
  int32_t* ck = cq + (B + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile table of the sequences (every CTA builds its own copy) ----
  uint32_t carry = 0;
  for (int base = 0; base < B; base += C::THREADS) {
    const int b = base + threadIdx.x;
    uint32_t n = 0;
    if (b < B) {
      const int q0 = __ldg(p.seqs.cu_q + b), q1 = __ldg(p.seqs.cu_q + b + 1);
      const int k0 = __ldg(p.seqs.cu_k + b), k1 = __ldg(p.seqs.cu_k + b + 1);
      const int T = q1 - q0, L = k1 - k0;
      const bool ok = q0 >= 0 && T >= 0 && T <= L && k0 >= 0 && k1 <= p.seqs.total_k &&
                      L <= p.seqs.max_k_len && q1 <= p.seqs.total_q;
      int cq0, cT, cL;  // the sequence restricted to the rows scored
      clip_seq(q0, q1, k0, k1, p.r0, p.r1, cq0, cT, cL);
      if (ok) n = (uint32_t)seq_tiles<QB>(cT, cL);
      else if (blockIdx.x == 0) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
      cq[b] = q0;
      ck[b] = k0;
    }
    uint32_t tot;
    const uint32_t excl = scan_block<C::THREADS / 32>(n, scan_ws, &tot);
    if (b < B) st[b] = (int32_t)(carry + excl);
    carry += tot;
  }
  if (p.hist)
    for (int i = threadIdx.x; i < C::HIST_BYTES / 4; i += C::THREADS) hs[i] = 0u;
  if (threadIdx.x == 0) {
    st[B] = (int32_t)carry;
    cq[B] = __ldg(p.seqs.cu_q + B);
    ck[B] = __ldg(p.seqs.cu_k + B);
  }
  cta_sync();
  SeqTab tabs{st, cq, ck, B};
  tabs.r0 = p.r0;
  tabs.r1 = p.r1;
  const int total = st[B];
  const int g0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int g1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  if (g0 >= g1) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1);
      mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], C::GROUP_WARPS);
    }
    mbar_init(drain, 1);
    mbar_init(epi_a, EPI_THREADS);
    mbar_init(epi_b, EPI_THREADS);
    for (int i = 0; i < C::NSC; ++i) mbar_init(&sc_empty[i], C::GROUP_WARPS);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
    if (FP8) prefetch_tmap(&smap);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch();  // the Top-K kernel may be scheduled (it waits)

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      Cursor<QB> cur;
      cur.locate(tabs, g0);
      int blocks_seen = 0, issued = 0;
      for (int g = g0, it = 0; g < g1; ++g, ++it) {
        if (g > g0) cur.advance(tabs);
        if (g == g0 || cur.j == 0) {
          dsa_check(cur.t >= 0 && cur.t < p.seqs.total_q, p.status);  // a query block inside q
          const int slot = blocks_seen % C::NQ;
          if (!mbar_wait(&q_empty[slot], ((blocks_seen / C::NQ) & 1) ^ 1, abort_flag, p.status,
                         DSA_FLAG_TIMEOUT)) break;
          mbar_arrive_expect_tx(&q_full[slot], C::QTILE);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_2d(qs + slot * C::QTILE + a * (C::N * 128), &qmap, &q_full[slot],
                        a * (128 / C::ES), cur.t * C::HI);
          ++blocks_seen;
        }
        const int s = it % C::NS;
        if (!mbar_wait(&k_empty[s], ((it / C::NS) & 1) ^ 1, abort_flag, p.status,
                       DSA_FLAG_TIMEOUT)) break;
        const int key0 = cur.k0 + cur.j * C::BM;
        float* sdst = scs + (it % NSCM) * (C::SC_SLOT / 4);
        if (FP8) {
          // the tile's key scales land with its keys (the MMA waits for both)
          const int sl = it % NSCM;
          if (!mbar_wait(&sc_empty[sl], ((it / NSCM) & 1) ^ 1, abort_flag, p.status,
                         DSA_FLAG_TIMEOUT)) break;
          mbar_arrive_expect_tx(&k_full[s], C::KTILE + (p.seqs.paged() ? C::BM * 4 : C::SC_BYTES));
        } else {
          mbar_arrive_expect_tx(&k_full[s], C::KTILE);
        }
        if (!p.seqs.paged()) {
          dsa_check(key0 >= 0 && key0 < p.seqs.cache_rows(), p.status);  // the tile starts in the cache
          if (FP8) tma_load_2d(sdst, &smap, &k_full[s], key0 & ~3, 0);
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_2d_hint(ks + s * C::KTILE + a * (C::BM * 128), &kmap, &k_full[s],
                             a * (128 / C::ES), key0, pol);
        } else {
          // page by page: chunks of cr rows; a chunk past the block's history or on a page
          // outside the cache is read out of bounds (zero fill) and never stored
          const int cr = tile_chunk_rows(p.seqs);
          const int s0 = cur.j * C::BM, nk = cur.pos + cur.nrow;
          for (int q = 0; q < C::BM / cr; ++q) {
            int64_t row = s0 + q * cr < nk ? key_row(p.seqs, cur.b, cur.k0, s0 + q * cr) : -2;
            if (row == -1) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
            if (row < 0) row = p.seqs.cache_rows();
            if (FP8) tma_load_2d(sdst + q * cr, &smap, &k_full[s], (int)row, 0);
            for (int a = 0; a < C::ATOMS; ++a)
              tma_load_2d_hint(ks + s * C::KTILE + a * (C::BM * 128) + q * cr * 128, &kmap,
                               &k_full[s], a * (128 / C::ES), (int)row, pol);
          }
        }
        issued = it + 1;
      }
      // every copy issued has landed before the CTA may exit
      for (int i = (issued > C::NS ? issued - C::NS : 0); i < issued; ++i)
        mbar_wait_drain(&k_full[i % C::NS], (i / C::NS) & 1);
      for (int i = (blocks_seen > C::NQ ? blocks_seen - C::NQ : 0); i < blocks_seen; ++i)
        mbar_wait_drain(&q_full[i % C::NQ], (i / C::NQ) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = FP8 ? idesc_e4m3(128, C::N) : idesc_bf16(128, C::N);
      Cursor<QB> cur;
      cur.locate(tabs, g0);
      int blocks_seen = 0;
      for (int g = g0, it = 0; g < g1; ++g, ++it) {
        if (g > g0) cur.advance(tabs);
        if (g == g0 || cur.j == 0) {
          if (!mbar_wait(&q_full[blocks_seen % C::NQ], (blocks_seen / C::NQ) & 1, abort_flag,
                         p.status, DSA_FLAG_TIMEOUT)) break;
          tc_fence_after();
          ++blocks_seen;
        }
        const int slot = (blocks_seen - 1) % C::NQ;
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
          const uint64_t bd = sdesc_sw128(b0 + atom * (C::N * 128) + off, 16, 1024);
          if (MX) mma_e4m3(tmem + acc * C::ACC_COLS + kk * C::N, ad, bd, idesc, false);
          else if (FP8) mma_e4m3(tmem + acc * C::ACC_COLS, ad, bd, idesc, kk > 0);
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
    // ---------------- epilogue: TMEM lane quarter warp % 4, rows rgrp * RPW .. ----------------
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int grp = C::GROUPS == 2 ? ew >> 2 : 0;   // tiles it with it % GROUPS == grp
    const int rgrp = C::GROUPS == 2 ? 0 : ew >> 2;  // QB = 4: rows {2 rgrp, 2 rgrp + 1}
    const int e = threadIdx.x - 64;  // 0 .. EPI_THREADS - 1
    float* wq = wsm + ew * C::RPW * C::HI;
    int nseg = 0, since = 0;
    Cursor<QB> cur;
    cur.locate(tabs, g0);
    float wreg[QB == 1 ? C::HI : 1];  // QB = 1: the row's head weights, in registers
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
      if (g > g0) cur.advance(tabs);
      if (g == g0 || cur.j == 0) {
        __syncwarp();
#pragma unroll
        for (int rr = 0; rr < C::RPW; ++rr) {
          const int r = rgrp * C::RPW + rr;
          const int64_t t = cur.t + (r < cur.nrow ? r : 0);
          float w0 = __ldg(p.w + t * C::HI + lane);
          float w1 = __ldg(p.w + t * C::HI + lane + 32);
          if (FP8 && !MX) {
            w0 *= __ldg(p.q_scale + t * C::HI + lane);
            w1 *= __ldg(p.q_scale + t * C::HI + lane + 32);
          }
          if (MX) {
            // heads 2·lane and 2·lane + 1: their four E8M0 group scales, paired per group
            const uint32_t* qb = reinterpret_cast<const uint32_t*>(p.q_scale) + t * C::HI;
            const uint32_t a0 = __ldg(qb + 2 * lane), a1 = __ldg(qb + 2 * lane + 1);
            float4* d = sqm + ew * (C::SQ_FLOATS / 4) + 2 * lane;
            d[0] = make_float4(e8m0_to_f32(a0 & 0xff), e8m0_to_f32(a1 & 0xff),
                               e8m0_to_f32((a0 >> 8) & 0xff), e8m0_to_f32((a1 >> 8) & 0xff));
            d[1] = make_float4(e8m0_to_f32((a0 >> 16) & 0xff), e8m0_to_f32((a1 >> 16) & 0xff),
                               e8m0_to_f32(a0 >> 24), e8m0_to_f32(a1 >> 24));
          }
          wq[rr * C::HI + lane] = w0;
          wq[rr * C::HI + lane + 32] = w1;
        }
        __syncwarp();
        if (QB == 1)
#pragma unroll
          for (int jj = 0; jj < C::HI; ++jj) wreg[jj] = wq[jj];
      }
      const bool mine = C::GROUPS == 1 || (it & 1) == grp;
      if (mine) {
      const int acc = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (it >> 1) & 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT)))
        break;
      tc_fence_after();
      float ksc = 1.f;
      if (FP8) {
        // this thread's key scale, landed with the tile (its MMA waited for both); keys past
        // the block read a neighbour's scale or the zero fill, and are not stored
        const int sl = it % NSCM;
        const int sh = p.seqs.paged() ? 0 : ((cur.k0 + cur.j * C::BM) & 3);
        ksc = scs[sl * (C::SC_SLOT / 4) + sh + quarter * 32 + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc_empty[sl]);
      }
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * C::ACC_COLS +
                             rgrp * C::RPW * C::HI;
      // Σ_j w_j · ReLU(z_j) as four interleaved partial sums (a short dependency chain)
      float sum[C::RPW];
      if (MX) {
        // this key's four group scales (one 4-byte word in the scale ring), each paired
        float2 ek[4];
        const uint32_t kb = __float_as_uint(ksc);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float f = e8m0_to_f32((kb >> (8 * g)) & 0xff);
          ek[g] = make_float2(f, f);
        }
        const float4* sq = sqm + ew * (C::SQ_FLOATS / 4);
        float2 part[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int hc = 0; hc < C::HI / 16; ++hc) {
          uint32_t r[64];  // groups 0..3 of heads 16·hc .. 16·hc + 15
          tmem_ld16x4(taddr + 16 * hc, C::N, r);
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2) {
            const int jp = 8 * hc + q2;  // head pair: heads 2·jp, 2·jp + 1
            const float4 s01 = sq[2 * jp], s23 = sq[2 * jp + 1];
            const float2 c0 = __fmul2_rn(ek[0], make_float2(s01.x, s01.y));
            const float2 c1 = __fmul2_rn(ek[1], make_float2(s01.z, s01.w));
            const float2 c2 = __fmul2_rn(ek[2], make_float2(s23.x, s23.y));
            const float2 c3 = __fmul2_rn(ek[3], make_float2(s23.z, s23.w));
            float2 z = __fmul2_rn(c0, make_float2(__uint_as_float(r[2 * q2]),
                                                  __uint_as_float(r[2 * q2 + 1])));
            z = __ffma2_rn(c1, make_float2(__uint_as_float(r[16 + 2 * q2]),
                                           __uint_as_float(r[16 + 2 * q2 + 1])), z);
            z = __ffma2_rn(c2, make_float2(__uint_as_float(r[32 + 2 * q2]),
                                           __uint_as_float(r[32 + 2 * q2 + 1])), z);
            z = __ffma2_rn(c3, make_float2(__uint_as_float(r[48 + 2 * q2]),
                                           __uint_as_float(r[48 + 2 * q2 + 1])), z);
            const float2 wp = make_float2(wreg[2 * jp], wreg[2 * jp + 1]);
            part[q2 & 1] = __ffma2_rn(wp, make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)),
                                      part[q2 & 1]);
          }
        }
        sum[0] = (part[0].x + part[1].x) + (part[0].y + part[1].y);
      } else {
#pragma unroll
        for (int rr = 0; rr < C::RPW; ++rr) {
          float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t r[32];
            tmem_ld32(taddr + rr * C::HI + 32 * h2, r);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const float wj = QB == 1 ? wreg[32 * h2 + jj] : wq[rr * C::HI + 32 * h2 + jj];
              part[jj & 3] = fmaf(wj, fmaxf(__uint_as_float(r[jj]), 0.f), part[jj & 3]);
            }
          }
          sum[rr] = (part[0] + part[1]) + (part[2] + part[3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      const int s = cur.j * C::BM + quarter * 32 + lane;
#pragma unroll
      for (int rr = 0; rr < C::RPW; ++rr) {
        const int r = rgrp * C::RPW + rr;  // the same in the whole warp
        const bool valid = r < cur.nrow && s <= cur.pos + r;
        float v = sum[rr];
        if (FP8 && !MX) v *= ksc;
        if (valid && dsa_check(cur.t + r - p.r0 >= 0 && cur.t + r < p.r1 && s < p.ld, p.status))
          p.scores[(int64_t)(cur.t + r - p.r0) * p.ld + s] = v;
        if (p.hist) {
          // scores of neighbouring keys share bins: one shared-memory atomic per bin per warp
          if (valid) {
            const uint32_t bin = order_key(v) >> 20;
            if (QB == 1) atomicAdd(&hs[bin], 1u);
            else atomicAdd(&hs[(r * kHistBins + bin) >> 1], 1u << (16 * (bin & 1)));
          }
        }
      }
      }  // mine
      const bool seg_end = g + 1 == g1 || cur.j + 1 == cur.ntiles;
      if (p.hist && (seg_end || (QB > 1 && ++since == kFlushItems))) {
        // add this CTA's counts to the rows' histograms, then start again from zero
        since = 0;
        mbar_arrive(epi_a);
        if (!__all_sync(0xffffffffu, mbar_wait(epi_a, nseg & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) break;
        if (QB == 1) {
          uint32_t* grow = p.hist + (int64_t)(cur.t - p.r0) * kHistBins;
          for (int bin = e; bin < kHistBins; bin += EPI_THREADS) {
            const uint32_t v = hs[bin];
            if (v) { atomicAdd(grow + bin, v); hs[bin] = 0u; }
          }
        } else {
          for (int wi = e; wi < cur.nrow * (kHistBins / 2); wi += EPI_THREADS) {
            const uint32_t v = hs[wi];
            if (v) {
              const int r = wi / (kHistBins / 2), b0 = 2 * (wi % (kHistBins / 2));
              uint32_t* grow = p.hist + (int64_t)(cur.t + r - p.r0) * kHistBins;
              if (v & 0xffffu) atomicAdd(grow + b0, v & 0xffffu);
              if (v >> 16) atomicAdd(grow + b0 + 1, v >> 16);
              hs[wi] = 0u;
            }
          }
        }
        mbar_arrive(epi_b);
        if (!__all_sync(0xffffffffu, mbar_wait(epi_b, nseg & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) break;
        ++nseg;
      }
    }
  }

  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool FP8, int QB, bool MX = false>
int launch_typed(const IndexerArgs& a, float* scores, int64_t ld, cudaStream_t stream) {
  using C = Cfg<FP8, QB, MX>;
  CUtensorMap kmap, qmap, smap;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int cr = tile_chunk_rows(a.seqs);  // key rows per copy (a page, for small pages)
  int rc = make_tmap_2d(&kmap, dt, a.k_idx, C::DI, (uint64_t)a.seqs.cache_rows(), C::ROWB,
                        128 / C::ES, (uint32_t)cr);
  if (rc != DSA_OK) return rc;
  rc = make_tmap_2d(&qmap, dt, a.q_idx, C::DI, (uint64_t)a.seqs.total_q * C::HI, C::ROWB,
                    128 / C::ES, C::N);
  if (rc != DSA_OK) return rc;
  if (FP8) {
    // k_scale as one row of total_k 4-byte words (no swizzle), read in boxes of 132: an fp32
    // scale per key, or (MX) a key's four E8M0 group scales
    const uint64_t rows = (uint64_t)a.seqs.cache_rows();
    rc = make_tmap_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.k_scale, rows, 1,
                      align_up((size_t)rows * 4, 16), a.seqs.paged() ? (uint32_t)cr : C::SC_BOX,
                      1, false);
    if (rc != DSA_OK) return rc;
  } else {
    smap = kmap;  // unused
  }
  const int smem = C::SMEM_FIXED + (int)align_up(3 * sizeof(int32_t) * (a.seqs.B + 1), 16);
  auto kern = indexer_tc_kernel<FP8, QB, MX>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("indexer_tc: smem attribute");
  const int r1 = a.row1 < a.seqs.total_q ? a.row1 : a.seqs.total_q;
  if (r1 <= a.row0) return DSA_OK;
  const int64_t bound = (int64_t)(r1 - a.row0) * ((a.seqs.max_k_len + C::BM - 1) / C::BM);
  const int grid = (int)(bound < num_sms() ? bound : num_sms());
  Params p{a.seqs, a.w, a.q_scale, a.k_scale, scores, ld, a.status, a.hist, a.row0, r1};
  DSA_LAUNCH(MX ? "indexer_tc_mxfp8"
             : FP8 ? (QB == 1 ? "indexer_tc_fp8" : "indexer_tc_fp8_qb4")
                   : (QB == 1 ? "indexer_tc_bf16" : "indexer_tc_bf16_qb4"),
             stream, kern<<<grid, C::THREADS, smem, stream>>>(kmap, qmap, smap, p));
  return check_launch("indexer_tc");
}

}  // namespace

bool indexer_tc_eligible(const IndexerArgs& a) {
  // tiles of the whole problem must stay below 2^31 (int32 item indices)
  const int64_t bound = (int64_t)a.seqs.total_q * ((a.seqs.max_k_len + 127) / 128);
  // (FP8: the key scales are read by TMA, which wants a 16-byte aligned base)
  const bool q8 = a.idx_dtype == DSA_FP8_E4M3 || a.idx_dtype == DSA_MXFP8_E4M3;
  return (a.idx_dtype == DSA_BF16 || q8) && a.h_idx == 64 && a.d_idx == 128 &&
         a.seqs.B <= kMaxSeqs && bound < (int64_t(1) << 31) &&
         (!q8 || (reinterpret_cast<uintptr_t>(a.k_scale) & 15) == 0);
}

// blocks of four query rows when sequences hold several queries each (prefill)
bool indexer_tc_blocks4(const IndexerArgs& a) {
  return a.seqs.B <= kQBMaxSeqs && a.seqs.total_q >= 4 * a.seqs.B;
}

int launch_indexer_tc(const IndexerArgs& a, float* scores, int64_t ld, cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  const bool qb4 = indexer_tc_blocks4(a);
  // MXFP8 keeps four accumulators per tile, which leaves TMEM room for one query row per block
  if (a.idx_dtype == DSA_MXFP8_E4M3) return launch_typed<true, 1, true>(a, scores, ld, stream);
  if (a.idx_dtype == DSA_FP8_E4M3)
    return qb4 ? launch_typed<true, 4>(a, scores, ld, stream)
               : launch_typed<true, 1>(a, scores, ld, stream);
  return qb4 ? launch_typed<false, 4>(a, scores, ld, stream)
             : launch_typed<false, 1>(a, scores, ld, stream);
}

}  // namespace dsa
