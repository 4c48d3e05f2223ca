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
// One persistent CTA per SM, all resident at once (cooperative launch).  The rows' key
// histories, cut into 128-key tiles and laid end to end in row order, are split into equal
// contiguous shares, one per CTA, so every SM streams the same number of bytes whatever the
// mix of history lengths; a share covers the end of one row, whole rows and the start of
// another ("runs").  Scoring: TMA brings the key tiles two at a time into a ring of pair
// stages, one thread issues tcgen05.mma (M = 128 keys x N = 64 heads x K = 128) for both
// tiles of a pair into one of two TMEM accumulator pairs against the run's query block
// (two query buffers), and eight epilogue warps (one per tile of the pair and TMEM lane
// quarter) reduce each key's 64 head logits to its score.  An N = 64 MMA takes ~50 clocks
// to issue and every barrier wait or commit costs about as much, so stages and accumulators
// come in pairs of tiles.  Each score stays in a column of tensor memory (up to 256 tiles,
// 32,768 keys, per CTA) and is counted into a histogram of its top 11 order-preserving
// key bits: in shared memory for the CTA's first and last runs (rows it shares with other
// CTAs; added into the row's histogram in global memory after scoring), straight in the
// row's global histogram for the rows wholly inside the CTA.
//
// Selection is exact and deterministic.  The CTAs holding runs of one row wait for each
// other through the row's counter (no grid-wide barrier); after scoring, two groups of four
// epilogue warps select for alternate runs of the CTA at the same time.
//   1. the row's histogram is complete: each run finds the digit B* holding the k-th
//      largest key, counts its keys above B*, and writes its keys in B* (the candidates,
//      with their positions) to the row's candidate list bucketed by the next five key
//      bits, with its bucket counts (a weighted sum over 64 heads spreads little, so 16
//      bits are needed before the keys left are few);
//   2. the list is complete: each run finds from the bucket counts the bucket of the k-th
//      key, reads that bucket's candidates of every run, resolves the remaining 16 key
//      bits by radix select over them (the exact key T of the k-th largest score and how
//      many keys equal to T are kept: those at the smallest positions), counts its keys
//      above and equal to T per (tile, lane quarter), adds the kept keys of the runs
//      before it, and writes its kept positions straight to their slots: the row's
//      selected positions in ascending order.
// Every wait is bounded (DSA_FLAG_TIMEOUT).
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
constexpr int kMaxRows = 128;            // query rows of a launch (one setup thread each)
constexpr int kMaxCtas = 256;            // CTAs of a launch (one per SM)
constexpr int kNB1 = 2048;               // first round: key bits 31..21
constexpr int kSub = 32;                 // candidates bucketed by key bits 20..16
constexpr int kNB2 = 128, kNB3 = 512;    // later rounds: key bits 15..9, 8..0
constexpr int kRec = kSub + 4;           // a run's record: bucket counts, keys above B*, pad
constexpr int kRowWords = 8;             // a row counter's own 32 bytes
// In the split of the tiles, every row's tiles are preceded by this many placeholder tiles,
// so a CTA whose share crosses a row start (and then selects for two runs, ~6 µs more)
// streams that many fewer tiles (~0.7 µs each) and ends with the others.
constexpr int kRowLead = 8;
// A row's counter (status block) has three 8-bit fields: the row's histogram is clear (set
// by the CTA holding its first tile), and the CTAs holding runs of the row whose counts,
// and whose candidates, are in.  There are two sets: a launch uses set (epoch & 1) and
// clears the other one, which the launch before it used.  The epoch is the launch's number,
// from a counter every CTA of every launch increments once (each launch has one CTA per SM).
constexpr uint32_t kZ = 1u, kA = 1u << 8, kB = 1u << 16;
static_assert(kScoreCol + kMaxTiles <= kTmemCols, "TMEM layout");
static_assert(kMaxRows <= kThreads, "one setup thread per row");

// A run: consecutive tiles of one row held by one CTA.
struct Run {
  int t, b, n, k;        // row, sequence, keys in its history, keys kept
  int k0;                // first cache row of the sequence (contiguous caches)
  int start, nt;         // the row's first tile in the launch's tile order, its tiles
  int l0, l1, j0;        // the CTA's tiles [l0, l1) are the row's tiles j0, j0 + 1, ...
  int pgo, pg0;          // paged caches: its pages' offset in the CTA's list, first page
  int nr, rank;          // CTAs holding runs of the row; this CTA's rank among them
  int cf, cl;            // the first and last of those CTAs
  int slot;              // its counts: shared-memory histogram 0 or 1, or -1 (global)
  uint32_t bstar, above;  // first round: the 11-bit digit B*, the row's keys above it
};

template <bool FP8>
struct Cfg {
  static constexpr int ES = FP8 ? 1 : 2;
  static constexpr int ROWB = kDI * ES;              // bytes per key row
  static constexpr int ATOMS = ROWB / 128;           // 128-byte swizzle atoms per row
  static constexpr int KTILE = kBM * ROWB;           // 32 KB bf16, 16 KB fp8
  static constexpr int STAGE = kPair * KTILE;
  static constexpr int QTILE = kHI * ROWB;           // a row's query heads
  static constexpr int NSS = FP8 ? 4 : 2;            // pair stages (128 KB either way)
  static constexpr int RING = NSS * STAGE;
  static constexpr int KSTEPS = FP8 ? 4 : 8;         // MMAs per tile (32 B of K each)
  // FP8: per-key scales by TMA with their key tile (132 floats from the tile's first key
  // rounded down to a multiple of 4), released by the epilogue; four spare slots
  static constexpr int NSC = FP8 ? kPair * NSS + 4 : 0;
  static constexpr int SC_BOX = kBM + 4;
  static constexpr int SC_BYTES = SC_BOX * 4;
  static constexpr int SC_SLOT = 640;
  // After scoring the key ring holds the CTA's scores (tile-major, 128 keys a tile), and
  // the query buffers and the first / last run's counts hold the runs' records of a row
  // and then a row's candidates (key, position).
  static constexpr int OFF_Q = RING;                          // two query buffers
  static constexpr int OFF_HS = OFF_Q + 2 * QTILE;            // first / last run's counts
  static constexpr int SPARE = 2 * QTILE + 2 * kNB1 * 4;      // those two, contiguous
  static constexpr uint32_t CAND_CAP = SPARE / 8;
  static_assert(kMaxCtas * kSub * 4 <= SPARE, "the runs' bucket counts of a row fit");
  static constexpr int OFF_HR = OFF_HS + 2 * kNB1 * 4;        // counts of the later rounds
  static constexpr int OFF_SC = OFF_HR + kNB3 * 4;            // FP8 scale ring
  static constexpr int OFF_PG = OFF_SC + NSC * SC_SLOT;       // the CTA's pages
  static constexpr int MAX_PG = kMaxTiles * (kBM / 16) + kMaxRows;  // 16-row pages at most
  static constexpr int OFF_RUN = OFF_PG + MAX_PG * 4;
  static constexpr int OFF_OWN = OFF_RUN + kMaxRows * (int)sizeof(Run);
  static constexpr int OFF_TB = OFF_OWN + kMaxRows * 8;        // the CTAs' first tiles
  static constexpr int OFF_SEG = OFF_TB + (kMaxCtas + 4) * 4;  // a row's runs: candidates
  static constexpr int OFF_MISC = OFF_SEG + 2 * kMaxCtas * 4;  // mbarriers (8-byte) first
  static constexpr int MISC = 1024;
  static constexpr int SMEM = OFF_MISC + MISC + 1024 /*alignment*/;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(OFF_Q % 1024 == 0 && QTILE % 1024 == 0, "swizzled TMA tiles: 1024-byte aligned");
  static_assert(OFF_SC % 128 == 0 && SC_SLOT % 128 == 0, "TMA destinations: 128-byte aligned");
  static_assert(OFF_RUN % 8 == 0 && OFF_OWN % 8 == 0 && OFF_TB % 16 == 0 && OFF_SEG % 16 == 0,
                "tables");
  static_assert(OFF_MISC % 16 == 0, "mbarriers: 8-byte aligned");
};

struct Params {
  Seqs seqs;
  int top_k;
  const float* w;
  const float* q_scale;
  const float* k_scale;
  int32_t* idx;
  float* vals;
  uint32_t* status;
  uint32_t* launch;   // the launch counter
  uint32_t* rowsync;  // [2][kMaxRows][kRowWords] the rows' counters
  uint32_t* hist;     // [total_q][kNB1] every row's counts of key bits 31..21
  uint32_t* rec;      // [total_q][gridDim.x][kRec] every run's record, by its rank in the row
  uint2* cand;        // [total_q][cand_ld] every row's candidates (key, position), each
                      // run's at the run's first key position, by bucket
  int64_t cand_ld;
};

struct Xch {
  uint32_t epoch;                  // this launch's number
  uint32_t mytiles;                // the CTA's tiles
  uint32_t res[4];                 // find_digit's answer
  uint32_t gtb, eqb;               // kept keys above / equal to T before the run
  uint32_t ncand;                  // the run's candidates staged
  uint32_t ab;                     // keys above the 16-bit digit in the row's earlier runs
  uint32_t d5, above, nc, gt;      // bucket of the 16-bit digit, keys above it / in it; run's keys above B*
  uint32_t bcnt[kSub], boff[kSub], bcur[kSub];  // the run's candidates by bucket
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Packed query row t -> (sequence, position) from the sequences' offsets in shared memory;
// the same checks as query_row_info.
__device__ __forceinline__ bool row_info_smem(const Seqs& s, const int* cuq, const int* cuk,
                                              int t, RowInfo& r, uint32_t* status) {
  int lo = 0, hi = s.B - 1;
  while (lo < hi) {  // last b with cu_q[b] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (cuq[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int q0 = cuq[lo], q1 = cuq[lo + 1], k0 = cuk[lo], k1 = cuk[lo + 1];
  const int T = q1 - q0, L = k1 - k0;
  if (!(t >= q0 && t < q1 && T <= L && k0 >= 0 && k1 <= s.total_k && L <= s.max_k_len &&
        q1 <= s.total_q)) {
    atomicOr(status, DSA_FLAG_BAD_SEQS);
    return false;
  }
  r.b = lo;
  r.pos = L - T + (t - q0);
  r.k0 = k0;
  r.L = L;
  return true;
}

// One thread: waits (bounded) until the 8-bit field at bit `sh` of a row counter reaches
// n.  A CTA whose own work already failed stops waiting (its results are not written).
__device__ __forceinline__ void row_wait(const uint32_t* c, int sh, uint32_t n,
                                         volatile int* abort, uint32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (((ld_acquire_gpu(c) >> sh) & 255u) < n) {
    if (*abort) return;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(status, DSA_FLAG_TIMEOUT);
      return;
    }
    __nanosleep(20);
  }
  __threadfence();
}

// h[bin] += 1 for every active lane, one atomic per distinct bin of the warp (the scores
// of a row crowd into few bins).  Shared or global memory.
__device__ __forceinline__ void warp_count(uint32_t* h, uint32_t bin, bool on) {
  const uint32_t act = __ballot_sync(0xffffffffu, on);
  if (!on) return;
  const uint32_t same = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == (uint32_t)(__ffs(same) - 1)) atomicAdd(&h[bin], (uint32_t)__popc(same));
}

// Exclusive sums over the CTA's threads of `v` held by lower / higher threads, with the
// total (two barriers).
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* ws, uint32_t* total,
                                               bool suffix = false) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = suffix ? __shfl_down_sync(0xffffffffu, x, o) : __shfl_up_sync(0xffffffffu, x, o);
    if (suffix ? lane + o < 32 : lane >= o) x += y;
  }
  // x: inclusive sum over the warp's lanes on the scanned side (and this lane)
  if (suffix ? lane == 0 : lane == 31) ws[warp] = x;
  cta_sync();
  uint32_t other = 0, tot = 0;
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = ws[w];
    if (suffix ? w > warp : w < warp) other += s;
    tot += s;
  }
  cta_sync();
  *total = tot;
  return other + x - v;
}

// The digit holding the need-th largest of the counts A[0..nb) (all threads; the same
// answer everywhere): (digit, count above it, count in it), through res[0..2].  GLOBAL: A
// was written by other CTAs (read through L2).
template <bool GLOBAL>
__device__ uint3 find_digit(const uint32_t* A, int nb, uint32_t need, uint32_t* res,
                            uint32_t* scan_ws) {
  constexpr int PER = (kNB1 + kThreads - 1) / kThreads;
  const int per = (nb + kThreads - 1) / kThreads;
  const int b0 = min(nb, (int)threadIdx.x * per), b1 = min(nb, b0 + per);
  uint32_t a[PER];
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    a[i] = b0 + i < b1 ? (GLOBAL ? __ldcg(A + b0 + i) : A[b0 + i]) : 0u;
    mine += a[i];
  }
  if (threadIdx.x == 0) res[0] = res[1] = res[2] = 0u;
  uint32_t total;
  const uint32_t above = block_scan(mine, scan_ws, &total, true);
  if (above < need && above + mine >= need) {  // exactly one thread
    uint32_t run = above;
#pragma unroll
    for (int i = PER - 1; i >= 0; --i) {
      if (b0 + i < b1 && run < need && run + a[i] >= need) {
        res[0] = (uint32_t)(b0 + i);
        res[1] = run;
        res[2] = a[i];
      }
      if (b0 + i < b1) run += a[i];
    }
  }
  cta_sync();
  const uint3 r = make_uint3(res[0], res[1], res[2]);
  cta_sync();  // res may be written again right after
  return r;
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
indexer_topk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap smap, Params p) {
  using C = Cfg<FP8>;
  constexpr int NSCM = C::NSC > 0 ? C::NSC : 1;
  constexpr int NBAR = 2 * C::NSS + 4 + 4 + 1 + C::NSC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ks = smem;
  uint8_t* qs = smem + C::OFF_Q;
  uint32_t* hs = reinterpret_cast<uint32_t*>(smem + C::OFF_HS);  // [2][kNB1]
  uint32_t* hr = reinterpret_cast<uint32_t*>(smem + C::OFF_HR);
  float* scs = reinterpret_cast<float*>(smem + C::OFF_SC);
  int32_t* pages = reinterpret_cast<int32_t*>(smem + C::OFF_PG);
  Run* runs = reinterpret_cast<Run*>(smem + C::OFF_RUN);
  int2* own = reinterpret_cast<int2*>(smem + C::OFF_OWN);
  int* tb = reinterpret_cast<int*>(smem + C::OFF_TB);
  int* seg_src = reinterpret_cast<int*>(smem + C::OFF_SEG);   // [kMaxCtas]
  uint32_t* seg_pref = reinterpret_cast<uint32_t*>(seg_src + kMaxCtas);
  float* sc = reinterpret_cast<float*>(smem);                  // after scoring: the scores
  uint32_t* spare = reinterpret_cast<uint32_t*>(smem + C::OFF_Q);  // after scoring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  uint64_t* k_full = bars;                   // [NSS]
  uint64_t* k_empty = k_full + C::NSS;       // [NSS]
  uint64_t* q_full = k_empty + C::NSS;       // [2]
  uint64_t* q_empty = q_full + 2;            // [2]
  uint64_t* acc_full = q_empty + 2;          // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain = acc_empty + 2;
  uint64_t* sc_empty = drain + 1;            // [NSC]
  Xch* X = reinterpret_cast<Xch*>(smem + C::OFF_MISC + 8 * NBAR);
  uint32_t* scan_ws = reinterpret_cast<uint32_t*>(X + 1);  // [kWarps]
  uint32_t* tmem_slot = scan_ws + kWarps;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert(8 * NBAR + sizeof(Xch) + 4 * (kWarps + 2) <= C::MISC, "misc");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int G = gridDim.x, g = blockIdx.x;
  const int total_q = p.seqs.total_q;

  uint32_t ticket = 0;
  if (tid == 0) {
    ticket = atomicAdd(p.launch, 1u);  // used once the setup below is done
    for (int i = 0; i < C::NSS; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < C::NSC; ++i) mbar_init(&sc_empty[i], 4);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
    if (FP8) prefetch_tmap(&smap);
  }
  for (int i = tid; i < 2 * kNB1; i += kThreads) hs[i] = 0u;

  // ---- the launch's tiles: every scored row's history in 128-key tiles, rows in order;
  // this CTA takes tiles [G0, G1) of that order (the same split in every CTA) ----
  // the sequences' offsets, in shared memory for the rows' lookups (one load each)
  const int B = p.seqs.B;
  const bool cu_smem = B < kMaxCtas;
  int* cuq = seg_src;
  int* cuk = reinterpret_cast<int*>(seg_pref);
  if (cu_smem)
    for (int i = tid; i <= B; i += kThreads) {
      cuq[i] = __ldg(p.seqs.cu_q + i);
      cuk[i] = __ldg(p.seqs.cu_k + i);
    }
  cta_sync();
  int my_nt = 0, rn = 0, rk = 0;
  RowInfo ri{};
  bool skip = false;
  if (tid < total_q && (cu_smem ? row_info_smem(p.seqs, cuq, cuk, tid, ri, p.status)
                                : query_row_info(p.seqs, tid, ri, p.status))) {
    rn = ri.pos + 1;
    rk = min(p.top_k, rn);
    skip = rk == rn && p.vals == nullptr;  // every key kept and no score wanted
    my_nt = skip ? 0 : (rn + kBM - 1) / kBM;
  }
  // positions in the split: the rows' tiles in order, each row's after kRowLead placeholders
  const int lead = my_nt > 0 ? kRowLead : 0;
  uint32_t tall;
  const int start = (int)block_scan((uint32_t)(lead + my_nt), scan_ws, &tall) + lead;
  for (int c = tid; c <= G; c += kThreads) tb[c] = (int)((int64_t)c * tall / G);
  cta_sync();
  const int G0 = tb[g], G1 = tb[g + 1];
  const bool ov = my_nt > 0 && G0 < G1 && start < G1 && start + my_nt > G0;
  uint32_t nrun;
  const uint32_t ri_ = block_scan(ov ? 1u : 0u, scan_ws, &nrun);
  const bool owned = skip && tid % G == g;  // written by this CTA without scoring
  uint32_t nown;
  const uint32_t oi = block_scan(owned ? 1u : 0u, scan_ws, &nown);
  const int ns = (int)nrun;
  if (ov) {
    // the CTAs holding the row's tiles (CTAs with empty shares hold none)
    auto cta_of = [&](int x) {
      int c = (int)((int64_t)x * G / tall);
      while (c + 1 < G && tb[c + 1] <= x) ++c;
      while (c > 0 && tb[c] > x) --c;
      return c;
    };
    const int cf = cta_of(start), cl = cta_of(start + my_nt - 1);
    int nr = 0, rank = 0;
    for (int c = cf; c <= cl; ++c) {
      const int ne = tb[c] < tb[c + 1];
      nr += ne;
      if (c < g) rank += ne;
    }
    Run& r = runs[ri_];
    r.t = tid; r.b = ri.b; r.n = rn; r.k = rk; r.k0 = ri.k0;
    r.start = start; r.nt = my_nt;
    r.l0 = 0;  // the CTA's tiles are numbered after the placeholders are left out (below)
    r.l1 = min(start + my_nt, G1) - max(start, G0);
    r.j0 = max(start, G0) - start;
    r.pgo = r.pg0 = 0;
    r.nr = nr;
    r.rank = rank;
    r.cf = cf;
    r.cl = cl;
    // the first and the last run count in shared memory (their rows are shared with other
    // CTAs); runs between them are whole rows of this CTA and count in global memory
    r.slot = ri_ == 0 ? 0 : ((int)ri_ == ns - 1 ? 1 : -1);
    r.bstar = r.above = 0u;
  }
  if (owned) own[oi] = make_int2(tid, rn);
  cta_sync();
  if (tid == 0) {
    X->epoch = ticket / (uint32_t)G;
    int acc = 0;  // the runs' tiles, numbered consecutively
    for (int i = 0; i < ns; ++i) {
      runs[i].l0 = acc;
      acc += runs[i].l1;
      runs[i].l1 = acc;
    }
    X->mytiles = acc;
  }
  cta_sync();
  const int mytiles = (int)X->mytiles;
  const int npairs = (mytiles + kPair - 1) / kPair;
  const uint32_t epoch = X->epoch;
  uint32_t* rsync = p.rowsync + (epoch & 1u) * (kMaxRows * kRowWords);  // this launch's set
  if (tid == 0) {
    uint32_t* other = p.rowsync + ((epoch + 1u) & 1u) * (kMaxRows * kRowWords);
    for (int t = g; t < kMaxRows; t += G) other[t * kRowWords] = 0u;
  }
  // the histograms of the rows that start in this CTA's share are cleared here
  for (int i = 0; i < ns; ++i) {
    const Run& r = runs[i];
    if (r.k == r.n || r.rank != 0) continue;
    uint4* h1 = reinterpret_cast<uint4*>(p.hist + (int64_t)r.t * kNB1);
    for (int j = tid; j < kNB1 / 4; j += kThreads) h1[j] = make_uint4(0u, 0u, 0u, 0u);
  }
  // paged caches: the block-table entries of this CTA's keys, fetched once (the producer
  // would otherwise wait for each lookup before it can issue the copy)
  if (p.seqs.paged()) {
    const int ps = p.seqs.page_size;
    if (tid == 0) {
      int off = 0;
      for (int i = 0; i < ns; ++i) {
        Run& r = runs[i];
        r.pg0 = r.j0 * kBM / ps;
        r.pgo = off;
        off += (min((r.j0 + r.l1 - r.l0) * kBM, r.n) - 1) / ps - r.pg0 + 1;
      }
    }
    cta_sync();
    for (int i = 0; i < ns; ++i) {
      const Run& r = runs[i];
      const int npg = (min((r.j0 + r.l1 - r.l0) * kBM, r.n) - 1) / ps - r.pg0 + 1;
      for (int j = tid; j < npg; j += kThreads)
        pages[r.pgo + j] = __ldg(p.seqs.block_table + (int64_t)r.b * p.seqs.max_pages + r.pg0 + j);
    }
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    __threadfence();  // the cleared histograms before their marks
    for (int i = 0; i < ns; ++i)
      if (runs[i].k < runs[i].n && runs[i].rank == 0) atomicAdd(rsync + runs[i].t * kRowWords, kZ);
    griddep_launch();  // the attention kernel may be scheduled (it waits)
  }

  // ================= scoring: this CTA's tiles G0 .. G1-1 =================
  const int quarter = warp & 3;
  const int half = (warp - 2) >> 2;          // epilogue: tile 2p + half of pair p
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  if (warp == 0) {
    // ---- TMA producer: pair p = tiles 2p, 2p + 1 into stage p % NSS; a run's query
    // block into buffer (run % 2) before its first tile ----
    if (lane == 0 && mytiles > 0) {
      const int sc_bytes = p.seqs.paged() ? kBM * 4 : C::SC_BYTES;
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0, c = 0, qn = 0;
      for (int pp = 0; pp < npairs; ++pp) {
        const int ss = pp % C::NSS;
        const int nt = min(kPair, mytiles - kPair * pp);
        bool ok = true;
        for (int j = 0; j < nt && ok; ++j) {
          const int il = kPair * pp + j;
          while (il >= runs[c].l1) ++c;
          if (c == qn) {  // first tile of run c: its query block
            const int qb = c & 1;
            ok = mbar_wait(&q_empty[qb], ((c >> 1) & 1) ^ 1, abort_flag, p.status, DSA_FLAG_TIMEOUT);
            if (!ok) break;
            mbar_arrive_expect_tx(&q_full[qb], C::QTILE);
            dsa_check(runs[c].t >= 0 && runs[c].t < p.seqs.total_q, p.status);
            for (int a = 0; a < C::ATOMS; ++a)
              tma_load_2d(qs + qb * C::QTILE + a * (kHI * 128), &qmap, &q_full[qb],
                          a * (128 / C::ES), runs[c].t * kHI);
            ++qn;
          }
        }
        if (!ok) break;
        if (!mbar_wait(&k_empty[ss], ((pp / C::NSS) & 1) ^ 1, abort_flag, p.status,
                       DSA_FLAG_TIMEOUT)) break;
        if (FP8)
          for (int j = 0; j < nt && ok; ++j) {
            const int it = kPair * pp + j, sl = it % NSCM;
            ok = mbar_wait(&sc_empty[sl], ((it / NSCM) & 1) ^ 1, abort_flag, p.status,
                           DSA_FLAG_TIMEOUT);
          }
        if (!ok) break;
        mbar_arrive_expect_tx(&k_full[ss], nt * (C::KTILE + (FP8 ? sc_bytes : 0)));
        int rc = c;  // run of the pair's last tile; its first may be in the run before
        for (int j = 0; j < nt; ++j) {
          const int it = kPair * pp + j;
          while (rc > 0 && it < runs[rc].l0) --rc;
          while (it >= runs[rc].l1) ++rc;
          const Run& r = runs[rc];
          const int s0 = (r.j0 + it - r.l0) * kBM;  // the tile's first key position
          uint8_t* kdst = ks + ss * C::STAGE + j * C::KTILE;
          float* sdst = scs + (it % NSCM) * (C::SC_SLOT / 4);
          if (!p.seqs.paged()) {
            const int key0 = r.k0 + s0;
            dsa_check(key0 >= 0 && key0 < p.seqs.cache_rows(), p.status);
            if (FP8) tma_load_2d(sdst, &smap, &k_full[ss], key0 & ~3, 0);
            for (int a = 0; a < C::ATOMS; ++a)
              tma_load_2d_hint(kdst + a * (kBM * 128), &kmap, &k_full[ss], a * (128 / C::ES),
                               key0, pol);
          } else {
            // page by page: chunks of cr rows; a chunk past the history or on a page outside
            // the cache is read out of bounds (zero fill) and never selected
            const int ps = p.seqs.page_size, cr = tile_chunk_rows(p.seqs);
            for (int q = 0; q < kBM / cr; ++q) {
              const int pos = s0 + q * cr;
              int64_t row = -2;
              if (pos < r.n) {
                const int pg = pages[r.pgo + pos / ps - r.pg0];
                row = pg >= 0 && pg < p.seqs.num_pages ? (int64_t)pg * ps + pos % ps : -1;
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
      for (int i = (qn > 2 ? qn - 2 : 0); i < qn; ++i) mbar_wait_drain(&q_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: both tiles of a pair, then one commit each for the stage and the
    // accumulator pair; a run's query buffer is released after its last tile ----
    if (lane == 0 && mytiles > 0) {
      const uint32_t idesc = FP8 ? idesc_e4m3(128, kHI) : idesc_bf16(128, kHI);
      // descriptors of the ring's and of query buffer 0's first K-step; a K-step adds
      // its byte offset / 16 to the start-address field
      const uint64_t bd0 = sdesc_sw128(smem_u32(qs), 16, 1024);
      const uint64_t ad0 = sdesc_sw128(smem_u32(ks), 16, 1024);
      int c = 0, qw = -1;
      bool ok = true;
      for (int pp = 0; pp < npairs && ok; ++pp) {
        const int ss = pp % C::NSS, acc = pp & 1;
        if (!mbar_wait(&acc_empty[acc], ((pp >> 1) & 1) ^ 1, abort_flag, p.status,
                       DSA_FLAG_TIMEOUT)) break;
        if (!mbar_wait(&k_full[ss], (pp / C::NSS) & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT))
          break;
        tc_fence_after();
        const int nt = min(kPair, mytiles - kPair * pp);
        for (int j = 0; j < nt; ++j) {
          const int il = kPair * pp + j;
          while (il >= runs[c].l1) ++c;
          if (c != qw) {
            ok = mbar_wait(&q_full[c & 1], (c >> 1) & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT);
            if (!ok) break;
            tc_fence_after();
            qw = c;
          }
          const uint64_t as = ad0 + (uint64_t)((ss * C::STAGE + j * C::KTILE) >> 4);
          const uint64_t bs = bd0 + (uint64_t)(((c & 1) * C::QTILE) >> 4);
          const uint32_t d = tmem + acc * kAccCols + j * kHI;
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int atom = (kk * 32) / 128, off = (kk * 32) % 128;
            const uint64_t ad = as + (uint64_t)((atom * (kBM * 128) + off) >> 4);
            const uint64_t bd = bs + (uint64_t)((atom * (kHI * 128) + off) >> 4);
            if (FP8) mma_e4m3(d, ad, bd, idesc, kk > 0);
            else mma_bf16(d, ad, bd, idesc, kk > 0);
          }
          if (il + 1 == runs[c].l1) mma_commit(&q_empty[c & 1]);
        }
        if (!ok) break;
        mma_commit(&k_empty[ss]);
        mma_commit(&acc_full[acc]);
      }
      // every MMA issued has completed before TMEM is read for selection or released
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---- epilogue: warp (half, quarter) reduces tile 2p + half of every pair p ----
    // (before the first tile: the histogram of this CTA's first run, if another CTA clears
    // it, is clear before this CTA adds its counts after scoring)
    if (warp == 2 && lane == 0 && ns > 0 && runs[0].k < runs[0].n && runs[0].rank != 0)
      row_wait(rsync + runs[0].t * kRowWords, 0, 1u, abort_flag, p.status);
    float wreg[kHI];  // the run's head weights (FP8: times the query scales)
    int c = -1;
    uint32_t* hc = nullptr;  // where run c's keys are counted
    for (int pp = 0; pp < npairs; ++pp) {
      const int acc = pp & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (pp >> 1) & 1, abort_flag,
                                             p.status, DSA_FLAG_TIMEOUT)))
        break;
      tc_fence_after();
      const int it = kPair * pp + half;
      if (it < mytiles) {
        int cn = c < 0 ? 0 : c;
        while (it >= runs[cn].l1) ++cn;
        if (cn != c) {
          c = cn;
          const int64_t wo = (int64_t)runs[c].t * kHI;
#pragma unroll
          for (int j = 0; j < kHI; ++j) {
            float wj = __ldg(p.w + wo + j);
            if (FP8) wj *= __ldg(p.q_scale + wo + j);
            wreg[j] = wj;
          }
          hc = runs[c].slot >= 0 ? hs + runs[c].slot * kNB1 : p.hist + (int64_t)runs[c].t * kNB1;
        }
        const Run& r = runs[c];
        const int s0 = (r.j0 + it - r.l0) * kBM;
        float ksc = 1.f;
        if (FP8) {
          // this thread's key scale, landed with the tile; keys past the row read a
          // neighbour's scale or the zero fill and are never selected
          const int sl = it % NSCM;
          const int sh = p.seqs.paged() ? 0 : ((r.k0 + s0) & 3);
          ksc = scs[sl * (C::SC_SLOT / 4) + sh + quarter * 32 + lane];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sc_empty[sl]);
        }
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t rr[32];
          tmem_ld32(lane_base + acc * kAccCols + half * kHI + 32 * hh, rr);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            part[jj & 3] = fmaf(wreg[32 * hh + jj], fmaxf(__uint_as_float(rr[jj]), 0.f), part[jj & 3]);
        }
        float v = (part[0] + part[1]) + (part[2] + part[3]);
        if (FP8) v *= ksc;
        tmem_st1(lane_base + kScoreCol + half * kHalfCols + pp, __float_as_uint(v));
        if (r.k < r.n)  // the row selects: count its key
          warp_count(hc, order_key(v) >> 21, s0 + quarter * 32 + lane < r.n);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  // ---- the scores out of tensor memory into the key ring: tile il's key j at
  // sc[il * 128 + j], so a run's keys lie in position order ----
  if (warp >= 2) {
    const int ncol = (mytiles - half + 1) / 2;  // this half's tiles: 2c + half
    for (int cb = 0; cb < ncol; cb += 32) {
      uint32_t rr[32];
      tmem_ld32(lane_base + kScoreCol + half * kHalfCols + cb, rr);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (cb + i < ncol) sc[(2 * (cb + i) + half) * kBM + quarter * 32 + lane] = __uint_as_float(rr[i]);
    }
  }
  // the first and last runs' counts into their rows' histograms, then every counting run
  // of this CTA arrives
  for (int s = 0; s < 2; ++s) {
    const int i = s == 0 ? 0 : ns - 1;
    if (ns == 0 || (s == 1 && ns < 2) || runs[i].k == runs[i].n) continue;
    uint32_t* gh = p.hist + (int64_t)runs[i].t * kNB1;
    for (int j = tid; j < kNB1; j += kThreads) {
      const uint32_t v = hs[s * kNB1 + j];
      if (v) atomicAdd(gh + j, v);
    }
  }
  cta_sync();
  if (tid < ns && runs[tid].k < runs[tid].n) {
    __threadfence();
    atomicAdd(rsync + runs[tid].t * kRowWords, kA);
  }
  const uint32_t lt = (1u << lane) - 1u;

  // ---- first round per run: B* (11 bits), the run's keys above it, and its keys in B*
  // (the candidates), bucketed by the next five key bits, to the row's list at the run's
  // first key position; the run's record: its bucket counts and its keys above B* ----
  for (int i = 0; i < ns; ++i) {
    Run& r = runs[i];
    if (r.k == r.n) continue;  // every key kept: nothing to select
    const int s_lo = r.j0 * kBM, kb = r.l0 * kBM;
    const int nkeys = min((r.l1 - r.l0) * kBM, r.n - s_lo);  // the run's keys in the history
    uint32_t* rc = rsync + r.t * kRowWords;
    if (tid == 0) row_wait(rc, 8, (uint32_t)r.nr, abort_flag, p.status);
    if (tid < kSub) X->bcnt[tid] = X->bcur[tid] = 0u;
    if (tid == 0) X->gt = X->ncand = 0u;
    cta_sync();
    const uint32_t bstar =
        find_digit<true>(p.hist + (int64_t)r.t * kNB1, kNB1, (uint32_t)r.k, X->res, scan_ws).x;
    const uint32_t above = X->res[1];  // (find_digit's answer stays until the next call)
    // one pass over the run's keys (4 a thread at a time): keys above B* counted, keys in
    // B* staged in shared memory
    uint2* stage = reinterpret_cast<uint2*>(spare);
    uint32_t gt_acc = 0;
    for (int j0 = 0; j0 < nkeys; j0 += 4 * kThreads) {
      const int j = j0 + 4 * tid;
      uint32_t kk[4] = {0u, 0u, 0u, 0u};
      if (j < nkeys) {
        const float4 v4 = *reinterpret_cast<const float4*>(sc + kb + j);
        kk[0] = order_key(v4.x);
        kk[1] = order_key(v4.y);
        kk[2] = order_key(v4.z);
        kk[3] = order_key(v4.w);
      }
      uint32_t cm = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = j + e < nkeys;
        gt_acc += ok && (kk[e] >> 21) > bstar;
        if (ok && (kk[e] >> 21) == bstar) cm |= 1u << e;
      }
      // the warp's candidates take consecutive staging slots
      const uint32_t mine = (uint32_t)__popc(cm);
      uint32_t inc = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const uint32_t wtot = __shfl_sync(0xffffffffu, inc, 31);
      uint32_t base = 0;
      if (lane == 0 && wtot) base = atomicAdd(&X->ncand, wtot);
      uint32_t at = __shfl_sync(0xffffffffu, base, 0) + inc - mine;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (cm >> e & 1u) {
          if (at < C::CAND_CAP) stage[at] = make_uint2(kk[e], (uint32_t)(s_lo + j + e));
          ++at;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gt_acc += __shfl_xor_sync(0xffffffffu, gt_acc, o);
    if (lane == 0 && gt_acc) atomicAdd(&X->gt, gt_acc);
    cta_sync();
    const uint32_t nst = X->ncand;
    const bool staged = nst <= C::CAND_CAP;
    // the candidates' bucket counts: from the staged list, else from the keys again
    for (int u0 = 0; u0 < (staged ? (int)nst : nkeys); u0 += kThreads) {
      const int u = u0 + tid;
      bool on;
      uint32_t key;
      if (staged) {
        on = u < (int)nst;
        key = on ? stage[u].x : 0u;
      } else {
        key = u < nkeys ? order_key(sc[kb + u]) : 0u;
        on = u < nkeys && (key >> 21) == bstar;
      }
      warp_count(X->bcnt, (key >> 16) & (kSub - 1), on);
    }
    cta_sync();
    uint32_t* rec = p.rec + ((int64_t)r.t * G + r.rank) * kRec;
    if (tid < kSub) {
      uint32_t o = 0;
      for (int b = 0; b < tid; ++b) o += X->bcnt[b];
      X->boff[tid] = o;
      rec[tid] = X->bcnt[tid];
    }
    if (tid == kSub) rec[kSub] = X->gt;
    if (tid == 0) {
      r.bstar = bstar;
      r.above = above;
      X->ncand = 0u;
    }
    cta_sync();
    // the candidates to the row's list at the run's first key position, bucket by bucket
    uint2* gl = p.cand + (int64_t)r.t * p.cand_ld + s_lo;
    const int64_t room = p.cand_ld - s_lo;
    for (int u0 = 0; u0 < (staged ? (int)nst : nkeys); u0 += kThreads) {
      const int u = u0 + tid;
      bool on;
      uint2 cd;
      if (staged) {
        on = u < (int)nst;
        cd = on ? stage[u] : make_uint2(0u, 0u);
      } else {
        cd = make_uint2(u < nkeys ? order_key(sc[kb + u]) : 0u, (uint32_t)(s_lo + u));
        on = u < nkeys && (cd.x >> 21) == bstar;
      }
      const uint32_t act = __ballot_sync(0xffffffffu, on);
      if (on) {
        // one shared-memory atomic per bucket of the warp, the lanes in order behind it
        const uint32_t b = (cd.x >> 16) & (kSub - 1);
        const uint32_t same = __match_any_sync(act, b);
        const int lead = __ffs(same) - 1;
        uint32_t bb = 0;
        if (lane == lead) bb = X->boff[b] + atomicAdd(&X->bcur[b], (uint32_t)__popc(same));
        bb = __shfl_sync(act, bb, lead);
        const uint32_t at = bb + (uint32_t)__popc(same & lt);
        if ((int64_t)at < room) gl[at] = cd;
      }
    }
    cta_sync();
    if (tid == 0) {
      __threadfence();
      atomicAdd(rc, kB);
    }
  }
  const bool failed = *abort_flag != 0;

  // ---- per run: the exact threshold T from the row's candidates, then every kept key to
  // its slot ----
  for (int i = 0; i < ns; ++i) {
    const Run& r = runs[i];
    const int n = r.n, k = r.k, s_lo = r.j0 * kBM, kb = r.l0 * kBM;
    const int nkeys = min((r.l1 - r.l0) * kBM, n - s_lo);
    int32_t* irow = p.idx + (int64_t)r.t * p.top_k;
    float* vrow = p.vals ? p.vals + (int64_t)r.t * p.top_k : nullptr;
    if (k == n) {
      // every key of the history is kept: position s goes to slot s
      if (!failed)
        for (int j = tid; j < nkeys; j += kThreads) {
          if (!dsa_check(s_lo + j < p.top_k, p.status)) break;
          irow[s_lo + j] = s_lo + j;
          if (vrow) vrow[s_lo + j] = sc[kb + j];
        }
      if (r.j0 == 0)
        for (int j = n + tid; j < p.top_k; j += kThreads) {
          irow[j] = -1;
          if (vrow) vrow[j] = -INFINITY;
        }
      continue;
    }
    if (tid == 0) row_wait(rsync + r.t * kRowWords, 16, (uint32_t)r.nr, abort_flag, p.status);
    cta_sync();
    const uint32_t* rec = p.rec + (int64_t)r.t * G * kRec;
    const uint2* gl = p.cand + (int64_t)r.t * p.cand_ld;
    // The row's runs by rank j: their records give the row's bucket totals and so the
    // 16-bit digit (the bucket d5 holding the k-th key), then where each run's candidates
    // in d5 start (seg_src) and how many candidates of d5 the runs before it have
    // (seg_pref), and the keys above the digit in the runs before this one.
    if (r.nr <= 32) {
      if (warp == 0) {  // one warp: lane j holds run j's record
        uint4 q[kRec / 4];
        if (lane < r.nr) {
          const uint4* rj = reinterpret_cast<const uint4*>(rec + (int64_t)lane * kRec);
#pragma unroll
          for (int u = 0; u < kRec / 4; ++u) q[u] = __ldcg(rj + u);
        }
        const uint32_t* x = reinterpret_cast<const uint32_t*>(q);
        for (int c0 = r.cf, jb = 0; c0 <= r.cl; c0 += 32) {
          const int c = c0 + lane;
          const bool ne = c <= r.cl && tb[c] < tb[c + 1];
          const uint32_t m = __ballot_sync(0xffffffffu, ne);
          if (ne) seg_src[jb + __popc(m & lt)] = (max(r.start, tb[c]) - r.start) * kBM;
          jb += __popc(m);
        }
        if (lane < r.nr)
#pragma unroll
          for (int b = 0; b < kSub; ++b) spare[lane * kSub + b] = x[b];
        __syncwarp();
        uint32_t tot = 0;  // lane b: bucket b of the row
        for (int j = 0; j < r.nr; ++j) tot += spare[j * kSub + lane];
        uint32_t suf = tot;  // buckets >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
          if (lane + o < 32) suf += y;
        }
        const uint32_t need0 = (uint32_t)k - r.above;
        const uint32_t win = __ballot_sync(0xffffffffu, suf - tot < need0 && suf >= need0);
        const int d5 = win ? __ffs(win) - 1 : 0;
        const uint32_t above2 = r.above + __shfl_sync(0xffffffffu, suf - tot, d5);
        const uint32_t nc = __shfl_sync(0xffffffffu, tot, d5);
        uint32_t cj = 0, oj = 0, aj = 0;
        if (lane < r.nr) {
          aj = x[kSub];
#pragma unroll
          for (int b = 0; b < kSub; ++b) {
            if (b < d5) oj += x[b];
            else if (b > d5) aj += x[b];
            else cj = x[b];
          }
        }
        uint32_t inc = cj;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        if (lane < r.nr) {
          seg_pref[lane] = inc - cj;
          seg_src[lane] += (int)oj;
        }
        const uint32_t ab = __reduce_add_sync(0xffffffffu, lane < r.rank ? aj : 0u);
        if (__shfl_sync(0xffffffffu, inc, 31) != nc && lane == 0) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
        if (lane == 0) {
          X->d5 = (uint32_t)d5;
          X->above = above2;
          X->nc = nc;
          X->ab = ab;
          X->gtb = X->eqb = 0u;
        }
      }
    } else {
      {
        const int c = r.cf + tid;
        const bool ne = c <= r.cl && tb[c] < tb[c + 1];
        uint32_t nne;
        const uint32_t j = block_scan(ne ? 1u : 0u, scan_ws, &nne);
        if (ne) seg_src[j] = (max(r.start, tb[c]) - r.start) * kBM;
      }
      uint4 q[kRec / 4];
      if (tid < r.nr) {
        const uint4* rj = reinterpret_cast<const uint4*>(rec + (int64_t)tid * kRec);
#pragma unroll
        for (int u = 0; u < kRec / 4; ++u) q[u] = __ldcg(rj + u);
        const uint32_t* x = reinterpret_cast<const uint32_t*>(q);
#pragma unroll
        for (int b = 0; b < kSub; ++b) spare[tid * kSub + b] = x[b];
      }
      cta_sync();
      if (tid < kSub) {
        uint32_t tot = 0;
        for (int j = 0; j < r.nr; ++j) tot += spare[j * kSub + tid];
        X->bcnt[tid] = tot;
      }
      cta_sync();
      if (tid == 0) {
        const uint32_t need0 = (uint32_t)k - r.above;
        uint32_t run = 0;
        X->d5 = 0u;
        X->above = r.above;
        X->nc = 0u;
        for (int b = kSub - 1; b >= 0; --b) {
          if (run + X->bcnt[b] >= need0) {
            X->d5 = (uint32_t)b;
            X->above = r.above + run;
            X->nc = X->bcnt[b];
            break;
          }
          run += X->bcnt[b];
        }
        X->gtb = X->eqb = 0u;
      }
      cta_sync();
      const uint32_t d5 = X->d5;
      uint32_t cj = 0, ab = 0;
      if (tid < r.nr) {
        const uint32_t* x = reinterpret_cast<const uint32_t*>(q);
        uint32_t oj = 0, aj = x[kSub];
#pragma unroll
        for (int b = 0; b < kSub; ++b) {
          if (b < (int)d5) oj += x[b];
          else if (b > (int)d5) aj += x[b];
          else cj = x[b];
        }
        seg_src[tid] += (int)oj;
        if (tid < r.rank) ab = aj;
      }
      uint32_t ncs, abs_;
      const uint32_t pre = block_scan(cj, scan_ws, &ncs);
      if (tid < r.nr) seg_pref[tid] = pre;
      block_scan(ab, scan_ws, &abs_);
      if (tid == 0) {
        X->ab = abs_;
        if (ncs != X->nc) atomicOr(p.status, DSA_FLAG_BAD_SEQS);
      }
    }
    cta_sync();
    const uint32_t d5 = X->d5, nc = X->nc, above_before = X->ab;
    auto cand_g = [&](uint32_t jj) -> uint2 {  // the jj-th candidate of the bucket, from L2
      int lo = 0, hi = r.nr - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_pref[mid] <= jj) lo = mid; else hi = mid - 1;
      }
      const int64_t at = (int64_t)seg_src[lo] + (jj - seg_pref[lo]);
      return at < p.cand_ld ? __ldcg(gl + at) : make_uint2(0u, 0x7fffffffu);
    };
    uint32_t T, need;
    if (nc <= 128) {
      // few candidates: one warp finds T bit by bit (the largest key with at least `want`
      // candidates at or above it), the ties kept, and the earlier runs' kept candidates
      if (warp == 0) {
        uint32_t ck[4];
        int cp[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t j = (uint32_t)(lane + 32 * u);
          const uint2 cd = j < nc ? cand_g(j) : make_uint2(0u, 0x7fffffffu);
          ck[u] = cd.x;
          cp[u] = (int)cd.y;
        }
        const uint32_t want = (uint32_t)k - X->above;
        const uint32_t hi = (r.bstar << 21) | (d5 << 16);
        uint32_t lo = 0;
        for (int b = 15; b >= 0; --b) {
          const uint32_t trial = hi | lo | (1u << b);
          uint32_t c = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u) c += (lane + 32 * u < (int)nc) && ck[u] >= trial;
          if (__reduce_add_sync(0xffffffffu, c) >= want) lo |= 1u << b;
        }
        const uint32_t t = hi | lo;
        uint32_t ca = 0, cb = 0, ce = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const bool in = lane + 32 * u < (int)nc;
          ca += in && ck[u] > t;
          cb += in && ck[u] > t && cp[u] < s_lo;
          ce += in && ck[u] == t && cp[u] < s_lo;
        }
        ca = __reduce_add_sync(0xffffffffu, ca);
        cb = __reduce_add_sync(0xffffffffu, cb);
        ce = __reduce_add_sync(0xffffffffu, ce);
        if (lane == 0) {
          X->res[0] = t;
          X->res[1] = want - ca;  // keys equal to T that are kept
          X->gtb = cb;
          X->eqb = ce;
        }
      }
      cta_sync();
      T = X->res[0];
      need = X->res[1];
    } else {
      // many candidates (flat scores): radix select over the last 16 bits, 7 + 9
      uint2* stage = reinterpret_cast<uint2*>(spare);
      const bool staged = nc <= C::CAND_CAP;
      if (staged)
        for (uint32_t j = tid; j < nc; j += kThreads) stage[j] = cand_g(j);
      for (int j = tid; j < kNB2; j += kThreads) hr[j] = 0u;
      cta_sync();
      auto cand_at = [&](uint32_t j) -> uint2 { return staged ? stage[j] : cand_g(j); };
      need = (uint32_t)k - X->above;
      for (uint32_t i0 = 0; i0 < nc; i0 += kThreads) {
        const uint32_t j = i0 + tid;
        warp_count(hr, j < nc ? (cand_at(j).x >> 9) & (kNB2 - 1) : 0u, j < nc);
      }
      cta_sync();
      const uint3 d2 = find_digit<false>(hr, kNB2, need, X->res, scan_ws);
      need -= d2.y;
      const uint32_t prefix = (r.bstar << 21) | (d5 << 16) | (d2.x << 9);
      for (int j = tid; j < kNB3; j += kThreads) hr[j] = 0u;
      cta_sync();
      for (uint32_t i0 = 0; i0 < nc; i0 += kThreads) {
        const uint32_t j = i0 + tid;
        const uint32_t key = j < nc ? cand_at(j).x : 0u;
        warp_count(hr, key & (kNB3 - 1), j < nc && (key & 0xfffffe00u) == prefix);
      }
      cta_sync();
      const uint3 d3 = find_digit<false>(hr, kNB3, need, X->res, scan_ws);
      need -= d3.y;
      T = prefix | d3.x;
      uint32_t gtb = 0, eqb = 0;
      for (uint32_t j = tid; j < nc; j += kThreads) {
        const uint2 cd = cand_at(j);
        if ((int)cd.y < s_lo) {
          gtb += cd.x > T;
          eqb += cd.x == T;
        }
      }
      uint32_t sg, se;
      block_scan(gtb, scan_ws, &sg);
      block_scan(eqb, scan_ws, &se);
      if (tid == 0) {
        X->gtb = sg;
        X->eqb = se;
      }
      cta_sync();
    }
    // kept: keys above T, and the first `need` keys equal to T by position.  Each thread
    // takes a contiguous range of the run's keys; one scan gives each range its slots.
    uint32_t bgt = above_before + X->gtb, beq = X->eqb;
    {
      const int per = (((nkeys + kThreads - 1) / kThreads) + 3) & ~3;
      const int e0 = min(nkeys, tid * per), e1 = min(nkeys, e0 + per);
      uint32_t ng = 0, nq = 0;
      for (int j = e0; j < e1; ++j) {
        const uint32_t key = order_key(sc[kb + j]);
        ng += key > T;
        nq += key == T;
      }
      uint32_t tot;
      const uint32_t pre2 = block_scan(ng | (nq << 16), scan_ws, &tot);
      if (!failed) {
        uint32_t gb = bgt + (pre2 & 0xffffu), eb = beq + (pre2 >> 16);
        for (int j = e0; j < e1; ++j) {
          const float v = sc[kb + j];
          const uint32_t key = order_key(v);
          int slot = -1;
          if (key > T) {
            slot = (int)(gb + min(eb, need));
            ++gb;
            dsa_check(slot < k, p.status);  // every key above the threshold has a slot
          } else if (key == T) {
            if (eb < need) slot = (int)(gb + eb);
            ++eb;
          }
          if (slot >= 0 && slot < k) {
            irow[slot] = s_lo + j;
            if (vrow) vrow[slot] = v;
          }
        }
      }
      bgt += tot & 0xffffu;
      beq += tot >> 16;
    }
    if (tid == 0 && r.rank == r.nr - 1 && (bgt + min(beq, need) != (uint32_t)k || beq < need))
      atomicOr(p.status, DSA_FLAG_BAD_SEQS);  // the row's last run: every kept key accounted for
    cta_sync();  // the tables and sums are reused by the next run
  }
  // rows written without scoring: every key kept, no scores requested
  for (uint32_t i = 0; i < nown; ++i) {
    const int2 o = own[i];
    int32_t* irow = p.idx + (int64_t)o.x * p.top_k;
    for (int j = tid; j < p.top_k; j += kThreads) irow[j] = j < o.y ? j : -1;
  }

  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool FP8>
int launch_typed(const IndexerArgs& a, int top_k, int32_t* idx, float* vals, void* scratch,
                 cudaStream_t stream) {
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
  const int G = num_sms();  // always one CTA per SM: the launch counter counts in steps of G
  if (G > kMaxCtas) return set_error(DSA_ERR_UNSUPPORTED, "indexer_topk: %d SMs", G);
  IndexerTopkScratch sc = indexer_topk_scratch(a, scratch);
  Params p{a.seqs, top_k, a.w, a.q_scale, a.k_scale, idx, vals, a.status,
           a.status + kLaunchWord, a.status + kRowSyncWord, sc.hist, sc.rec, sc.cand,
           a.seqs.max_k_len};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: CTAs wait for others
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
  DSA_LAUNCH(FP8 ? "indexer_topk_fp8" : "indexer_topk_bf16", stream,
             e = cudaLaunchKernelEx(&cfg, kern, kmap, qmap, smap, p));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "indexer_topk: %s", cudaGetErrorString(e));
  return check_launch("indexer_topk");
}

}  // namespace

// Exchange buffers: per row its first-round histogram, its runs' records and its candidate
// list (at most every key of the row).
IndexerTopkScratch indexer_topk_scratch(const IndexerArgs& a, void* base) {
  const size_t q = (size_t)a.seqs.total_q;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_hist = take(q * kNB1 * 4);
  const size_t o_rec = take(q * (size_t)num_sms() * kRec * 4);
  const size_t o_cand = take(q * (size_t)a.seqs.max_k_len * 8);
  IndexerTopkScratch s{};
  s.bytes = off;
  if (base) {
    char* b = static_cast<char*>(base);
    s.hist = reinterpret_cast<uint32_t*>(b + o_hist);
    s.rec = reinterpret_cast<uint32_t*>(b + o_rec);
    s.cand = reinterpret_cast<uint2*>(b + o_cand);
  }
  return s;
}

// Decode-shaped problems of up to 128 rows whose tiles fit in the CTAs' tensor memory
// (256 tiles per SM).
bool indexer_topk_eligible(const IndexerArgs& a) {
  const int64_t ntiles = ((int64_t)a.seqs.max_k_len + kBM - 1) / kBM;
  return (a.idx_dtype == DSA_BF16 || a.idx_dtype == DSA_FP8_E4M3) && a.h_idx == kHI &&
         a.d_idx == kDI && a.seqs.total_q <= kMaxRows &&
         (int64_t)a.seqs.total_q * (ntiles + kRowLead) <= (int64_t)num_sms() * kMaxTiles &&
         (a.idx_dtype != DSA_FP8_E4M3 || (reinterpret_cast<uintptr_t>(a.k_scale) & 15) == 0);
}

int launch_indexer_topk(const IndexerArgs& a, int top_k, int32_t* idx, float* vals, void* scratch,
                        cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  return a.idx_dtype == DSA_FP8_E4M3 ? launch_typed<true>(a, top_k, idx, vals, scratch, stream)
                                     : launch_typed<false>(a, top_k, idx, vals, scratch, stream);
}

}  // namespace dsa
