// Sparse Flash Attention over the MLA latent cache on tcgen05 tensor cores,
// for H = 128 query heads, latent d_c = 512 + rope 64 (D = 576), bf16.
//
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
// LLMs", §2.2 and §4.1: the sparse attention core gathers the latent rows at the
// Top-K positions and attends over them chunk by chunk, IO-aware; "Day0 Inference
// Adaptation and Performance Optimization for a New Architecture Domestic LLM on
// Ascend", §4: SFA reads the KV cache at the indexer's position set.)
//
//   S[h, i] = scale · q[t,h,:] · kv[row_i, :]        (all 576 columns)
//   out[t,h,:] = Σ_i softmax_i(S[h,:]) · kv[row_i, 0:512],  lse[t,h] = log Σ_i exp S[h,i]
//
// Why a CTA pair.  All 128 heads share each gathered latent row, so heads are
// the MMA's M = 128.  A single CTA would need the whole query block (128 x 576
// bf16 = 144 KB) and a 128 x 512 fp32 output accumulator, which is all 512 TMEM
// columns with no room for the logits.  So a 2-CTA cluster splits the work:
//  * logits: CTA 0 takes columns 0..287, CTA 1 columns 288..575 (18 K-steps
//    each); each computes a partial S over its columns and sends it to the other
//    through distributed shared memory (in log2 units, as fp16); both CTAs add the
//    same two fp16 partials, so they hold identical logits and take identical
//    softmax decisions;
//  * values: CTA 0 accumulates output columns 0..255, CTA 1 columns 256..511.
// So CTA 0 gathers columns 0..287 of every selected row and CTA 1 columns
// 256..575.  The CTA's 288 query columns live in TMEM (the logit MMA reads its A
// operand from there), which leaves shared memory to a 4-stage ring of gathered
// rows and double send and receive exchange buffers.  TMEM: O (128 x 256 fp32) |
// Q (144 columns of bf16 pairs) | S (128 x 64 fp32) | P (64 bf16 per head) | 8
// columns for passing per-head values between the two softmax groups.
//
// Per chunk of 64 selected rows:
//  * two producer warps (32 rows each): the 16-byte pieces of the CTA's columns
//    go straight into the 128-byte-swizzled operand layout with cp.async;
//    completion arrives on the stage's mbarrier;
//  * MMA thread: S = Q_cols · KV_cols^T (M=128, N=64, K=288; A from TMEM, B
//    K-major in shared memory), then, once P is ready, O += P · V (M=128, N=256,
//    K=64; P from TMEM, V read MN-major straight from the gathered tile);
//  * softmax warps: two groups of four take alternate chunks, so two chunks are in
//    flight (one group waits for its exchange while the other computes); a thread
//    holds one head's 64 columns of its group's chunk.  It reads its partial logits
//    from TMEM (S is then free for the next chunk's MMA), scales them to log2 units,
//    rounds them to fp16 and stages them; each warp ships its 4 KB block to the peer
//    with one bulk copy.  Processing adds the peer's fp16 partials to the thread's own
//    (the same sum in both CTAs), takes the chunk max, moves the running reference
//    (shared by the two groups through TMEM; it moves only when the max grows by more
//    than 2^8, and O is then rescaled) and writes P = 2^(x - m) as bf16 into TMEM,
//    where the P·V MMA reads it as its A operand.
//
// Work schedule.  With many query rows, cluster c takes whole rows c, c + clusters, ...
// With few (decode), the rows' chunk slots (ceil(top_k / 64) per row) are laid end to
// end and cut into one contiguous, equal share per cluster, so every cluster gathers
// the same number of chunks; a row cut by share boundaries is attended in pieces.  Each
// piece but the row's first writes its partial (O, max, sum) and counts itself in; the
// first piece, the last one its cluster attends (the others come first in theirs), waits
// for the others' count, then merges their partials with its own O, still in tensor
// memory, in piece order.
// Every wait is bounded (DSA_FLAG_TIMEOUT).
#include <cuda_fp16.h>

#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kH = 128;        // heads (MMA M)
constexpr int kD = 576;        // latent + rope
constexpr int kDC = 512;       // value columns
constexpr int kNC = 64;        // selected rows per chunk
constexpr int kQK = kD / 2;    // logit columns per CTA
constexpr int kKSteps = kQK / 16;
constexpr int kAtoms = 5;                     // 128-byte column atoms of a gathered row
constexpr int kKVStage = kAtoms * kNC * 128;  // 40 KB
constexpr int kStages = 4;
constexpr int kXBytes = kH * kNC * 2;         // 16 KB: one chunk of the peer's partial logits (fp16)
constexpr int kMaxTopK = 2048;
constexpr int kThreads = 352;                 // producer, MMA, 8 softmax warps, producer
constexpr int kBarBytes = 48 * 8;             // mbarriers and flags
constexpr int kSmem = kStages * kKVStage + 4 * kXBytes + kBarBytes + 1024;
constexpr int kTmemCols = 512;
constexpr int kOCol = 0;                      // O: 256 fp32 columns
constexpr int kQCol = 256;                    // Q: 144 columns (2 bf16 each)
constexpr int kSCol = 400;                    // S: 64 fp32 columns
constexpr int kPCol = 464;                    // P: 32 columns (2 bf16 each)
constexpr int kXCol = 496;                    // 4 columns: the two groups' sums, 2 phases
constexpr int kMCol = 500;                    // 2 columns: the reference decided at a chunk, by parity
constexpr float kRescaleLog2 = 8.0f;          // rescale O only when the max grows > 2^8
static_assert(kMCol + 4 <= kTmemCols, "TMEM layout");
static_assert(kStages * kKVStage >= kH * 256 * 4, "merge staging area");

struct Params {
  Seqs seqs;
  int top_k;
  float scale_log2;  // softmax scale · log2(e)
  int pieces;        // 1: equal contiguous shares of chunk slots; 0: whole rows
  int C;             // chunk slots of a row: max(1, ceil(top_k / 64))
  int64_t tot;       // total_q * C
  int nclusters;     // clusters of the attention grid
  int out_f32;
  const __nv_bfloat16* q;
  const int32_t* idx;
  const __nv_bfloat16* kv;
  void* out;
  float* lse;
  float4* part_o;    // [(total_q + clusters - 1) * 2][64][128] float4 (pieces)
  float* part_ml;    // [(total_q + clusters - 1) * 2][128][2]
  int32_t* lists;    // [gridDim.x][kMaxTopK]: each CTA's compacted cache rows of its unit
  uint32_t* pcount;  // [total_q][2]: pieces of a cut row whose partials are written, by CTA half
  uint32_t* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 64 consecutive TMEM columns of this warp's 32 lanes (one load, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// Two floats to an f16 pair, rounded to nearest and saturated to the largest finite
// magnitude (lo in the low half).
__device__ __forceinline__ uint32_t f16x2_satfinite(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Sequence of packed query row t, by a 32-way search over cu_q (whole warp).
__device__ __forceinline__ int seq_of_row(const Seqs& s, int t, int lane) {
  int lo = 0, hi = s.B;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int probe = lo + lane * step;
    const int v = probe < hi ? __ldg(s.cu_q + probe) : INT_MAX;
    const unsigned bal = __ballot_sync(0xffffffffu, v <= t);
    const int m = 31 - __clz(bal);  // last probe at or below t (probe 0 always is)
    lo = lo + m * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

// A piece of work: chunk slots [a, b) of query row t, i.e. idx[t, 64a : min(64b, top_k)).
struct Piece {
  int t, a, b;
};

// Share of cluster c in the laid-out chunk slots: [B(c), B(c + 1)), B(c) = floor(c·tot/ncl).
__device__ __forceinline__ int64_t share_begin(const Params& p, int c, int ncl) {
  return (int64_t)c * p.tot / ncl;
}
// The cluster whose share holds chunk slot x: the last c with B(c) <= x.
__device__ __forceinline__ int share_of(const Params& p, int64_t x, int ncl) {
  return (int)(((x + 1) * ncl - 1) / p.tot);
}

// The k-th piece of cluster cid's work; false past its end.
__device__ __forceinline__ bool piece_at(const Params& p, int cid, int ncl, int k, Piece& pc) {
  if (!p.pieces) {
    pc.t = cid + k * ncl;
    pc.a = 0;
    pc.b = p.C;
    return pc.t < p.seqs.total_q;
  }
  const int64_t x0 = share_begin(p, cid, ncl), x1 = share_begin(p, cid + 1, ncl);
  const int t = (int)(x0 / p.C) + k;
  const int64_t r0 = (int64_t)t * p.C;
  if (r0 >= x1) return false;
  pc.t = t;
  pc.a = k == 0 ? (int)(x0 - r0) : 0;
  pc.b = (int)min((int64_t)p.C, x1 - r0);
  return true;
}

// The clusters [cf, cf + np) whose shares hold row t's chunk slots (np = 1: not cut).
__device__ __forceinline__ void row_pieces(const Params& p, int t, int ncl, int& cf, int& np) {
  if (!p.pieces) { cf = -1; np = 1; return; }
  cf = share_of(p, (int64_t)t * p.C, ncl);
  np = share_of(p, (int64_t)(t + 1) * p.C - 1, ncl) - cf + 1;
}

// PAGED: key rows through the block table (a separate instantiation, so that the packed
// layout's index compaction stays as short as it is without paging).
template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
sfa_tc_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* kvs = smem;                                                    // [kStages][5][64][128 B]
  uint4* xs = reinterpret_cast<uint4*>(kvs + kStages * kKVStage);         // [2][8][128] x 8 fp16
  uint4* xsend = xs + 2 * (kXBytes / 16);                                  // [2][8][128]: ours, staged
  uint64_t* bars = reinterpret_cast<uint64_t*>(xsend + 2 * (kXBytes / 16));
  int32_t* list = p.lists + (int64_t)blockIdx.x * kMaxTopK;  // global: written and read here
  uint64_t* kv_full = bars;              // [kStages] 64 producer lanes (cp.async completion)
  uint64_t* kv_empty = bars + 4;         // [kStages]
  uint64_t* s_empty = bars + 9;          // the 4 warps of the chunk's group have read S
  uint64_t* q_full = bars + 10;          // 8 softmax warps have stored Q
  uint64_t* p_full = bars + 11;          // the 4 warps of the chunk's group have stored P
  uint64_t* x_full = bars + 14;          // [2] the peer's bulk copies land here (16 KB)
  uint64_t* x_empty = bars + 16;         // [2] the peer's 4 warps of the group: buffer read
  uint64_t* meta_full = bars + 18;
  uint64_t* meta_empty = bars + 19;
  uint64_t* drain = bars + 20;           // MMA drain
  uint64_t* hsync = bars + 24;           // the 8 softmax warps: the two groups' sums exchanged
  volatile int* meta_nv = reinterpret_cast<volatile int*>(bars + 25);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 26);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 27);
  uint64_t* dec = bars + 29;             // [2] by chunk parity: its group published the reference
  // Per chunk parity (a softmax group waits only for its own chunks' phases, so that no
  // parity wait can run ahead of the barrier):
  uint64_t* s_full = bars + 31;          // [2] the chunk's logit MMA is complete
  uint64_t* pv_done = bars + 33;         // [2] the chunk's P·V MMA is complete (P, O free)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int gbase = rank ? 256 : 0;            // first kv column gathered = first output column
  const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&kv_full[i], 64); mbar_init(&kv_empty[i], 1); }
    mbar_init(s_empty, 4);
    mbar_init(q_full, 8);
    mbar_init(p_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&x_full[i], 1); mbar_init(&x_empty[i], 4);
      mbar_init(&dec[i], 4);
      mbar_init(&s_full[i], 1); mbar_init(&pv_done[i], 1);
    }
    mbar_init(meta_full, 1); mbar_init(meta_empty, 10);
    mbar_init(drain, 1);
    mbar_init(hsync, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 10) {
    // -------- producer warps: index compaction (warp 0), gathers (32 rows each) --------
    const int pw = warp == 0 ? 0 : 1;
    int gc = 0;
    bool stop = false;
    Piece pc;
    for (int ui = 0; !stop && piece_at(p, cluster_id, nclusters, ui, pc); ++ui) {
      const int t = pc.t;
      int nv;
      if (pw == 0) {
        const int b = seq_of_row(p.seqs, t, lane);
        int q0 = 0, q1 = 0, k0 = 0, k1 = 0;
        if (lane == 0) {
          q0 = __ldg(p.seqs.cu_q + b); q1 = __ldg(p.seqs.cu_q + b + 1);
          k0 = __ldg(p.seqs.cu_k + b); k1 = __ldg(p.seqs.cu_k + b + 1);
        }
        q0 = __shfl_sync(0xffffffffu, q0, 0); q1 = __shfl_sync(0xffffffffu, q1, 0);
        k0 = __shfl_sync(0xffffffffu, k0, 0); k1 = __shfl_sync(0xffffffffu, k1, 0);
        const int pos = (k1 - k0) - (q1 - q0) + (t - q0);
        const bool ok = t >= q0 && t < q1 && q1 - q0 <= k1 - k0 && k0 >= 0 &&
                        k1 <= p.seqs.total_k && k1 - k0 <= p.seqs.max_k_len;
        // valid entries of the piece's slots of idx[t, :], in slot order -> list (absolute
        // key rows).  Each lane owns a contiguous run of up to 64 slots, loaded all at once
        // (independent loads).  The Top-K kernel that writes idx may still be running: wait
        // for it here, after the work that does not depend on it.  The loads are coherent
        // (L2) ones: idx changes while this grid runs, so the read-only non-coherent path,
        // which may be scheduled or cached as if the data were fixed for the whole launch,
        // must not carry them.
        griddep_wait();
        const int slo = pc.a * kNC, shi = min(pc.b * kNC, p.top_k);
        const int32_t* irow = p.idx + (int64_t)t * p.top_k + slo;
        const int len = max(shi - slo, 0);
        const int seg = (len + 31) / 32;
        const int s0 = lane * seg;
        int v[kMaxTopK / 32];
#pragma unroll
        for (int j = 0; j < kMaxTopK / 32; ++j)
          v[j] = (ok && j < seg && s0 + j < len) ? __ldcg(irow + s0 + j) : -1;
        // valid entries: in [0, pos] (and, paged, on a page inside the cache; those become
        // their cache rows here, the others -1)
        int cnt = 0;
        bool bad = false;
        if (!PAGED) {
#pragma unroll
          for (int j = 0; j < kMaxTopK / 32; ++j) {
            const bool valid = v[j] >= 0 && v[j] <= pos;
            bad |= !valid && v[j] != -1;
            cnt += valid;
          }
        } else {
#pragma unroll
          for (int j = 0; j < kMaxTopK / 32; ++j) {
            const bool in_range = v[j] >= 0 && v[j] <= pos;
            const int row = in_range ? key_row(p.seqs, b, k0, v[j]) : -1;
            const bool valid = row >= 0;
            bad |= !valid && v[j] != -1;
            v[j] = valid ? row : -1;
            cnt += valid;
          }
        }
        if (bad && rank == 0) atomicOr(p.status, DSA_FLAG_BAD_INDEX);
        int before = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, before, o);
          if (lane >= o) before += y;
        }
        nv = __shfl_sync(0xffffffffu, before, 31);
        before -= cnt;
        // the previous unit's list is no longer read by either producer
        if (!__all_sync(0xffffffffu, mbar_wait(meta_empty, (ui & 1) ^ 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT)))
          break;
        if (!PAGED) {
#pragma unroll
          for (int j = 0; j < kMaxTopK / 32; ++j)
            if (v[j] >= 0 && v[j] <= pos) list[before++] = k0 + v[j];
        } else {
#pragma unroll
          for (int j = 0; j < kMaxTopK / 32; ++j)
            if (v[j] >= 0) list[before++] = v[j];
        }
        __syncwarp();
        if (lane == 0) { *meta_nv = nv; mbar_arrive(meta_full); }
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(meta_full, ui & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT)))
          break;
        nv = *meta_nv;
      }
      const int n = nv;
      const int nch = (n + kNC - 1) / kNC;
      // lane = (row sub-index r4 = lane / 8, 16-byte piece lane % 8) for whole atoms;
      // (r8 = lane / 4, piece lane % 4) for CTA 0's half atom (columns 256..287)
      const int r4 = lane >> 3, jp = lane & 7;
      const int r8 = lane >> 2, jh = lane & 3;
      const int natoms = rank ? 5 : 4;
      const int rbase = 32 * pw;
      // this warp's key rows of chunk c (the tail repeats a valid row, masked later): loaded
      // a chunk ahead, so their latency hides behind the previous chunk's copies
      int rowid[8], rowh[4];
      auto load_rows = [&](int c) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const int jj = c * kNC + rbase + g * 4 + r4;
          rowid[g] = list[jj < n ? jj : 0];
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int jj = c * kNC + rbase + g * 8 + r8;
          rowh[g] = list[jj < n ? jj : 0];
        }
      };
      if (nch > 0) load_rows(0);
      for (int c = 0; c < nch; ++c, ++gc) {
        const int st = gc % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&kv_empty[st], ((gc / kStages) & 1) ^ 1,
                                               abort_flag, p.status, DSA_FLAG_TIMEOUT))) {
          stop = true; break;
        }
        int cur[8], curh[4];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          cur[g] = rowid[g];
          if (!dsa_check(cur[g] >= 0 && cur[g] < p.seqs.cache_rows(), p.status)) cur[g] = 0;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          curh[g] = rowh[g];
          if (!dsa_check(curh[g] >= 0 && curh[g] < p.seqs.cache_rows(), p.status)) curh[g] = 0;
        }
        if (c + 1 < nch) load_rows(c + 1);
        const uint32_t dst0 = smem_u32(kvs + st * kKVStage);
        for (int a = 0; a < natoms; ++a) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const int r = rbase + g * 4 + r4;
            const __nv_bfloat16* src = p.kv + (int64_t)cur[g] * kD + gbase + a * 64 + jp * 8;
            cp_async16(dst0 + a * (kNC * 128) + r * 128 + ((jp ^ (r & 7)) * 16), src);
          }
        }
        if (rank == 0) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int r = rbase + g * 8 + r8;
            const __nv_bfloat16* src = p.kv + (int64_t)curh[g] * kD + 256 + jh * 8;
            cp_async16(dst0 + 4 * (kNC * 128) + r * 128 + ((jh ^ (r & 7)) * 16), src);
          }
        }
        cp_async_arrive_noinc(&kv_full[st]);
      }
      __syncwarp();
      if (pw == 1 && lane == 0) mbar_arrive(meta_empty);  // done reading this unit's list
    }
    // every copy issued has landed before the CTA may exit
    cp_async_wait_all();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(kH, kNC);                  // K-major A and B
      const uint32_t idesc_pv = idesc_bf16(kH, 256, false, true);    // V is MN-major
      const uint32_t kv0 = smem_u32(kvs);
      const int koff = rank ? 2 : 0;  // CTA 1's logit columns start half-way into atom 0
      int gc = 0;
      bool stop = false;
      Piece pc;
      for (int ui = 0; !stop && piece_at(p, cluster_id, nclusters, ui, pc); ++ui) {
        if (!mbar_wait(meta_full, ui & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT)) break;
        const int nv = *meta_nv;
        mbar_arrive(meta_empty);
        const int nch = (nv + kNC - 1) / kNC;
        if (!mbar_wait(q_full, ui & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT)) break;
        tc_fence_after();
        if (nch == 0) continue;
        // The softmax warps release S(c) early (they stage it and move on) and hand back P(c)
        // late, so the logit MMA of a chunk may go ahead of the P·V of an earlier one: issue
        // whichever has its inputs ready (bounded polling).
        const int g0 = gc;
        int si = 0, pi = 0;
        uint32_t spins = 0;
        uint64_t t0 = 0;
        while (pi < nch) {
          bool did = false;
          if (si < nch) {
            const int g = g0 + si, st = g % kStages;
            if (mbar_test(smem_u32(&kv_full[st]), (g / kStages) & 1) &&
                mbar_test(smem_u32(s_empty), (g & 1) ^ 1)) {
              fence_proxy_async_smem();  // the cp.async writes, seen by the tensor core
              tc_fence_after();
              // descriptor of the stage's first K-step; later K-steps add their byte offset / 16
              // to its start-address field
              const uint64_t bd0 = sdesc_sw128(kv0 + st * kKVStage, 16, 1024);
#pragma unroll
              for (int i = 0; i < kKSteps; ++i) {
                const int k = i + koff;
                const uint64_t bd = bd0 + (uint64_t)(((k >> 2) * (kNC * 128) + (k & 3) * 32) >> 4);
                mma_bf16_ts(tmem + kSCol, tmem + kQCol + i * 8, bd, idesc_s, i ? 1u : 0u);
              }
              mma_commit(&s_full[g & 1]);
              ++si;
              did = true;
            }
          }
          if (pi < si) {
            const int g = g0 + pi;
            if (mbar_test(smem_u32(p_full), g & 1)) {
              tc_fence_after();
              const uint32_t vb = kv0 + (g % kStages) * kKVStage;
#pragma unroll
              for (int kk = 0; kk < kNC / 16; ++kk) {  // P from TMEM: 16 rows = 8 columns a step
                const uint64_t bd = sdesc_sw128(vb + kk * 2048, kNC * 128, 1024);
                mma_bf16_ts(tmem + kOCol, tmem + kPCol + kk * 8, bd, idesc_pv,
                            (pi > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(&kv_empty[g % kStages]);
              mma_commit(&pv_done[g & 1]);
              ++pi;
              did = true;
            }
          }
          if (did) { spins = 0; continue; }
          if (spins++ == 0) t0 = globaltimer_ns();
          if ((spins & 15u) == 0) {
            if (*abort_flag) { stop = true; break; }
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              *abort_flag = 1;
              atomicOr(p.status, DSA_FLAG_TIMEOUT);
              stop = true;
              break;
            }
          }
        }
        gc = g0 + nch;
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------- softmax / epilogue: two groups of 4 warps take alternate chunks (group g takes
    // the chunks with global index = g mod 2); thread = (head, all 64 columns of a chunk) -------
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;          // warps 2..5: even chunks, 6..9: odd chunks
    const int h = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t xs_peer = mapa(smem_u32(xs), peer);  // our partials go there
    const uint32_t x_full_peer = mapa(smem_u32(x_full), peer);
    const uint32_t x_empty_peer = mapa(smem_u32(x_empty), peer);
    const bool gleader = quarter == 2 && lane == 0;     // first warp of the group (2 or 6)
    int gc = 0, nsync = 0;
    bool stop = false;
    // Stage chunk g (this group's): read the thread's 64 partial logits from TMEM (then S
    // is free for the next logit MMA), scale them to log2 units, round to fp16 and keep
    // them; each warp writes its 4 KB block (32 heads x 64 columns) of the group's send
    // buffer and ships it to the same place in the peer's receive buffer with one bulk
    // copy, which completes on the peer's x_full (16 KB a chunk).  The link between the
    // two SMs moves ~12 B per clock: fp16 halves the time fp32 would take and keeps 2^-11
    // relative precision, below the bf16 rounding P gets anyway; bulk copies (rather than
    // per-thread remote stores, which update the peer's mbarrier every 16 bytes) leave the
    // peer's tensor core undisturbed.
    auto stage = [&](int g, uint32_t (&own)[32]) -> bool {
      const uint32_t xph = (g >> 1) & 1;  // parity of the use count of buffer grp
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[grp], xph, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) return false;
      tc_fence_after();
      {
        uint32_t r[64];
        tmem_ld64(lane_base + kSCol, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);  // S is free for the next chunk's logit MMA
#pragma unroll
        for (int e = 0; e < 32; ++e)
          own[e] = f16x2_satfinite(__uint_as_float(r[2 * e]) * p.scale_log2,
                                   __uint_as_float(r[2 * e + 1]) * p.scale_log2);
      }
      // our x_full will take this chunk's bytes from the peer
      if (gleader) mbar_arrive_expect_tx(&x_full[grp], kXBytes);
      // the peer has read what we sent two chunks ago, so our copy of it is complete
      if (!__all_sync(0xffffffffu, mbar_wait(&x_empty[grp], xph ^ 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) return false;
      uint4* xout = xsend + grp * (kXBytes / 16) + quarter * 256;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        xout[q * 32 + lane] = make_uint4(own[4 * q], own[4 * q + 1], own[4 * q + 2], own[4 * q + 3]);
      fence_proxy_async_smem();  // our generic writes, seen by the bulk copy
      __syncwarp();
      if (lane == 0)
        bulk_s2peer(xs_peer + (uint32_t)(grp * kXBytes + quarter * 4096), xout, 4096,
                    x_full_peer + (uint32_t)(grp * 8));
      return true;
    };
    // combine a per-head value with the other group's: both groups' warps reach the same
    // TMEM lanes, so the value goes through a TMEM column (bounded 8-warp exchange)
    auto exchange = [&](float v) -> float {
      const uint32_t col = lane_base + kXCol + 2 * (nsync & 1);
      tmem_st1(col + grp, __float_as_uint(v));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(hsync);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(hsync, nsync & 1, abort_flag, p.status,
                                                        DSA_FLAG_TIMEOUT));
      ++nsync;
      if (!ok) { stop = true; return 0.f; }
      tc_fence_after();
      return __uint_as_float(tmem_ld1(col + (1 - grp)));
    };
    // the reference max decided at chunk g (by the group that owns it): TMEM column
    // kMCol + (g & 1), published on dec[g & 1]
    auto decided = [&](int g) -> float {
      if (!__all_sync(0xffffffffu, mbar_wait(&dec[g & 1], (g >> 1) & 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) { stop = true; return 0.f; }
      tc_fence_after();
      return __uint_as_float(tmem_ld1(lane_base + kMCol + (g & 1)));
    };
    Piece pc;
    for (int ui = 0; !stop && piece_at(p, cluster_id, nclusters, ui, pc); ++ui) {
      const int t = pc.t;
      int cf, np;
      row_pieces(p, t, nclusters, cf, np);
      // this thread's 72 query columns (144 bf16) -> TMEM, the logit MMA's A operand.
      // The previous piece's logit MMAs are complete: both groups have passed the sum
      // exchange that ends it, after all of its chunks were staged.
      {
        const int tq = dsa_check(t >= 0 && t < p.seqs.total_q, p.status) ? t : 0;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + ((int64_t)tq * kH + h) * kD + (rank ? kQK : 0) + 144 * grp);
        uint4 qv[18];
#pragma unroll
        for (int i = 0; i < 18; ++i) qv[i] = __ldg(src + i);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[4 * i] = qv[i].x; w[4 * i + 1] = qv[i].y; w[4 * i + 2] = qv[i].z; w[4 * i + 3] = qv[i].w;
        }
        tmem_st32(lane_base + kQCol + 72 * grp, w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[4 * i] = qv[8 + i].x; w[4 * i + 1] = qv[8 + i].y;
          w[4 * i + 2] = qv[8 + i].z; w[4 * i + 3] = qv[8 + i].w;
        }
        tmem_st32(lane_base + kQCol + 72 * grp + 32, w);
        const uint32_t w8[8] = {qv[16].x, qv[16].y, qv[16].z, qv[16].w,
                                qv[17].x, qv[17].y, qv[17].z, qv[17].w};
        tmem_st8(lane_base + kQCol + 72 * grp + 64, w8);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(meta_full, ui & 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) break;
      const int nv = *meta_nv;
      __syncwarp();
      if (lane == 0) mbar_arrive(meta_empty);
      const int n = nv;
      const int nch = (n + kNC - 1) / kNC;
      // m_mine: the reference this group's share l of the sum is relative to
      float m_mine = -INFINITY, l = 0.f;
      const int g0 = gc;
      for (int c = (g0 & 1) == grp ? 0 : 1; c < nch; c += 2) {
        const int g = g0 + c;
        uint32_t own[32];  // this chunk's fp16 partials of our CTA (64 columns)
        if (!stage(g, own)) { stop = true; break; }
        const int rows_in = min(kNC, n - c * kNC);
        if (!__all_sync(0xffffffffu, mbar_wait(&x_full[grp], (g >> 1) & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) {
          stop = true; break;
        }
        // logits = our CTA's fp16 partial + the peer's (fp16 + fp16 is the same sum in both
        // CTAs, so both take the same softmax decisions)
        const uint4* oth = xs + grp * (kXBytes / 16) + quarter * 256;
        float s[64];
        float m_c = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 b4 = oth[q * 32 + lane];
          const uint32_t bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&own[4 * q + e]));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&bv[e]));
            const int i = 8 * q + 2 * e;
            s[i] = i < rows_in ? fa.x + fb.x : -INFINITY;
            s[i + 1] = i + 1 < rows_in ? fa.y + fb.y : -INFINITY;
            m_c = fmaxf(m_c, fmaxf(s[i], s[i + 1]));
          }
        }
        __syncwarp();
        // the reads above are done: the peer may refill its send into this buffer
        if (lane == 0) mbar_arrive_remote_relaxed(x_empty_peer + (uint32_t)(grp * 8));
        // running reference, shared by the two groups: it moves only when the max grows by
        // more than 2^8; O (and the other group's share of the sum) follow it lazily
        const float m_prev = c > 0 ? decided(g - 1) : -INFINITY;
        if (stop) break;
        const bool grow = m_c > m_prev + kRescaleLog2;
        const float m_new = grow ? m_c : m_prev;
        tmem_st1(lane_base + kMCol + (g & 1), __float_as_uint(m_new));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dec[grp]);
        if (l > 0.f && m_new > m_mine) l *= ex2(m_mine - m_new);
        m_mine = m_new;
        if (__any_sync(0xffffffffu, grow && c > 0)) {
          // O holds the chunks before g at reference m_prev: rescale it once P·V(g - 1) is in
          if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1,
                                                 abort_flag, p.status, DSA_FLAG_TIMEOUT))) {
            stop = true; break;
          }
          tc_fence_after();
          const float factor = grow ? ex2(m_prev - m_new) : 1.f;
          for (int b = 0; b < 8; ++b) {  // the CTA's 256 output columns of head h
            uint32_t r[32];
            const uint32_t ta = lane_base + kOCol + 32 * b;
            tmem_ld32(ta, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * factor);
            tmem_st32(ta, r);
          }
          tc_fence_before();
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex2(s[2 * i] - m_new), ex2(s[2 * i + 1] - m_new));
          const float2 f2 = __bfloat1622float2(b2);
          l += f2.x + f2.y;
          pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        // P·V(g - 1) has read P (for g = 0 the wait passes: its barrier has no phase yet)
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1,
                                               abort_flag, p.status, DSA_FLAG_TIMEOUT))) {
          stop = true; break;
        }
        tc_fence_after();
        tmem_st32(lane_base + kPCol, pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (stop) break;
      gc = g0 + nch;

      // ---- epilogue of the piece ----
      const bool have = nch > 0;
      float m_ref = -INFINITY;
      if (have) {
        const int gl = gc - 1;  // the piece's last chunk decided the final reference
        m_ref = (gl & 1) == grp ? m_mine : decided(gl);
        if (stop) break;
        if (l > 0.f && m_ref > m_mine) l *= ex2(m_mine - m_ref);
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[gl & 1], (gl >> 1) & 1, abort_flag,
                                               p.status, DSA_FLAG_TIMEOUT))) break;
        tc_fence_after();
      }
      const float lo_sum = exchange(l);  // the other group's share
      if (stop) break;
      const float ltot = grp == 0 ? l + lo_sum : lo_sum + l;  // same order in both groups
      const int half = grp;
      const int ocol = 128 * half;     // this thread's 128 output columns (of the CTA's 256)
      if (np == 1) {
        const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
        uint8_t* orow = static_cast<uint8_t*>(p.out) +
                        (((int64_t)t * kH + h) * kDC + gbase + ocol) * (p.out_f32 ? 4 : 2);
        for (int b = 0; b < 4; ++b) {
          uint32_t r[32];
          if (have) tmem_ld32(lane_base + kOCol + ocol + 32 * b, r);
          else
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          if (p.out_f32) {
            float4* o = reinterpret_cast<float4*>(orow) + 8 * b;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                 __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
          } else {
            uint4* o = reinterpret_cast<uint4*>(orow) + 4 * b;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[8 * i + 2 * e]) * inv,
                                                                __uint_as_float(r[8 * i + 2 * e + 1]) * inv);
                w4[e] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              o[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
        if (rank == 0 && half == 0 && p.lse)
          p.lse[(int64_t)t * kH + h] =
              ltot > 0.f ? (m_ref + log2f(ltot)) * 0.69314718055994531f : -INFINITY;
      } else if (cluster_id != cf) {
        // a piece of a cut row (not its first): its partial (O, m, l), then it counts itself in
        const int64_t slot = (int64_t)(cluster_id + t) * 2 + rank;
        float4* po = p.part_o + slot * (64 * kH);
        for (int b = 0; b < 4; ++b) {
          uint32_t r[32];
          if (have) tmem_ld32(lane_base + kOCol + ocol + 32 * b, r);
          else
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[(32 * half + 8 * b + i) * kH + h] =
                make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
        if (half == 0) {
          p.part_ml[(slot * kH + h) * 2] = m_ref;
          p.part_ml[(slot * kH + h) * 2 + 1] = ltot;
        }
        __syncwarp();
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 softmax warps' writes are done
        if (warp == 2 && lane == 0) {
          __threadfence();
          atomicAdd(p.pcount + 2 * t + rank, 1u);
        }
      } else {
        // the row's first piece: once the others have counted themselves in, out =
        // Σ_j w_j O_j / Σ_j w_j l_j with w_j = 2^(m_j - M), M = max m_j over the pieces with
        // keys, summed in piece order (this piece, the first, from tensor memory)
        if (warp == 2 && lane == 0) {
          uint32_t* pc = p.pcount + 2 * t + rank;
          const uint64_t t0 = globaltimer_ns();
          while (*reinterpret_cast<volatile uint32_t*>(pc) < (uint32_t)(np - 1)) {
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              *abort_flag = 1;
              atomicOr(p.status, DSA_FLAG_TIMEOUT);
              break;
            }
            __nanosleep(32);
          }
          __threadfence();
          *pc = 0u;  // every other piece has counted itself in: reset for the next call
        }
        __syncwarp();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
        float M = ltot > 0.f ? m_ref : -INFINITY;
        for (int j = 1; j < np; ++j) {
          const float2 v = __ldcg(ml + ((int64_t)(cf + j + t) * 2 + rank) * kH + h);
          if (v.y > 0.f) M = fmaxf(M, v.x);
        }
        const float wl = ltot > 0.f ? ex2(m_ref - M) : 0.f;
        float wsum = wl * ltot;
        for (int j = 1; j < np; ++j) {
          const float2 v = __ldcg(ml + ((int64_t)(cf + j + t) * 2 + rank) * kH + h);
          if (v.y > 0.f) wsum = fmaf(ex2(v.x - M), v.y, wsum);
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        uint8_t* orow = static_cast<uint8_t*>(p.out) +
                        (((int64_t)t * kH + h) * kDC + gbase + ocol) * (p.out_f32 ? 4 : 2);
        for (int b = 0; b < 4; ++b) {  // 32 of the thread's 128 columns at a time
          uint32_t r[32];
          if (have) tmem_ld32(lane_base + kOCol + ocol + 32 * b, r);
          else
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = wl * __uint_as_float(r[i]);
          for (int j = 1; j < np; ++j) {
            const int64_t sl = (int64_t)(cf + j + t) * 2 + rank;
            const float2 v = __ldcg(ml + sl * kH + h);
            const float w = v.y > 0.f ? ex2(v.x - M) : 0.f;
            const float4* src = p.part_o + sl * (64 * kH) + (32 * half + 8 * b) * kH + h;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = __ldcg(src + i * kH);
              acc[4 * i] = fmaf(w, x.x, acc[4 * i]);
              acc[4 * i + 1] = fmaf(w, x.y, acc[4 * i + 1]);
              acc[4 * i + 2] = fmaf(w, x.z, acc[4 * i + 2]);
              acc[4 * i + 3] = fmaf(w, x.w, acc[4 * i + 3]);
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] *= inv;
          if (p.out_f32) {
            float4* op = reinterpret_cast<float4*>(orow) + 8 * b;
#pragma unroll
            for (int i = 0; i < 8; ++i) op[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
          } else {
            uint4* op = reinterpret_cast<uint4*>(orow) + 4 * b;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * i + 2 * e], acc[8 * i + 2 * e + 1]);
                w4[e] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              op[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
        if (rank == 0 && half == 0 && p.lse)
          p.lse[(int64_t)t * kH + h] = wsum > 0.f ? (M + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // neither CTA leaves while its peer may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // On the normal path every peer copy into this CTA completed on an x_full phase that a wait
  // above consumed, and every remote arrive precedes the peer's release at the cluster
  // barrier.  After a timeout a consumer may have stopped waiting while a 4 KB copy the peer
  // issued before its own barrier arrival is still landing: such a CTA stays resident for a
  // further 100 us (far longer than a shared-memory copy takes) before it exits.
  if (threadIdx.x == 0 && *abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) __nanosleep(1000);
  }
}

}  // namespace

bool sfa_tc_eligible(const SfaArgs& a) {
  return a.kv_dtype == DSA_BF16 && a.h == kH && a.d_c == kDC && a.d_rope == kD - kDC &&
         a.top_k <= kMaxTopK && (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.kv) & 15) == 0;
}

// Equal contiguous shares of the rows' chunk slots (pieces) when whole rows would load
// the clusters unevenly: fewer than four rows per cluster (and no more rows than the
// status block has piece counts for).
bool sfa_tc_pieces(int total_q) {
  return total_q > 0 && total_q < 2 * num_sms() && total_q <= kPieceRows;
}

// Per-CTA compacted key-row lists (the grid has at most num_sms CTAs), then, with pieces,
// the partial (O, m, l) slots: one per cluster and row it touches, slot = cluster + row <
// total_q + clusters.
size_t sfa_tc_scratch_bytes(int total_q) {
  const size_t lists = align_up((size_t)num_sms() * kMaxTopK * 4, 256);
  if (!sfa_tc_pieces(total_q)) return lists;
  const size_t slots = ((size_t)total_q + num_sms() / 2) * 2;
  return lists + align_up(slots * kH * 256 * 4, 256) + align_up(slots * kH * 2 * 4, 256);
}

int launch_sfa_tc(const SfaArgs& a, void* scratch, cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  const bool pieces = sfa_tc_pieces(a.seqs.total_q);
  Params p{};
  p.seqs = a.seqs;
  p.top_k = a.top_k;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.pieces = pieces ? 1 : 0;
  p.C = a.top_k > kNC ? (a.top_k + kNC - 1) / kNC : 1;
  p.tot = (int64_t)a.seqs.total_q * p.C;
  p.out_f32 = a.out_dtype == DSA_F32;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.idx = a.idx;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.out = a.out;
  p.lse = a.lse;
  p.status = a.status;
  p.pcount = a.status + kPieceWord;
  char* b = static_cast<char*>(scratch);
  p.lists = reinterpret_cast<int32_t*>(b);
  b += align_up((size_t)num_sms() * kMaxTopK * 4, 256);
  if (pieces) {
    const size_t slots = ((size_t)a.seqs.total_q + num_sms() / 2) * 2;
    p.part_o = reinterpret_cast<float4*>(b);
    b += align_up(slots * kH * 256 * 4, 256);
    p.part_ml = reinterpret_cast<float*>(b);
  }
  auto kern = a.seqs.paged() ? sfa_tc_kernel<true> : sfa_tc_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess)
    return check_launch("sfa_tc: smem attribute");
  const int64_t units = pieces ? p.tot : (int64_t)a.seqs.total_q;
  const int max_clusters = num_sms() / 2;
  int clusters = (int)(units < max_clusters ? units : max_clusters);
  // two clusters a row when that fits: shares end on half rows (two pieces a row), which
  // beats a few more clusters whose shares cut rows into three or four pieces
  if (pieces && 2 * a.seqs.total_q <= max_clusters && p.C % 2 == 0) clusters = 2 * a.seqs.total_q;
  p.nclusters = clusters;
  cudaError_t e = cudaSuccess;
  DSA_LAUNCH("sfa_tc", stream,
             e = launch_pdl(kern, dim3(2 * clusters), dim3(kThreads), kSmem, stream, p));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "sfa_tc: %s", cudaGetErrorString(e));
  return check_launch("sfa_tc");
}

}  // namespace dsa
