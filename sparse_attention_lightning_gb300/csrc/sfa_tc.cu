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
// columns for swapping per-head values between the two halves.
//
// Per chunk of 64 selected rows:
//  * two producer warps (32 rows each): the 16-byte pieces of the CTA's columns
//    go straight into the 128-byte-swizzled operand layout with cp.async;
//    completion arrives on the stage's mbarrier;
//  * MMA thread: S = Q_cols · KV_cols^T (M=128, N=64, K=288; A from TMEM, B
//    K-major in shared memory), then, once P is ready, O += P · V (M=128, N=256,
//    K=64; P from TMEM, V read MN-major straight from the gathered tile);
//  * softmax warps (two warpgroups; a thread per head and half of the chunk's
//    columns): read their 32 partial logits from TMEM (S is then free for the next
//    chunk's MMA), scale them to log2 units, round to fp16 and stage them; the last
//    warp to stage ships the CTA's 16 KB to the peer with one bulk copy.  A chunk is
//    staged before the previous one is processed whenever its logits are ready, so
//    the exchange overlaps the softmax.  Processing adds the peer's fp16 partials to
//    the thread's own (the same sum in both CTAs), takes the chunk max (the two halves
//    of a head swap theirs through TMEM), keeps a running max (O is rescaled only when
//    it grows by more than 2^8) and writes its half of P = 2^(x - m) as bf16 into
//    TMEM, where the P·V MMA reads it as its A operand.
//
// Decode rows are split over 2 clusters when there are few queries; the second
// cluster of a row to finish merges the other's partial (O, max, sum) into its own.
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
constexpr int kXCol = 496;                    // 4 columns: the two halves' sums, 2 phases
constexpr int kMCol = 500;                    // 4 columns: the two halves' chunk maxima, 2 phases
constexpr float kRescaleLog2 = 8.0f;          // rescale O only when the max grows > 2^8
static_assert(kMCol + 4 <= kTmemCols, "TMEM layout");
static_assert(kStages * kKVStage + 2 * kXBytes >= kH * 256 * 4, "merge staging area");

struct Params {
  Seqs seqs;
  int top_k;
  float scale_log2;  // softmax scale · log2(e)
  int nsplit;
  int out_f32;
  const __nv_bfloat16* q;
  const int32_t* idx;
  const __nv_bfloat16* kv;
  void* out;
  float* lse;
  float4* part_o;    // [total_q * nsplit * 2][64][128] float4 (nsplit > 1)
  float* part_ml;    // [total_q * nsplit * 2][128][2]
  int* counters;     // [total_q * 2], zero at launch
  int32_t* lists;    // [gridDim.x][kMaxTopK]: each CTA's compacted key rows of its unit
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

// The split `sp` of a row with nv selected keys: rows [lo, lo + n) of its list.
__device__ __forceinline__ void unit_range(int nv, int sp, int nsplit, int& lo, int& n) {
  lo = (int)((int64_t)nv * sp / nsplit);
  n = (int)((int64_t)nv * (sp + 1) / nsplit) - lo;
}

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
  uint64_t* s_full = bars + 8;
  uint64_t* s_empty = bars + 9;          // 8 softmax warps have read S
  uint64_t* q_full = bars + 10;          // 8 softmax warps have stored Q
  uint64_t* p_full = bars + 11;
  uint64_t* p_empty = bars + 12;
  uint64_t* pv_done = bars + 13;
  uint64_t* x_full = bars + 14;          // [2] the peer's st.async bytes land here
  uint64_t* x_empty = bars + 16;         // [2] the peer's 8 softmax warps: buffer read
  uint64_t* meta_full = bars + 18;
  uint64_t* meta_empty = bars + 19;
  uint64_t* drain = bars + 20;           // [2]: MMA drain, merge copy
  uint64_t* sync_a = bars + 22;          // 256 softmax threads: partials written
  uint64_t* sync_b = bars + 23;          // the arrival count has been taken
  uint64_t* hsync = bars + 24;           // the 8 softmax warps: per-head halves exchanged
  volatile int* meta_nv = reinterpret_cast<volatile int*>(bars + 25);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 26);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 27);
  int* s_last = reinterpret_cast<int*>(bars + 28);
  uint64_t* pairb = bars + 29;           // [4] the two softmax warps of a lane quarter
  uint32_t* x_count = reinterpret_cast<uint32_t*>(bars + 33);  // [2] staging arrivals, ever

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int gbase = rank ? 256 : 0;            // first kv column gathered = first output column
  const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int nunits = p.seqs.total_q * p.nsplit;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&kv_full[i], 64); mbar_init(&kv_empty[i], 1); }
    mbar_init(s_full, 1); mbar_init(s_empty, 8);
    mbar_init(q_full, 8);
    mbar_init(p_full, 8); mbar_init(p_empty, 1); mbar_init(pv_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&x_full[i], 1); mbar_init(&x_empty[i], 8);
      x_count[i] = 0;
    }
    for (int i = 0; i < 4; ++i) mbar_init(&pairb[i], 2);
    mbar_init(meta_full, 1); mbar_init(meta_empty, 10);
    mbar_init(drain, 1);
    mbar_init(drain + 1, 1);
    mbar_init(sync_a, 256);
    mbar_init(sync_b, 1);
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
    for (int u = cluster_id, ui = 0; u < nunits && !stop; u += nclusters, ++ui) {
      const int t = u / p.nsplit, sp = u - t * p.nsplit;
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
        // valid entries of idx[t, :] in slot order -> list (absolute key rows).  Each lane
        // owns a contiguous run of up to 64 slots, loaded all at once (independent loads).
        // The Top-K kernel that writes idx may still be running: wait for it here, after
        // the work that does not depend on it.
        griddep_wait();
        const int32_t* irow = p.idx + (int64_t)t * p.top_k;
        const int seg = (p.top_k + 31) / 32;
        const int s0 = lane * seg;
        int v[kMaxTopK / 32];
#pragma unroll
        for (int j = 0; j < kMaxTopK / 32; ++j)
          v[j] = (ok && j < seg && s0 + j < p.top_k) ? __ldg(irow + s0 + j) : -1;
        int cnt = 0;
        bool bad = false;
#pragma unroll
        for (int j = 0; j < kMaxTopK / 32; ++j) {
          const bool valid = v[j] >= 0 && v[j] <= pos;
          bad |= !valid && v[j] != -1;
          cnt += valid;
        }
        if (bad && sp == 0 && rank == 0) atomicOr(p.status, DSA_FLAG_BAD_INDEX);
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
#pragma unroll
        for (int j = 0; j < kMaxTopK / 32; ++j)
          if (v[j] >= 0 && v[j] <= pos) list[before++] = k0 + v[j];
        __syncwarp();
        if (lane == 0) { *meta_nv = nv; mbar_arrive(meta_full); }
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(meta_full, ui & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT)))
          break;
        nv = *meta_nv;
      }
      int lo, n;
      unit_range(nv, sp, p.nsplit, lo, n);
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
          rowid[g] = list[lo + (jj < n ? jj : 0)];
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int jj = c * kNC + rbase + g * 8 + r8;
          rowh[g] = list[lo + (jj < n ? jj : 0)];
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
        for (int g = 0; g < 8; ++g) cur[g] = rowid[g];
#pragma unroll
        for (int g = 0; g < 4; ++g) curh[g] = rowh[g];
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
      for (int u = cluster_id, ui = 0; u < nunits && !stop; u += nclusters, ++ui) {
        if (!mbar_wait(meta_full, ui & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT)) break;
        const int nv = *meta_nv;
        mbar_arrive(meta_empty);
        const int sp = u % p.nsplit;
        int lo, n;
        unit_range(nv, sp, p.nsplit, lo, n);
        const int nch = (n + kNC - 1) / kNC;
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
              mma_commit(s_full);
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
              mma_commit(p_empty);
              mma_commit(pv_done);
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
    // ---------------- softmax / epilogue: 2 warpgroups; thread = (head, half of the chunk) ----
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;        // warps 2..5: columns 0..31, warps 6..9: 32..63
    const int h = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t xs_peer = mapa(smem_u32(xs), peer);  // our partial goes there
    const uint32_t x_full_peer = mapa(smem_u32(x_full), peer);
    const uint32_t x_empty_peer = mapa(smem_u32(x_empty), peer);
    const bool leader = threadIdx.x == 64;
    int gc = 0, nsync = 0;
    bool stop = false;
    // Stage chunk g: read this thread's 32 partial logits from TMEM (then S is free for
    // the next logit MMA), scale them to log2 units, round to fp16 and write them to the
    // staging buffer ([8][128] x 8 halves: both halves of every head).  The last of the 8
    // warps to stage ships the 16 KB to the peer with one bulk copy that completes on the
    // peer's x_full.  The link between the two SMs moves ~12 B per clock: fp16 halves the
    // time fp32 would take and keeps 2^-11 relative precision, below the bf16 rounding P
    // gets anyway; one bulk copy (rather than per-thread remote stores, which update the
    // peer's mbarrier every 16 bytes) leaves the peer's tensor core undisturbed.
    auto stage = [&](int g, uint32_t (&own)[16]) -> bool {
      const int xb = g & 1;
      const uint32_t xph = (g >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, g & 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) return false;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(lane_base + kSCol + 32 * half, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      // our x_full will take this chunk's bytes from the peer
      if (leader) mbar_arrive_expect_tx(&x_full[xb], kXBytes);
      // the peer has read what we sent two chunks ago, so our copy of it is complete
      if (!__all_sync(0xffffffffu, mbar_wait(&x_empty[xb], xph ^ 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) return false;
      uint4* xout = xsend + xb * (kXBytes / 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(r[8 * q + 2 * e]) * p.scale_log2;
          const float b = __uint_as_float(r[8 * q + 2 * e + 1]) * p.scale_log2;
          const __half2 h2 = __floats2half2_rn(fminf(fmaxf(a, -65504.f), 65504.f),
                                               fminf(fmaxf(b, -65504.f), 65504.f));
          w[e] = *reinterpret_cast<const uint32_t*>(&h2);
          own[4 * q + e] = w[e];
        }
        xout[(4 * half + q) * kH + h] = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();  // our generic writes, seen by the bulk copy
      __syncwarp();
      if (lane == 0) {
        uint32_t before;
        asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                     : "=r"(before) : "r"(smem_u32(&x_count[xb])) : "memory");
        if ((before & 7u) == 7u)
          bulk_s2peer(xs_peer + (uint32_t)(xb * kXBytes), xout, kXBytes,
                      x_full_peer + (uint32_t)(xb * 8));
      }
      return true;
    };
    // the other half's chunk maximum of head h (the warp pair of this lane quarter)
    auto pair_max = [&](float v, int g) -> float {
      const uint32_t col = lane_base + kMCol + 2 * (g & 1);
      tmem_st1(col + half, __float_as_uint(v));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pairb[quarter]);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&pairb[quarter], g & 1, abort_flag,
                                                        p.status, DSA_FLAG_TIMEOUT));
      if (!ok) { stop = true; return v; }
      tc_fence_after();
      return fmaxf(v, __uint_as_float(tmem_ld1(col + (1 - half))));
    };
    // combine a per-head value with the other half's: both halves' warps reach the same
    // TMEM lanes, so the value goes through a TMEM column (bounded 8-warp exchange)
    auto exchange = [&](float v) -> float {
      const uint32_t col = lane_base + kXCol + 2 * (nsync & 1);
      tmem_st1(col + half, __float_as_uint(v));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(hsync);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(hsync, nsync & 1, abort_flag, p.status,
                                                        DSA_FLAG_TIMEOUT));
      ++nsync;
      if (!ok) { stop = true; return 0.f; }
      tc_fence_after();
      return __uint_as_float(tmem_ld1(col + (1 - half)));
    };
    for (int u = cluster_id, ui = 0; u < nunits && !stop; u += nclusters, ++ui) {
      const int t = u / p.nsplit, sp = u - t * p.nsplit;
      // this thread's 72 query columns (144 bf16) -> TMEM, the logit MMA's A operand.
      // The previous unit's logit MMAs are complete: this thread has read all their S.
      {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + ((int64_t)t * kH + h) * kD + (rank ? kQK : 0) + 144 * half);
        uint4 qv[18];
#pragma unroll
        for (int i = 0; i < 18; ++i) qv[i] = __ldg(src + i);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[4 * i] = qv[i].x; w[4 * i + 1] = qv[i].y; w[4 * i + 2] = qv[i].z; w[4 * i + 3] = qv[i].w;
        }
        tmem_st32(lane_base + kQCol + 72 * half, w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[4 * i] = qv[8 + i].x; w[4 * i + 1] = qv[8 + i].y;
          w[4 * i + 2] = qv[8 + i].z; w[4 * i + 3] = qv[8 + i].w;
        }
        tmem_st32(lane_base + kQCol + 72 * half + 32, w);
        const uint32_t w8[8] = {qv[16].x, qv[16].y, qv[16].z, qv[16].w,
                                qv[17].x, qv[17].y, qv[17].z, qv[17].w};
        tmem_st8(lane_base + kQCol + 72 * half + 64, w8);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(meta_full, ui & 1, abort_flag, p.status,
                                             DSA_FLAG_TIMEOUT))) break;
      const int nv = *meta_nv;
      __syncwarp();
      if (lane == 0) mbar_arrive(meta_empty);
      int lo, n;
      unit_range(nv, sp, p.nsplit, lo, n);
      const int nch = (n + kNC - 1) / kNC;
      float m_ref = -INFINITY, l = 0.f;  // l: this half's share of the sum
      const int g0 = gc;
      uint32_t cur[16], nxt[16];  // this thread's staged fp16 partials (32 columns)
      if (nch > 0 && !stage(g0, cur)) break;
      for (int c = 0; c < nch; ++c, ++gc) {
        // stage the next chunk first when its logits are already there, so its exchange is
        // in flight while this one is processed; otherwise process this one first
        bool early = false;
        if (c + 1 < nch) {
          early = __all_sync(0xffffffffu, mbar_test(smem_u32(s_full), (gc + 1) & 1));
          if (early && !stage(gc + 1, nxt)) { stop = true; break; }
        }
        const int rows_in = min(kNC, n - c * kNC);
        const int xb = gc & 1;               // exchange buffer
        const uint32_t xph = (gc >> 1) & 1;  // parity of its use count
        if (!__all_sync(0xffffffffu, mbar_wait(&x_full[xb], xph, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) {
          stop = true; break;
        }
        // logits of this thread's 32 columns = its CTA's fp16 partial + the peer's (fp16 + fp16
        // is the same sum in both CTAs, so both take the same softmax decisions)
        const uint4* oth = xs + xb * (kXBytes / 16);
        float s[32];
        float m_c = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 b4 = oth[(4 * half + q) * kH + h];
          const uint32_t bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&cur[4 * q + e]));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&bv[e]));
            const int i = 8 * q + 2 * e;
            s[i] = 32 * half + i < rows_in ? fa.x + fb.x : -INFINITY;
            s[i + 1] = 32 * half + i + 1 < rows_in ? fa.y + fb.y : -INFINITY;
            m_c = fmaxf(m_c, fmaxf(s[i], s[i + 1]));
          }
        }
        __syncwarp();
        // the reads above fed m_c: the peer may refill the buffer
        if (lane == 0) mbar_arrive_remote_relaxed(x_empty_peer + (uint32_t)(xb * 8));
        m_c = pair_max(m_c, gc);  // the same chunk maximum in both halves
        if (stop) break;
        // running max: move the reference only when it grows by more than 2^8
        const bool grow = m_c > m_ref + kRescaleLog2;
        const float m_new = grow ? m_c : m_ref;
        const float factor = grow ? ex2(m_ref - m_new) : 1.f;
        l *= factor;
        if (__any_sync(0xffffffffu, grow && c > 0)) {
          if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (gc - 1) & 1, abort_flag, p.status,
                                                 DSA_FLAG_TIMEOUT))) { stop = true; break; }
          tc_fence_after();
          for (int b = 0; b < 4; ++b) {  // this half's 128 output columns
            uint32_t r[32];
            const uint32_t ta = lane_base + kOCol + 128 * half + 32 * b;
            tmem_ld32(ta, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * factor);
            tmem_st32(ta, r);
          }
          tc_fence_before();
        }
        m_ref = m_new;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = s[2 * i];
          const float x1 = s[2 * i + 1];
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex2(x0 - m_ref), ex2(x1 - m_ref));
          const float2 f2 = __bfloat1622float2(b2);
          l += f2.x + f2.y;
          pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(p_empty, (gc & 1) ^ 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) { stop = true; break; }
        tc_fence_after();
        tmem_st16(lane_base + kPCol + 16 * half, pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        if (c + 1 < nch && !early && !stage(gc + 1, nxt)) { stop = true; break; }
#pragma unroll
        for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
      }
      if (stop) break;

      // ---- epilogue of the unit ----
      const bool have = nch > 0;
      if (have) {
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (gc - 1) & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) break;
        tc_fence_after();
      }
      const float lo_sum = exchange(l);  // the other half's share
      if (stop) break;
      const float ltot = half == 0 ? l + lo_sum : lo_sum + l;  // same order in both halves
      const int ocol = 128 * half;     // this thread's 128 output columns (of the CTA's 256)
      if (p.nsplit == 1) {
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
      } else {
        // split of a row: publish (O, m, l); the second split of the row to finish merges
        const int64_t slot = ((int64_t)t * p.nsplit + sp) * 2 + rank;
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
        // all 256 partial rows are out before the arrival count moves (bounded waits)
        __threadfence();
        mbar_arrive(sync_a);
        if (leader) {
          const bool okw = mbar_wait(sync_a, ui & 1, abort_flag, p.status, DSA_FLAG_TIMEOUT);
          *s_last = okw && atomicAdd(p.counters + t * 2 + rank, 1) == p.nsplit - 1;
          mbar_arrive(sync_b);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(sync_b, ui & 1, abort_flag, p.status,
                                               DSA_FLAG_TIMEOUT))) break;
        if (*s_last) {
          // The other split's (O, m, l) of this column half: one bulk copy of its
          // 128 KB into the (now idle) query/KV area, then each thread merges.
          __threadfence();
          const int64_t other = ((int64_t)t * p.nsplit + (1 - sp)) * 2 + rank;
          float4* po2 = reinterpret_cast<float4*>(kvs);  // idle ring + exchange area
          if (leader) {
            fence_proxy_async_all();
            mbar_arrive_expect_tx(drain + 1, kH * 256 * 4);
            for (int c = 0; c < 8; ++c)
              bulk_load(po2 + c * 1024, p.part_o + other * (64 * kH) + c * 1024, 16384, drain + 1);
          }
          // merged in split order (split 0 first), whichever split runs the merge, so the
          // result does not depend on which one finished last
          const float mo = __ldcg(p.part_ml + (other * kH + h) * 2);
          const float lo2 = __ldcg(p.part_ml + (other * kH + h) * 2 + 1);
          const bool first = sp == 0;
          const float m0 = first ? m_ref : mo, l0 = first ? ltot : lo2;
          const float m1 = first ? mo : m_ref, l1 = first ? lo2 : ltot;
          const float M = fmaxf(m0, m1);
          const float w0 = l0 > 0.f ? ex2(m0 - M) : 0.f;
          const float w1 = l1 > 0.f ? ex2(m1 - M) : 0.f;
          const float wsum = w0 * l0 + w1 * l1;
          const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
          if (!__all_sync(0xffffffffu, mbar_wait(drain + 1, 0, abort_flag, p.status,
                                                 DSA_FLAG_TIMEOUT))) break;
          uint8_t* orow = static_cast<uint8_t*>(p.out) +
                          (((int64_t)t * kH + h) * kDC + gbase + ocol) * (p.out_f32 ? 4 : 2);
          for (int b = 0; b < 4; ++b) {
            uint32_t r[32];
            if (have) tmem_ld32(lane_base + kOCol + ocol + 32 * b, r);
            else
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = 0u;
            float o[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = po2[(32 * half + 8 * b + i) * kH + h];
              const float xo[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float own = __uint_as_float(r[4 * i + e]);
                const float a0 = first ? own : xo[e], a1 = first ? xo[e] : own;
                o[4 * i + e] = (w0 * a0 + w1 * a1) * inv;
              }
            }
            if (p.out_f32) {
              float4* op = reinterpret_cast<float4*>(orow) + 8 * b;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                op[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            } else {
              uint4* op = reinterpret_cast<uint4*>(orow) + 4 * b;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * i + 2 * e], o[8 * i + 2 * e + 1]);
                  w4[e] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                op[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            }
          }
          if (rank == 0 && half == 0 && p.lse)
            p.lse[(int64_t)t * kH + h] = wsum > 0.f ? (M + log2f(wsum)) * 0.69314718055994531f
                                                    : -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // neither CTA leaves while its peer may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool sfa_tc_eligible(const SfaArgs& a) {
  return a.kv_dtype == DSA_BF16 && a.h == kH && a.d_c == kDC && a.d_rope == kD - kDC &&
         a.top_k <= kMaxTopK && (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.kv) & 15) == 0;
}

// Split each row over 2 clusters when that still leaves every cluster one unit.  With a
// split, units = 2 * total_q <= num_sms / 2 = clusters, so a cluster never runs a second
// unit: the merge may stage the partner's partial in the idle ring and exchange buffers.
int sfa_tc_nsplit(int total_q) { return total_q > 0 && num_sms() >= 4 * total_q ? 2 : 1; }

// Per-CTA compacted key-row lists (the grid has at most num_sms CTAs), then, with a
// split, the partial (O, m, l) slots and the per-row arrival counters.
size_t sfa_tc_scratch_bytes(int total_q) {
  const size_t lists = align_up((size_t)num_sms() * kMaxTopK * 4, 256);
  const int ns = sfa_tc_nsplit(total_q);
  if (ns == 1) return lists;
  const size_t slots = (size_t)total_q * ns * 2;
  return lists + align_up(slots * kH * 256 * 4, 256) + align_up(slots * kH * 2 * 4, 256) +
         align_up((size_t)total_q * 2 * 4, 256);
}

int sfa_tc_clear_counters(const SfaArgs& a, void* scratch, cudaStream_t stream) {
  const int ns = sfa_tc_nsplit(a.seqs.total_q);
  if (ns == 1 || a.seqs.total_q == 0) return DSA_OK;
  const size_t slots = (size_t)a.seqs.total_q * ns * 2;
  char* b = static_cast<char*>(scratch) + align_up((size_t)num_sms() * kMaxTopK * 4, 256) +
            align_up(slots * kH * 256 * 4, 256) + align_up(slots * kH * 2 * 4, 256);
  cudaError_t e = cudaMemsetAsync(b, 0, (size_t)a.seqs.total_q * 2 * 4, stream);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "sfa_tc: %s", cudaGetErrorString(e));
  return DSA_OK;
}

int launch_sfa_tc(const SfaArgs& a, void* scratch, cudaStream_t stream, bool counters_zeroed) {
  if (a.seqs.total_q == 0) return DSA_OK;
  const int ns = sfa_tc_nsplit(a.seqs.total_q);
  Params p{};
  p.seqs = a.seqs;
  p.top_k = a.top_k;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.nsplit = ns;
  p.out_f32 = a.out_dtype == DSA_F32;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.idx = a.idx;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.out = a.out;
  p.lse = a.lse;
  p.status = a.status;
  char* b = static_cast<char*>(scratch);
  p.lists = reinterpret_cast<int32_t*>(b);
  b += align_up((size_t)num_sms() * kMaxTopK * 4, 256);
  if (ns > 1) {
    const size_t slots = (size_t)a.seqs.total_q * ns * 2;
    p.part_o = reinterpret_cast<float4*>(b);
    b += align_up(slots * kH * 256 * 4, 256);
    p.part_ml = reinterpret_cast<float*>(b);
    b += align_up(slots * kH * 2 * 4, 256);
    p.counters = reinterpret_cast<int*>(b);
    if (!counters_zeroed) {
      const int rc = sfa_tc_clear_counters(a, scratch, stream);
      if (rc != DSA_OK) return rc;
    }
  }
  if (cudaFuncSetAttribute(sfa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess)
    return check_launch("sfa_tc: smem attribute");
  const int64_t units = (int64_t)a.seqs.total_q * ns;
  const int max_clusters = num_sms() / 2;
  const int clusters = (int)(units < max_clusters ? units : max_clusters);
  cudaError_t e = cudaSuccess;
  DSA_LAUNCH("sfa_tc", stream,
             e = launch_pdl(sfa_tc_kernel, dim3(2 * clusters), dim3(kThreads), kSmem, stream, p));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "sfa_tc: %s", cudaGetErrorString(e));
  return check_launch("sfa_tc");
}

}  // namespace dsa
