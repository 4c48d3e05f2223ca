// Internal declarations shared by the translation units of libdsa.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dsa.h"

namespace dsa {

// ----------------------------------------------------------------------------
// Workspace layout: [0, 16384) status block (word 0: status flags; word kLaunchWord: the
// fused decode indexer's launch count; from word kRowSyncWord: its per-row counters, two
// sets of 128 rows x 8 words; from word kPieceWord: the sparse attention's piece counts);
// scratch regions follow, 256-aligned.
constexpr size_t kStatusBytes = 16384;
constexpr int kLaunchWord = 32;
constexpr int kRowSyncWord = 256;
// from word kPieceWord: the sparse attention's per-(row, CTA half) counts of the pieces of
// a cut row whose partials are written (reset by the piece that merges them)
constexpr int kPieceWord = kRowSyncWord + 2 * 128 * 8;
constexpr int kPieceRows = (int)(kStatusBytes / 4 - kPieceWord) / 2;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Sequence layout as the kernels see it.
struct Seqs {
  const int32_t* cu_q;
  const int32_t* cu_k;
  int B;
  int total_q;
  int total_k;
  int max_k_len;
  // Paged caches (page_size > 0): key position s of sequence b is the cache row
  // block_table[b * max_pages + s / page_size] * page_size + s % page_size.  Otherwise
  // the keys of sequence b are the rows cu_k[b] .. cu_k[b+1]-1.
  const int32_t* block_table = nullptr;
  int page_size = 0, max_pages = 0, num_pages = 0;
  __host__ __device__ bool paged() const { return page_size > 0; }
  // rows of the key caches (k_idx, kv, k_scale)
  __host__ __device__ int64_t cache_rows() const {
    return paged() ? (int64_t)num_pages * page_size : (int64_t)total_k;
  }
};

struct RowInfo {
  int b;      // sequence
  int pos;    // position of the query in its sequence
  int k0;     // first packed key row of the sequence
  int L;      // keys in the sequence
};

// Packed query row t -> (sequence, position).  Returns false (and flags the
// status word) when cu_q/cu_k are inconsistent with the descriptor.
__device__ __forceinline__ bool query_row_info(const Seqs& s, int t, RowInfo& r,
                                               uint32_t* status) {
  int lo = 0, hi = s.B - 1;
  while (lo < hi) {  // last b with cu_q[b] <= t
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(s.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q0 = __ldg(s.cu_q + b), q1 = __ldg(s.cu_q + b + 1);
  const int k0 = __ldg(s.cu_k + b), k1 = __ldg(s.cu_k + b + 1);
  const int T = q1 - q0, L = k1 - k0;
  const bool ok = t >= q0 && t < q1 && T <= L && k0 >= 0 && k1 <= s.total_k &&
                  L <= s.max_k_len && q1 <= s.total_q;
  if (!ok) {
    atomicOr(status, DSA_FLAG_BAD_SEQS);
    return false;
  }
  r.b = b;
  r.pos = L - T + (t - q0);
  r.k0 = k0;
  r.L = L;
  return true;
}

// Cache row of key position `pos` of sequence b (k0 = cu_k[b]); -1 when the block table
// points outside the cache.  (Cache rows stay below 2^31; page_size is a power of two.)
__device__ __forceinline__ int key_row(const Seqs& s, int b, int k0, int pos) {
  if (!s.paged()) return k0 + pos;
  const int sh = __ffs(s.page_size) - 1;
  const int pg = __ldg(s.block_table + (int64_t)b * s.max_pages + (pos >> sh));
  if ((unsigned)pg >= (unsigned)s.num_pages) return -1;
  return (pg << sh) | (pos & (s.page_size - 1));
}

// Rows a 128-key tile is loaded in: a paged tile comes page by page.
__host__ __device__ __forceinline__ int tile_chunk_rows(const Seqs& s) {
  return s.paged() && s.page_size < 128 ? s.page_size : 128;
}

// ----------------------------------------------------------------------------
// Element loads (widening to fp32).
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__nv_fp8_e4m3 v) { return static_cast<float>(v); }

// Checked builds (-DDSA_CHECKED, built as libdsa_checked.so): the kernels test their internal
// invariants on the device (gather rows inside the cache, tile coordinates and query rows in
// range, output slots below top_k).  A failed test sets DSA_FLAG_CHECK in the status word and
// the caller clamps or skips the access; nothing traps.  Ordinary builds compile every test
// away (dsa_check is constant true).
#ifdef DSA_CHECKED
__device__ __forceinline__ bool dsa_check(bool ok, uint32_t* status) {
  if (!ok) atomicOr(status, DSA_FLAG_CHECK);
  return ok;
}
#else
__device__ __forceinline__ bool dsa_check(bool, uint32_t*) { return true; }
#endif

// An E8M0 scale byte (the MX formats' shared scale) as fp32: 2^(e - 127).  e = 0 is the
// fp32 subnormal 2^-127; e = 255 (NaN) is excluded by the interface.
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ void store_f32(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_f32(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 folds to +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// ----------------------------------------------------------------------------
// Host side: error reporting and launch tracing (defined in dsa_api.cu).
int set_error(int code, const char* fmt, ...);
void trace_pre(const char* name, cudaStream_t s);
void trace_post(cudaStream_t s);
int check_launch(const char* what);

// A 2-D tiled tensor map (128-byte swizzle unless `swizzle` is false, 256-byte L2
// promotion, zero fill): `rows` rows of `inner` elements, `row_bytes` apart; box =
// box_inner x box_rows.
int make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                 uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                 bool swizzle = true);
int num_sms();

#define DSA_LAUNCH(name, stream, ...)   \
  do {                                  \
    ::dsa::trace_pre(name, stream);     \
    __VA_ARGS__;                        \
    ::dsa::trace_post(stream);          \
  } while (0)

// ----------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the
// kernel before it in the stream is still running; it must run griddep_wait() before it
// reads anything that kernel writes.  griddep_launch() lets the next such kernel start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------
// Kernel launchers (each defined in its own .cu).
struct IndexerArgs {
  Seqs seqs;
  int h_idx, d_idx, idx_dtype;
  const void* q_idx;
  const void* k_idx;
  const float* w;
  const float* q_scale;
  const float* k_scale;
  uint32_t* status;
  uint32_t* hist = nullptr;  // tensor-core path: also fill the Top-K histogram (zero on entry)
  // Only the packed query rows [row0, row1) are scored; their scores (and histograms) go
  // to rows t - row0 of the output.
  int row0 = 0, row1 = 0x7fffffff;
};

int launch_indexer_scores_simt(const IndexerArgs& a, float* scores, int64_t ld,
                               cudaStream_t stream);

// tcgen05 indexer (H_I = 64, d_I = 128, bf16 or FP8): writes scores[t, s] for s <= pos(t).
bool indexer_tc_eligible(const IndexerArgs& a);
int launch_indexer_tc(const IndexerArgs& a, float* scores, int64_t ld, cudaStream_t stream);
// Whether the tcgen05 indexer scores blocks of four query rows (prefill-shaped problems).
bool indexer_tc_blocks4(const IndexerArgs& a);

// The fused indexer for rows that carry their own history (decode): scores, head weights
// and the causal Top-K in one cooperative kernel, one CTA per SM over equal shares of all
// rows' key tiles, scores kept in tensor memory; writes idx (ascending positions, -1
// padded) and optionally vals.  Its exchange buffers (per-row histograms and candidate
// lists) live in `scratch` (indexer_topk_scratch(a, nullptr).bytes); the thread blocks
// sharing a row wait for each other through the row's counter in the status block.
struct IndexerTopkScratch {
  size_t bytes;
  uint32_t* hist;
  uint32_t* rec;
  uint2* cand;
};
IndexerTopkScratch indexer_topk_scratch(const IndexerArgs& a, void* base);
bool indexer_topk_eligible(const IndexerArgs& a);
int launch_indexer_topk(const IndexerArgs& a, int top_k, int32_t* idx, float* vals,
                        void* scratch, cudaStream_t stream);

// Fill scores[t, s] = -inf for pos(t) < s < ld.
int launch_mask_tail(const Seqs& seqs, float* scores, int64_t ld, uint32_t* status,
                     cudaStream_t stream);

// Per-row histogram of score keys by their top 12 bits (order_key(s) >> 20).
constexpr int kHistBins = 4096;

struct TopkArgs {
  Seqs seqs;
  int top_k;
  const float* scores;
  int64_t ld;
  int32_t* idx;
  float* vals;
  uint32_t* status;
  const uint32_t* hist = nullptr;  // [rows][kHistBins] or null
  // Only the packed query rows [row0, row0 + nrows) are selected (nrows < 0: all); their
  // scores (and histograms) are rows t - row0 of `scores` (and `hist`).
  int row0 = 0, nrows = -1;
  __host__ __device__ int rows() const { return nrows < 0 ? seqs.total_q - row0 : nrows; }
};
int launch_topk_rows(const TopkArgs& a, cudaStream_t stream);
// Shared-memory-resident variant for rows of at most topk_smem_max_keys() keys.
int topk_smem_max_keys();
int launch_topk_smem(const TopkArgs& a, cudaStream_t stream);
// One 256-thread CTA streaming each row, histogram-seeded (a.hist set).
// buf [rows][buf_ld] int32, buf_ld >= max_k_len: candidates of rows that do not fit
// in shared memory.
int launch_topk_stream(const TopkArgs& a, int32_t* buf, int64_t buf_ld, cudaStream_t stream);

struct SfaArgs {
  Seqs seqs;
  int h, d_c, d_rope, top_k, kv_dtype, out_dtype;
  float scale;
  const void* q;
  const void* kv;
  const int32_t* idx;
  void* out;
  float* lse;
  uint32_t* status;
};
int launch_sfa_simt(const SfaArgs& a, cudaStream_t stream);

// tcgen05 SFA (H = 128, d_c = 512, d_rope = 64, bf16) on 2-CTA clusters; with few query
// rows a second kernel merges the rows cut into pieces.
bool sfa_tc_eligible(const SfaArgs& a);
size_t sfa_tc_scratch_bytes(int total_q);
int launch_sfa_tc(const SfaArgs& a, void* scratch, cudaStream_t stream);

}  // namespace dsa
