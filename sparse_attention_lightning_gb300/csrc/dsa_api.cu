// C ABI of libdsa.so: argument checks, workspace carving, kernel dispatch,
// status word, error strings and launch tracing.  See include/dsa.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {

// One thread waits, through the kernels' bounded wait, on an mbarrier that nothing arrives at:
// it gives up after limit_ns, ORs DSA_FLAG_TIMEOUT into the status word and returns.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  abort_flag = 0;
  tc::fence_barrier_init();
  tc::mbar_wait_for(&bar, 0, limit_ns, &abort_flag, status, DSA_FLAG_TIMEOUT);
}

// ----------------------------------------------------------------------------
// Errors.
static thread_local std::string g_last_error;

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DSA_OK;
}

// ----------------------------------------------------------------------------
// Device properties and tensor maps.
int num_sms() {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 1;
  }
  return n[dev];
}

int make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                 uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                 bool swizzle) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
      return set_error(DSA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    fn = reinterpret_cast<EncodeFn>(f);
  }
  if (rows == 0) rows = 1;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DSA_OK;
}

// ----------------------------------------------------------------------------
// Launch tracing: an event pair around each launch while enabled.
namespace {
struct TraceRec {
  std::string name;
  cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
int g_trace_cap = 0;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;
int g_trace_open = -1;  // record awaiting its end event
}  // namespace

void trace_pre(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on || (int)g_trace.size() >= g_trace_cap) return;
  const size_t i = g_trace.size();
  TraceRec r{name, g_event_pool[2 * i], g_event_pool[2 * i + 1]};
  cudaEventRecord(r.a, s);
  g_trace.push_back(r);
  g_trace_open = (int)i;
}

void trace_post(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_trace_open < 0) return;
  cudaEventRecord(g_trace[g_trace_open].b, s);
  g_trace_open = -1;
}

// ----------------------------------------------------------------------------
// Descriptor checks.
namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_ptr(const void* p, const char* name, bool nullable = false) {
  if (!p) {
    if (nullable) return DSA_OK;
    return set_error(DSA_ERR_INVALID_ARG, "%s is NULL", name);
  }
  if (!aligned16(p)) return set_error(DSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return DSA_OK;
}

int check_problem(const dsa_problem* p, bool need_indexer, bool need_attn) {
  if (!p) return set_error(DSA_ERR_INVALID_ARG, "problem descriptor is NULL");
  if (p->num_seqs < 1) return set_error(DSA_ERR_INVALID_ARG, "num_seqs = %d", p->num_seqs);
  if (p->total_q < 0 || p->total_k < 1)
    return set_error(DSA_ERR_INVALID_ARG, "total_q = %d, total_k = %d", p->total_q, p->total_k);
  if (p->max_k_len < 1 || p->max_k_len > p->total_k || p->max_q_len < 0 ||
      p->max_q_len > p->max_k_len)
    return set_error(DSA_ERR_INVALID_ARG, "max_q_len = %d, max_k_len = %d", p->max_q_len,
                     p->max_k_len);
  if (p->max_k_len > (1 << 30)) return set_error(DSA_ERR_UNSUPPORTED, "max_k_len > 2^30");
  if (p->top_k < 1 || p->top_k > 2048)
    return set_error(DSA_ERR_UNSUPPORTED, "top_k = %d (supported 1..2048)", p->top_k);
  if (!p->cu_q || !p->cu_k) return set_error(DSA_ERR_INVALID_ARG, "cu_q/cu_k is NULL");
  if (p->page_size != 0) {
    const int ps = p->page_size;
    if (ps < 16 || (ps & (ps - 1)) != 0)
      return set_error(DSA_ERR_UNSUPPORTED, "page_size = %d (a power of two >= 16)", ps);
    if (!p->block_table) return set_error(DSA_ERR_INVALID_ARG, "paged caches need a block_table");
    if (((uintptr_t)p->block_table & 15u) != 0)
      return set_error(DSA_ERR_INVALID_ARG, "block_table is not 16-byte aligned");
    if (p->num_pages < 1 || p->max_pages < 1 || (int64_t)p->max_pages * ps < p->max_k_len)
      return set_error(DSA_ERR_INVALID_ARG, "num_pages = %d, max_pages = %d do not cover max_k_len",
                       p->num_pages, p->max_pages);
    if ((int64_t)p->num_pages * ps >= (int64_t(1) << 31))
      return set_error(DSA_ERR_UNSUPPORTED, "num_pages * page_size >= 2^31");
  }
  if (need_indexer) {
    if (p->h_idx < 1 || p->h_idx > 128)
      return set_error(DSA_ERR_UNSUPPORTED, "h_idx = %d (supported 1..128)", p->h_idx);
    if (p->d_idx < 16 || p->d_idx > 256 || p->d_idx % 16)
      return set_error(DSA_ERR_UNSUPPORTED, "d_idx = %d (supported 16..256, multiple of 16)",
                       p->d_idx);
    if (p->idx_dtype != DSA_F32 && p->idx_dtype != DSA_BF16 && p->idx_dtype != DSA_FP8_E4M3 &&
        p->idx_dtype != DSA_MXFP8_E4M3)
      return set_error(DSA_ERR_INVALID_ARG, "idx_dtype = %d", p->idx_dtype);
    if (p->idx_dtype == DSA_MXFP8_E4M3 && p->d_idx % 32)
      return set_error(DSA_ERR_UNSUPPORTED, "MXFP8 needs d_idx a multiple of 32 (d_idx = %d)",
                       p->d_idx);
  }
  if (need_attn) {
    if (p->h < 1 || p->h > 128) return set_error(DSA_ERR_UNSUPPORTED, "h = %d (1..128)", p->h);
    if (p->d_c < 16 || p->d_c > 1024 || p->d_c % 16)
      return set_error(DSA_ERR_UNSUPPORTED, "d_c = %d (16..1024, multiple of 16)", p->d_c);
    if (p->d_rope < 0 || p->d_rope > 256 || p->d_rope % 16)
      return set_error(DSA_ERR_UNSUPPORTED, "d_rope = %d (0..256, multiple of 16)", p->d_rope);
    if (p->kv_dtype != DSA_F32 && p->kv_dtype != DSA_BF16)
      return set_error(DSA_ERR_UNSUPPORTED, "kv_dtype = %d (F32 or BF16)", p->kv_dtype);
    if (p->out_dtype != DSA_F32 && p->out_dtype != DSA_BF16)
      return set_error(DSA_ERR_UNSUPPORTED, "out_dtype = %d (F32 or BF16)", p->out_dtype);
    if (!(p->sm_scale >= 0.f) || isinf(p->sm_scale))
      return set_error(DSA_ERR_INVALID_ARG, "sm_scale must be finite and >= 0");
  }
  return DSA_OK;
}

Seqs seqs_of(const dsa_problem* p) {
  Seqs s{p->cu_q, p->cu_k, p->num_seqs, p->total_q, p->total_k, p->max_k_len};
  if (p->page_size > 0) {
    s.block_table = p->block_table;
    s.page_size = p->page_size;
    s.max_pages = p->max_pages;
    s.num_pages = p->num_pages;
  }
  return s;
}

float scale_of(const dsa_problem* p) {
  return p->sm_scale > 0.f ? p->sm_scale : 1.0f / sqrtf((float)(p->d_c + p->d_rope));
}

// Scratch regions after the status block.
struct Carve {
  size_t off = kStatusBytes;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  }
};

// Workspace score rows are padded to 32 floats (128 B) so every row is aligned.
int64_t scores_ld(const dsa_problem* p) { return ((int64_t)p->max_k_len + 31) / 32 * 32; }
size_t idx_bytes(const dsa_problem* p) { return (size_t)p->total_q * p->top_k * 4; }

IndexerArgs indexer_args(const dsa_problem* p, const void* q_idx, const void* k_idx,
                         const float* w, const float* q_scale, const float* k_scale,
                         void* ws) {
  const bool fp8 = p->idx_dtype == DSA_FP8_E4M3 || p->idx_dtype == DSA_MXFP8_E4M3;
  return IndexerArgs{seqs_of(p), p->h_idx, p->d_idx, p->idx_dtype, q_idx, k_idx, w,
                     fp8 ? q_scale : nullptr, fp8 ? k_scale : nullptr,
                     static_cast<uint32_t*>(ws)};
}

// Rows that carry their own history (decode) run the one-kernel fused indexer, which keeps
// every score on chip; its scratch holds per-row histograms and candidate lists only.
// Prefill-shaped problems (several queries per
// sequence: the tensor-core indexer scores blocks of four rows against each key tile) and
// shapes that kernel does not cover score the rows in chunks: a chunk's scores go to a
// bounded workspace buffer (sized for L2, not for the whole problem) and its Top-K reads
// them back before the next chunk is scored.
bool row_fused(const dsa_problem* p) {
  const IndexerArgs ia = indexer_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  return indexer_topk_eligible(ia) && !indexer_tc_blocks4(ia);
}
bool tc_scores(const dsa_problem* p) {
  const IndexerArgs ia = indexer_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  return indexer_tc_eligible(ia);
}
int64_t spill_ld(const dsa_problem* p) { return ((int64_t)p->max_k_len + 3) / 4 * 4; }

// Bytes of chunk scratch per query row, and the rows of one chunk.
constexpr size_t kChunkBudget = size_t(256) << 20;
size_t chunk_row_bytes(const dsa_problem* p) {
  size_t b = (size_t)scores_ld(p) * 4;
  if (tc_scores(p)) b += (size_t)kHistBins * 4 + (size_t)spill_ld(p) * 4;
  return b;
}
int chunk_rows(const dsa_problem* p) {
  if (p->total_q == 0 || row_fused(p)) return 0;
  size_t r = kChunkBudget / chunk_row_bytes(p);
  if (r < 1) r = 1;
  return (int)(r < (size_t)p->total_q ? r : (size_t)p->total_q);
}

// Fused indexer scratch: the one-kernel path's exchange buffers; for the chunked path a
// chunk's scores [rows][scores_ld] f32,
// histograms [rows][kHistBins] and Top-K candidate positions [rows][spill_ld]; then the
// fused forward's indices and the attention scratch.
struct IndexerScratch {
  void* fused;  // the fused decode kernel's exchange buffers
  float* scores;
  uint32_t* hist;
  int32_t* spill;
  int32_t* idx;
  void* sfa;
};

// SFA scratch of the tensor-core path (per-CTA key-row lists, split-row partials).
size_t sfa_scratch_bytes(const dsa_problem* p) {
  const bool tc = p->kv_dtype == DSA_BF16 && p->h == 128 && p->d_c == 512 && p->d_rope == 64;
  return tc ? sfa_tc_scratch_bytes(p->total_q) : 0;
}

size_t carve_indexer(const dsa_problem* p, void* ws, IndexerScratch* out) {
  Carve c;
  const size_t rows = (size_t)chunk_rows(p);
  const bool tc = tc_scores(p);
  const IndexerArgs ia = indexer_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  const size_t o_fused = c.take(row_fused(p) ? indexer_topk_scratch(ia, nullptr).bytes : 0);
  const size_t o_scores = c.take(rows * scores_ld(p) * 4);
  const size_t o_hist = c.take(tc ? rows * kHistBins * 4 : 0);
  const size_t o_spill = c.take(tc ? rows * spill_ld(p) * 4 : 0);
  const size_t o_idx = c.take(idx_bytes(p));
  const size_t o_sfa = c.take(sfa_scratch_bytes(p));
  if (out) {
    char* b = static_cast<char*>(ws);
    out->fused = b + o_fused;
    out->scores = reinterpret_cast<float*>(b + o_scores);
    out->hist = tc ? reinterpret_cast<uint32_t*>(b + o_hist) : nullptr;
    out->spill = reinterpret_cast<int32_t*>(b + o_spill);
    out->idx = reinterpret_cast<int32_t*>(b + o_idx);
    out->sfa = b + o_sfa;
  }
  return c.off;
}

size_t ws_fused_indexer(const dsa_problem* p) { return carve_indexer(p, nullptr, nullptr); }
size_t ws_fused_forward(const dsa_problem* p) { return carve_indexer(p, nullptr, nullptr); }
size_t ws_sfa(const dsa_problem* p) {
  Carve c;
  c.take(sfa_scratch_bytes(p));
  return c.off;
}
size_t ws_indexer_scores(const dsa_problem*) { return kStatusBytes; }

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return set_error(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return set_error(DSA_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  if (ws_bytes < need)
    return set_error(DSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return DSA_OK;
}

#define DSA_TRY(expr)            \
  do {                           \
    int _rc = (expr);            \
    if (_rc != DSA_OK) return _rc; \
  } while (0)

int check_indexer_inputs(const dsa_problem* p, const void* q_idx, const void* k_idx,
                         const float* w, const float* q_scale, const float* k_scale) {
  DSA_TRY(check_ptr(q_idx, "q_idx", p->total_q == 0));
  DSA_TRY(check_ptr(k_idx, "k_idx"));
  DSA_TRY(check_ptr(w, "w", p->total_q == 0));
  if (p->idx_dtype == DSA_FP8_E4M3 || p->idx_dtype == DSA_MXFP8_E4M3) {
    DSA_TRY(check_ptr(q_scale, "q_scale", p->total_q == 0));
    DSA_TRY(check_ptr(k_scale, "k_scale"));
  }
  return DSA_OK;
}

int run_topk(const TopkArgs& ta, cudaStream_t s) {
  if (ta.seqs.max_k_len <= topk_smem_max_keys()) return launch_topk_smem(ta, s);
  return launch_topk_rows(ta, s);
}

int run_fused_indexer(const dsa_problem* p, const void* q_idx, const void* k_idx, const float* w,
                      const float* q_scale, const float* k_scale, int32_t* idx, float* vals,
                      void* ws, cudaStream_t s) {
  IndexerArgs ia = indexer_args(p, q_idx, k_idx, w, q_scale, k_scale, ws);
  IndexerScratch sc;
  carve_indexer(p, ws, &sc);
  if (row_fused(p)) return launch_indexer_topk(ia, p->top_k, idx, vals, sc.fused, s);
  const int64_t ld = scores_ld(p);
  const bool tc = tc_scores(p);
  const int rows = chunk_rows(p);
  for (int r0 = 0; r0 < p->total_q; r0 += rows) {
    const int r1 = r0 + rows < p->total_q ? r0 + rows : p->total_q;
    ia.row0 = r0;
    ia.row1 = r1;
    TopkArgs ta{seqs_of(p), p->top_k, sc.scores, ld, idx, vals, static_cast<uint32_t*>(ws)};
    ta.row0 = r0;
    ta.nrows = r1 - r0;
    if (tc) {
      ia.hist = sc.hist;
      cudaError_t e = cudaMemsetAsync(sc.hist, 0, (size_t)(r1 - r0) * kHistBins * 4, s);
      if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "hist clear: %s", cudaGetErrorString(e));
      DSA_TRY(launch_indexer_tc(ia, sc.scores, ld, s));
      ta.hist = sc.hist;
      DSA_TRY(launch_topk_stream(ta, sc.spill, spill_ld(p), s));
    } else {
      DSA_TRY(launch_indexer_scores_simt(ia, sc.scores, ld, s));
      DSA_TRY(run_topk(ta, s));
    }
  }
  return DSA_OK;
}

SfaArgs sfa_args(const dsa_problem* p, const void* q, const void* kv, const int32_t* idx,
                 void* out, float* lse, void* ws) {
  return SfaArgs{seqs_of(p), p->h, p->d_c, p->d_rope, p->top_k, p->kv_dtype, p->out_dtype,
                 scale_of(p), q, kv, idx, out, lse, static_cast<uint32_t*>(ws)};
}

int run_sfa(const dsa_problem* p, const void* q, const void* kv, const int32_t* idx, void* out,
            float* lse, void* ws, void* scratch, cudaStream_t s) {
  const SfaArgs sa = sfa_args(p, q, kv, idx, out, lse, ws);
  if (sfa_tc_eligible(sa)) return launch_sfa_tc(sa, scratch, s);
  return launch_sfa_simt(sa, s);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_status_str(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported problem";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSA_ERR_TIMEOUT: return "a bounded device wait timed out";
  }
  return "unknown status";
}

const char* dsa_last_error(void) { return g_last_error.c_str(); }

int dsa_workspace_size(const dsa_problem* p, int op, size_t* bytes) {
  if (!bytes) return set_error(DSA_ERR_INVALID_ARG, "bytes is NULL");
  switch (op) {
    case DSA_OP_INDEXER_SCORES:
      DSA_TRY(check_problem(p, true, false));
      *bytes = ws_indexer_scores(p);
      break;
    case DSA_OP_TOPK: DSA_TRY(check_problem(p, false, false)); *bytes = kStatusBytes; break;
    case DSA_OP_FUSED_INDEXER:
      DSA_TRY(check_problem(p, true, false));
      *bytes = ws_fused_indexer(p);
      break;
    case DSA_OP_SPARSE_MLA_ATTN:
      DSA_TRY(check_problem(p, false, true));
      *bytes = ws_sfa(p);
      break;
    case DSA_OP_FUSED_FORWARD:
      DSA_TRY(check_problem(p, true, true));
      *bytes = ws_fused_forward(p);
      break;
    default: return set_error(DSA_ERR_INVALID_ARG, "unknown op %d", op);
  }
  return DSA_OK;
}

int dsa_indexer_scores(const dsa_problem* p, const void* q_idx, const void* k_idx,
                       const float* w, const float* q_scale, const float* k_scale,
                       float* scores, int64_t ld, void* ws, size_t ws_bytes, void* stream) {
  DSA_TRY(check_problem(p, true, false));
  DSA_TRY(check_indexer_inputs(p, q_idx, k_idx, w, q_scale, k_scale));
  DSA_TRY(check_ptr(scores, "scores", p->total_q == 0));
  if (ld < p->max_k_len) return set_error(DSA_ERR_INVALID_ARG, "ld < max_k_len");
  DSA_TRY(check_ws(ws, ws_bytes, ws_indexer_scores(p)));
  IndexerArgs ia = indexer_args(p, q_idx, k_idx, w, q_scale, k_scale, ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (indexer_tc_eligible(ia)) {
    DSA_TRY(launch_indexer_tc(ia, scores, ld, s));
    return launch_mask_tail(seqs_of(p), scores, ld, static_cast<uint32_t*>(ws), s);
  }
  return launch_indexer_scores_simt(ia, scores, ld, s);
}

int dsa_topk(const dsa_problem* p, const float* scores, int64_t ld, int32_t* idx, float* vals,
             void* ws, size_t ws_bytes, void* stream) {
  DSA_TRY(check_problem(p, false, false));
  DSA_TRY(check_ptr(scores, "scores", p->total_q == 0));
  DSA_TRY(check_ptr(idx, "idx", p->total_q == 0));
  DSA_TRY(check_ptr(vals, "vals", true));
  if (ld < p->max_k_len) return set_error(DSA_ERR_INVALID_ARG, "ld < max_k_len");
  DSA_TRY(check_ws(ws, ws_bytes, kStatusBytes));
  TopkArgs ta{seqs_of(p), p->top_k, scores, ld, idx, vals, static_cast<uint32_t*>(ws)};
  return run_topk(ta, static_cast<cudaStream_t>(stream));
}

int dsa_fused_indexer(const dsa_problem* p, const void* q_idx, const void* k_idx,
                      const float* w, const float* q_scale, const float* k_scale,
                      int32_t* idx, float* vals, void* ws, size_t ws_bytes, void* stream) {
  DSA_TRY(check_problem(p, true, false));
  DSA_TRY(check_indexer_inputs(p, q_idx, k_idx, w, q_scale, k_scale));
  DSA_TRY(check_ptr(idx, "idx", p->total_q == 0));
  DSA_TRY(check_ptr(vals, "vals", true));
  DSA_TRY(check_ws(ws, ws_bytes, ws_fused_indexer(p)));
  return run_fused_indexer(p, q_idx, k_idx, w, q_scale, k_scale, idx, vals, ws,
                           static_cast<cudaStream_t>(stream));
}

int dsa_sparse_mla_attn(const dsa_problem* p, const void* q, const void* kv, const int32_t* idx,
                        void* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  DSA_TRY(check_problem(p, false, true));
  DSA_TRY(check_ptr(q, "q", p->total_q == 0));
  DSA_TRY(check_ptr(kv, "kv"));
  DSA_TRY(check_ptr(idx, "idx", p->total_q == 0));
  DSA_TRY(check_ptr(out, "out", p->total_q == 0));
  DSA_TRY(check_ptr(lse, "lse", true));
  DSA_TRY(check_ws(ws, ws_bytes, ws_sfa(p)));
  Carve c;
  void* scratch = static_cast<char*>(ws) + c.take(sfa_scratch_bytes(p));
  return run_sfa(p, q, kv, idx, out, lse, ws, scratch, static_cast<cudaStream_t>(stream));
}

int dsa_fused_forward(const dsa_problem* p, const void* q_idx, const void* k_idx,
                      const float* w, const float* q_scale, const float* k_scale,
                      const void* q, const void* kv, void* out, float* lse,
                      int32_t* idx_out, float* vals_out, void* ws, size_t ws_bytes,
                      void* stream) {
  DSA_TRY(check_problem(p, true, true));
  DSA_TRY(check_indexer_inputs(p, q_idx, k_idx, w, q_scale, k_scale));
  DSA_TRY(check_ptr(q, "q", p->total_q == 0));
  DSA_TRY(check_ptr(kv, "kv"));
  DSA_TRY(check_ptr(out, "out", p->total_q == 0));
  DSA_TRY(check_ptr(lse, "lse", true));
  DSA_TRY(check_ptr(idx_out, "idx_out", true));
  DSA_TRY(check_ptr(vals_out, "vals_out", true));
  DSA_TRY(check_ws(ws, ws_bytes, ws_fused_forward(p)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  IndexerScratch sc;
  carve_indexer(p, ws, &sc);
  int32_t* idx = idx_out ? idx_out : sc.idx;
  // the kernels run back to back: each may start while the one before it finishes
  DSA_TRY(run_fused_indexer(p, q_idx, k_idx, w, q_scale, k_scale, idx, vals_out, ws, s));
  return run_sfa(p, q, kv, idx, out, lse, ws, sc.sfa, s);
}

int dsa_clear_status(void* ws, void* stream) {
  if (!ws) return set_error(DSA_ERR_WORKSPACE, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "clear_status: %s", cudaGetErrorString(e));
  return DSA_OK;
}

int dsa_read_status(const void* ws, void* stream, uint32_t* flags) {
  if (!ws || !flags) return set_error(DSA_ERR_INVALID_ARG, "ws/flags is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "read_status: %s", cudaGetErrorString(e));
  if (*flags & DSA_FLAG_TIMEOUT) return set_error(DSA_ERR_TIMEOUT, "device wait timed out");
  return DSA_OK;
}

int dsa_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream) {
  if (!ws) return set_error(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return set_error(DSA_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  if (limit_ns == 0 || limit_ns > 100000000ull)
    return set_error(DSA_ERR_INVALID_ARG, "limit_ns must be in (0, 1e8]");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DSA_LAUNCH("wait_selftest", s,
             wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<uint32_t*>(ws), limit_ns));
  return check_launch("wait_selftest");
}

int dsa_trace_begin(int capacity) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (capacity < 0) return set_error(DSA_ERR_INVALID_ARG, "capacity < 0");
  for (size_t i = g_event_pool.size(); i < 2 * (size_t)capacity; ++i) {
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "trace: %s", cudaGetErrorString(e));
    g_event_pool.push_back(ev);
  }
  g_trace.clear();
  g_trace_cap = capacity;
  g_trace_open = -1;
  g_trace_on = true;
  return DSA_OK;
}

int dsa_trace_end(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  return DSA_OK;
}

int dsa_trace_count(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  return (int)g_trace.size();
}

int dsa_trace_get(int i, char* name, int name_len, float* ms) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (i < 0 || i >= (int)g_trace.size()) return set_error(DSA_ERR_INVALID_ARG, "trace index");
  const TraceRec& r = g_trace[i];
  if (name && name_len > 0) {
    strncpy(name, r.name.c_str(), (size_t)name_len - 1);
    name[name_len - 1] = 0;
  }
  if (ms) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, r.a, r.b);
    if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "trace: %s", cudaGetErrorString(e));
  }
  return DSA_OK;
}

}  // extern "C"
