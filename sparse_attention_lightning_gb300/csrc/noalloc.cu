// dsa_fused_indexer_static: the fused indexer with its scratch in a static
// device array, for callers that cannot allocate device memory.
//
// Who needs it: code that runs inside a host framework owning every byte of
// device memory (a fixed memory budget or its own caching allocator, with raw
// cudaMalloc forbidden), and latency-critical loops where a cudaMalloc or
// cudaFree would implicitly synchronise the device.  Such callers can hand us
// their inputs and outputs but not a workspace.
//
// The scratch lives in `g_static_scratch` below: a status block followed by
// the score rows.  Each device that loads this library holds the array until
// the process exits.  The first call on a device looks up the array's device
// address (cudaGetSymbolAddress, with that device current); make that first
// call before any stream capture.  All calls on a device share the array, so
// calls that overlap on the GPU (different streams, no ordering) race; the
// array keeps the last call's contents, and each call clears the status block
// before its kernels run.
#include <mutex>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr size_t kStaticScoreFloats = size_t(1) << 22;  // 16 MiB of fp32 scores
constexpr size_t kStaticBytes = kStatusBytes + kStaticScoreFloats * sizeof(float);

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up once).
int static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(DSA_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return set_error(DSA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DSA_OK;
}

bool ok16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_fused_indexer_static(const dsa_problem* p, const void* q_idx,
                                        const void* k_idx, const float* w, const float* q_scale,
                                        const float* k_scale, int32_t* idx, float* vals,
                                        uint32_t* flags_out, void* stream) {
  if (!p) return set_error(DSA_ERR_INVALID_ARG, "problem descriptor is NULL");
  // reuse the library's descriptor checks through the workspace-size query
  size_t ws_need = 0;
  int rc = dsa_workspace_size(p, DSA_OP_INDEXER_SCORES, &ws_need);
  if (rc != DSA_OK) return rc;
  const size_t need = (size_t)p->total_q * (size_t)p->max_k_len;
  if (need > kStaticScoreFloats)
    return set_error(DSA_ERR_UNSUPPORTED,
                     "dsa_fused_indexer_static: total_q*max_k_len = %zu exceeds the static "
                     "scratch of %zu scores",
                     need, kStaticScoreFloats);
  const bool fp8 = p->idx_dtype == DSA_FP8_E4M3 || p->idx_dtype == DSA_MXFP8_E4M3;
  const bool none = p->total_q == 0;
  if ((!q_idx && !none) || !k_idx || (!w && !none) || (!idx && !none))
    return set_error(DSA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (fp8 && ((!q_scale && !none) || !k_scale))
    return set_error(DSA_ERR_INVALID_ARG, "FP8 needs q_scale and k_scale");
  const void* ptrs[] = {q_idx, k_idx, w, q_scale, k_scale, idx, vals, flags_out};
  for (const void* q : ptrs)
    if (q && !ok16(q)) return set_error(DSA_ERR_INVALID_ARG, "a pointer is not 16-byte aligned");

  void* base = nullptr;
  rc = static_scratch(&base);
  if (rc != DSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(base);
  float* scores = reinterpret_cast<float*>(static_cast<char*>(base) + kStatusBytes);

  cudaError_t e = cudaMemsetAsync(status, 0, kStatusBytes, s);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "clear status: %s", cudaGetErrorString(e));
  Seqs seqs{p->cu_q, p->cu_k, p->num_seqs, p->total_q, p->total_k, p->max_k_len};
  if (p->page_size > 0) {  // paged key caches (checked by dsa_workspace_size above)
    seqs.block_table = p->block_table;
    seqs.page_size = p->page_size;
    seqs.max_pages = p->max_pages;
    seqs.num_pages = p->num_pages;
  }
  IndexerArgs ia{seqs, p->h_idx, p->d_idx, p->idx_dtype, q_idx, k_idx, w,
                 fp8 ? q_scale : nullptr, fp8 ? k_scale : nullptr, status};
  rc = launch_indexer_scores_simt(ia, scores, p->max_k_len, s);
  if (rc != DSA_OK) return rc;
  TopkArgs ta{seqs, p->top_k, scores, p->max_k_len, idx, vals, status};
  rc = launch_topk_rows(ta, s);
  if (rc != DSA_OK) return rc;
  if (flags_out) {
    e = cudaMemcpyAsync(flags_out, status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "flags: %s", cudaGetErrorString(e));
  }
  return DSA_OK;
}
