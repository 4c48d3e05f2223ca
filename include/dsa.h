/*
 * dsa.h — C ABI of libdsa.so, the GB300 (sm_103a) DSA hot path.
 *
 * DSA ("dynamic sparse attention") is the sparse-attention layer of a hybrid
 * MLA-based model.  A lightweight Lightning Indexer scores every historical
 * position of a query, keeps the Top-K positions, and Sparse Flash Attention
 * (SFA) attends over the MLA latent KV rows at just those positions
 * ("Day0 Inference Adaptation and Performance Optimization for New-Architecture
 * LLMs", §2.2 The Sparse Attention Path and §4.1 Indexer Fusion; "Day0 Inference
 * Adaptation and Performance Optimization for a New Architecture Domestic Large
 * Language Model on Ascend", §2 and §4).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Return value.  Every call returns a dsa_status code (0 = DSA_OK).  No C++
 *   exception crosses the ABI.  dsa_last_error() gives a message for the last
 *   failing call of the calling thread.
 * Pointers.  Every tensor pointer is caller-owned DEVICE memory (cudaMalloc or
 *   torch), 16-byte aligned.  The library never allocates, frees or retains
 *   them.  Tensors are dense, row-major, packed along tokens (no padding
 *   between sequences).
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Calls only enqueue work; argument checks are synchronous and a
 *   failing check launches nothing.
 * Workspace.  Every call takes a caller-owned device workspace of at least
 *   dsa_workspace_size() bytes.  Its first 16384 bytes are the status block.  Its
 *   first word is the device status word: kernels OR DSA_FLAG_* bits into it when
 *   they detect bad data (an index out of range, inconsistent cu_q/cu_k) or give
 *   up a bounded wait.  The word is sticky: clear it with dsa_clear_status() and
 *   read it with dsa_read_status().  The block's other words are counters through
 *   which the thread blocks of one kernel wait for each other; they must be zero
 *   before the workspace's first call (a zero-filled workspace, or
 *   dsa_clear_status()), and every call that completes without DSA_FLAG_TIMEOUT
 *   leaves them consistent.  After a call that set DSA_FLAG_TIMEOUT, call
 *   dsa_clear_status() before the next one.  The rest of the
 *   workspace is scratch owned by the call while it runs; calls sharing one
 *   workspace must be stream-ordered.  Its contents between calls are the
 *   caller's (a call never relies on earlier contents).
 * Sequences.  Query rows and key rows are packed: sequence b owns query rows
 *   cu_q[b] .. cu_q[b+1]-1 and key rows cu_k[b] .. cu_k[b+1]-1, with
 *   T_b = cu_q[b+1]-cu_q[b] <= L_b = cu_k[b+1]-cu_k[b].  The queries of a
 *   sequence are its last T_b tokens: query i of sequence b is at position
 *   pos = L_b - T_b + i and sees keys 0..pos of its own sequence (causal,
 *   inclusive; index computation is causal, "… New-Architecture LLMs" §6.2).
 *   Prefill has T_b = L_b (pos = i); decode has T_b = 1 (pos = L_b - 1).
 *   Positions written to / read from `idx` are local to the sequence.  The key-side
 *   tensors (k_idx, kv, k_scale) are either packed the same way or paged through a
 *   block table (dsa_problem.page_size, below).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 4

/* Return codes. */
enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, inconsistent descriptor */
  DSA_ERR_UNSUPPORTED = 2,  /* a valid combination this build has no kernel for */
  DSA_ERR_CUDA = 3,         /* a CUDA runtime call or a launch failed */
  DSA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than dsa_workspace_size() */
  DSA_ERR_TIMEOUT = 5       /* dsa_read_status saw DSA_FLAG_TIMEOUT */
};

/* Element types. */
enum dsa_dtype {
  DSA_F32 = 0,       /* IEEE binary32 */
  DSA_BF16 = 1,      /* bfloat16 */
  DSA_FP8_E4M3 = 2,  /* OCP FP8 E4M3 ("fn": no infinities), with fp32 scales */
  DSA_MXFP8_E4M3 = 3 /* MXFP8: E4M3 codes with one E8M0 scale (2^(e-127)) per 32 elements */
};

/* Device status flags (bits of the workspace status word). */
#define DSA_FLAG_BAD_INDEX 0x1u  /* SFA met an index outside [0, pos]; that entry was skipped */
#define DSA_FLAG_BAD_SEQS  0x2u  /* cu_q/cu_k inconsistent with the descriptor; rows were skipped */
#define DSA_FLAG_TIMEOUT   0x4u  /* a bounded on-device wait gave up; outputs are not valid */
#define DSA_FLAG_CHECK     0x8u  /* checked build only (libdsa_checked.so, -DDSA_CHECKED): an
                                  * internal invariant failed (a gather row outside the cache, a
                                  * tile coordinate or query row out of range, an output slot at
                                  * or past top_k); the access was clamped or skipped */

/* Operations, for dsa_workspace_size(). */
enum dsa_op {
  DSA_OP_INDEXER_SCORES = 1,
  DSA_OP_TOPK = 2,
  DSA_OP_FUSED_INDEXER = 3,
  DSA_OP_SPARSE_MLA_ATTN = 4,
  DSA_OP_FUSED_FORWARD = 5
};

/* Shape, types and sequence layout of one DSA problem. */
typedef struct dsa_problem {
  int32_t num_seqs;    /* B >= 1 */
  int32_t total_q;     /* ΣT_b >= 0: packed query rows */
  int32_t total_k;     /* ΣL_b >= 1: packed key rows */
  int32_t max_q_len;   /* max_b T_b (an upper bound is fine) */
  int32_t max_k_len;   /* max_b L_b (an upper bound is fine) */
  int32_t h_idx;       /* H_I: indexer heads */
  int32_t d_idx;       /* d_I: indexer head width */
  int32_t h;           /* H: MLA query heads (all share one latent row per key) */
  int32_t d_c;         /* latent width = value width */
  int32_t d_rope;      /* rope width; a latent row has D = d_c + d_rope columns */
  int32_t top_k;       /* k: positions kept per query */
  int32_t idx_dtype;   /* dsa_dtype of q_idx and k_idx (F32, BF16, FP8_E4M3, MXFP8_E4M3) */
  int32_t kv_dtype;    /* dsa_dtype of q and kv (F32 or BF16) */
  int32_t out_dtype;   /* dsa_dtype of out (F32 or BF16) */
  float sm_scale;      /* softmax scale; 0 selects 1/sqrt(D) */
  const int32_t* cu_q; /* device int32 [B+1], cu_q[0] = 0, cu_q[B] = total_q */
  const int32_t* cu_k; /* device int32 [B+1], cu_k[0] = 0, cu_k[B] = total_k */
  /* Paged key caches ("Day0 Inference Adaptation and Performance Optimization for
   * New-Architecture LLMs", §4.1: the fused indexer reads the paged K cache directly; "… on
   * Ascend", §4: the cache layout has to match the operators' addressing).  page_size = 0:
   * the caches are packed along tokens as described above (k_idx, kv and k_scale have
   * total_k rows, sequence b owning rows cu_k[b] .. cu_k[b+1]-1).  page_size > 0: the
   * caches hold num_pages pages of page_size rows each (num_pages * page_size rows), and
   * key position s of sequence b lives in cache row
   *   block_table[b * max_pages + s / page_size] * page_size + s % page_size;
   * cu_k then only gives the sequence lengths L_b = cu_k[b+1] - cu_k[b].  page_size must be
   * a power of two >= 16; max_pages * page_size >= max_k_len; num_pages * page_size < 2^31.  A block-table entry outside [0, num_pages) is reported with
   * DSA_FLAG_BAD_SEQS when the indexer reads it (those keys score 0) and with
   * DSA_FLAG_BAD_INDEX when attention meets one of its positions (the entry is skipped). */
  int32_t page_size;          /* 0 (contiguous) or the rows of a page */
  int32_t max_pages;          /* pages per block-table row */
  int32_t num_pages;          /* pages in the caches */
  const int32_t* block_table; /* device int32 [num_seqs][max_pages], or NULL if not paged */
} dsa_problem;

/* Limits of this build: 1 <= h_idx <= 128, d_idx in {16..256, multiple of 16},
 * 1 <= h <= 128, d_c in {16..1024, multiple of 16}, d_rope in {0..256, multiple
 * of 16}, 1 <= top_k <= 2048, max_k_len <= 2^30.  Outside them a call returns
 * DSA_ERR_UNSUPPORTED. */

/* Bytes of workspace `op` needs for problem `p` (always >= 16384). */
int dsa_workspace_size(const dsa_problem* p, int op, size_t* bytes);

/*
 * Lightning-Indexer relevance scores, materialised (for checking and
 * debugging; the fused calls below never write them to memory).
 *   scores[t, s] = Σ_j w[t,j] · ReLU(q_idx[t,j,:] · k_idx[s,:])   for s <= pos(t)
 *   scores[t, s] = -inf                                          for pos(t) < s < ld
 * ("… New-Architecture LLMs" §4.1: batched dot of the indexer query with the K
 * cache, then a weighted sum over heads; §2.2: each historical position gets a
 * relevance score.)
 * q_idx  [total_q, h_idx, d_idx] idx_dtype
 * k_idx  [total_k, d_idx]        idx_dtype
 * w      [total_q, h_idx]        f32 head weights
 * q_scale [total_q, h_idx] f32, k_scale [total_k] f32: dequantisation scales,
 *        required (and > 0) for FP8_E4M3, ignored (may be NULL) for F32/BF16:
 *        q = code·q_scale[t,j], k = code·k_scale[s].
 *        For MXFP8_E4M3 ("… New-Architecture LLMs" §5.1: index-side Q and K in
 *        MXFP8, one scale per 32 elements; d_idx a multiple of 32) the same two
 *        arguments point to E8M0 bytes instead: q_scale [total_q, h_idx, d_idx/32],
 *        k_scale [total_k, d_idx/32] (paged like k_idx), and
 *        q[t,j,c] = code·2^(q_scale[t,j,c/32] - 127), k[s,c] = code·2^(k_scale[s,c/32] - 127);
 *        byte 255 (NaN) is not allowed.
 * scores [total_q, ld] f32, ld >= max_k_len.
 */
int dsa_indexer_scores(const dsa_problem* p, const void* q_idx, const void* k_idx,
                       const float* w, const float* q_scale, const float* k_scale,
                       float* scores, int64_t ld, void* ws, size_t ws_bytes, void* stream);

/*
 * Causal Top-K of materialised scores (Top-K selection of the indexer,
 * "… New-Architecture LLMs" §4.1).  For each query row t, idx[t, 0..n-1]
 * (n = min(top_k, pos+1)) receives the positions of the n largest
 * scores[t, 0..pos], in ascending position order; among equal scores the
 * smaller positions are kept.  idx[t, n..top_k-1] = -1.
 * scores [total_q, ld] f32 (only columns 0..pos(t) are read)
 * idx    [total_q, top_k] int32
 * vals   [total_q, top_k] f32 or NULL: the selected scores (-inf in padding).
 */
int dsa_topk(const dsa_problem* p, const float* scores, int64_t ld, int32_t* idx, float* vals,
             void* ws, size_t ws_bytes, void* stream);

/*
 * The fused Lightning Indexer: scoring, head weighting and Top-K in one pass
 * over the K cache, writing only the selected positions ("… New-Architecture
 * LLMs" §4.1 fused_indexer(q_idx, k_cache, head_weights, top_k); "Optimizing
 * LLM Inference for New Architectures", §3: only the final Top-K indices leave
 * the operator).  Arguments and results are those of dsa_indexer_scores
 * followed by dsa_topk, except that the selected positions of a row may come
 * in any (deterministic) order: valid entries first, then -1 padding.
 */
int dsa_fused_indexer(const dsa_problem* p, const void* q_idx, const void* k_idx,
                      const float* w, const float* q_scale, const float* k_scale,
                      int32_t* idx, float* vals, void* ws, size_t ws_bytes, void* stream);

/*
 * Sparse Flash Attention over the MLA latent cache at the selected positions
 * ("… New-Architecture LLMs" §2.2 and §4.1: gather the selected KV rows and
 * attend over that subset; "… on Ascend" §4: SFA reads the KV cache at the
 * position set the indexer outputs).  For query row t and head h, over the
 * valid entries i of idx[t, :]:
 *   S_i = sm_scale · q[t,h,:] · kv[cu_k[b] + idx[t,i], :]        (all D columns)
 *   out[t,h,:] = Σ_i softmax(S)_i · kv[cu_k[b] + idx[t,i], 0:d_c]
 *   lse[t,h]   = log Σ_i exp(S_i)                                 (natural log)
 * q   [total_q, h, D] kv_dtype;  kv [total_k, D] kv_dtype (D = d_c + d_rope)
 * idx [total_q, top_k] int32: -1 entries are skipped; an entry outside
 *     [0, pos(t)] sets DSA_FLAG_BAD_INDEX and is skipped; order is free;
 *     a repeated entry counts as often as it appears.
 * out [total_q, h, d_c] out_dtype; lse [total_q, h] f32 or NULL.
 * A row with no valid entry gets out = 0 and lse = -inf.
 */
int dsa_sparse_mla_attn(const dsa_problem* p, const void* q, const void* kv, const int32_t* idx,
                        void* out, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * The whole DSA layer: dsa_fused_indexer then dsa_sparse_mla_attn on the same
 * stream ("… on Ascend" §4: the fused indexer's selected positions feed SFA).
 * idx_out [total_q, top_k] int32 and vals_out [total_q, top_k] f32 are optional
 * (NULL: kept in the workspace only).
 */
int dsa_fused_forward(const dsa_problem* p, const void* q_idx, const void* k_idx,
                      const float* w, const float* q_scale, const float* k_scale,
                      const void* q, const void* kv, void* out, float* lse,
                      int32_t* idx_out, float* vals_out, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * dsa_fused_indexer_static: dsa_fused_indexer for callers that cannot allocate
 * device memory.  The pages have no counterpart of this call; it exists for
 * code that runs inside a host framework owning all device memory (a fixed
 * budget or its own caching allocator, raw cudaMalloc forbidden) and for
 * latency-critical loops where cudaMalloc/cudaFree would synchronise the
 * device.  Such callers pass inputs and outputs but no workspace.
 *
 * Scratch is a static device array inside the library: a 16384-byte status block
 * plus room for 4,194,304 fp32 scores (16 MiB), held by every device that loads
 * the library until the process exits.  Problems with total_q * max_k_len above
 * 4,194,304 are rejected with DSA_ERR_UNSUPPORTED.  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).  Its first call on a
 * device looks up the array's address with that device current; make that first
 * call before any stream capture.  All calls on one device share the array:
 * calls that overlap on the GPU race, and the array keeps the last call's
 * contents.  Each call zeroes the status block first; if flags_out (device
 * memory, may be NULL) is given, the call's DSA_FLAG_* bits are copied there
 * at its end.  Other arguments and results are those of dsa_fused_indexer.
 */
int dsa_fused_indexer_static(const dsa_problem* p, const void* q_idx, const void* k_idx,
                             const float* w, const float* q_scale, const float* k_scale,
                             int32_t* idx, float* vals, uint32_t* flags_out, void* stream);

/*
 * The indexer prolog: Q quantisation and the head-weight projection, the two
 * input-preparation steps that share one stream ahead of the fused indexer
 * ("… New-Architecture LLMs" §4.2 Three-Stream Coordination for Indexer
 * Preprocessing: q_quant = quant(q_proj), w_proj = W_h @ x; "Optimizing LLM
 * Inference for New Architectures", §3), fused into one launch.  For token t:
 *   amax = max |q_proj[t, :, :]|,  scale = amax / 448 (fp32; 1 if amax = 0)
 *   q_codes[t, j, e] = E4M3(q_proj[t, j, e] / scale)  (fp32 division, round to
 *                      nearest even, saturated to ±448)
 *   q_scale[t, j]    = scale for every head j (one scale per token)
 *   w[t, j]          = Σ_c W_h[j, c] · x[t, c]   (fp32 accumulation)
 * These are the FP8 inputs (q_idx, q_scale, w) of dsa_fused_indexer.
 * q_proj  [total_q, h_idx, d_idx] bf16, d_idx a multiple of 8, or NULL (no
 *         quantisation; q_codes and q_scale are then ignored);
 * x       [total_q, d_model] bf16 and w_h [h_idx, d_model] bf16, d_model a
 *         positive multiple of 8, or both NULL (no projection; w ignored);
 * q_codes [total_q, h_idx, d_idx] uint8 (E4M3 codes), q_scale [total_q, h_idx]
 *         f32, w [total_q, h_idx] f32: outputs, caller-owned device memory.
 * q_proj, x, w_h and q_codes are 16-byte aligned; q_scale and w 4-byte.
 * One launch on `stream`, no workspace.  total_q = 0 launches nothing and
 * accepts NULL pointers.
 * DSA_ERR_INVALID_ARG for missing or misaligned pointers (or all inputs NULL),
 * DSA_ERR_UNSUPPORTED for sizes outside those limits.
 */
int dsa_indexer_prolog(int32_t total_q, int32_t h_idx, int32_t d_idx, int32_t d_model,
                       const void* q_proj, const void* x, const void* w_h, uint8_t* q_codes,
                       float* q_scale, float* w, void* stream);

/* Zero the workspace status block (the status word and the kernels' counters; enqueued on
 * `stream`). */
int dsa_clear_status(void* ws, void* stream);

/* Self-test of the bounded-wait path every kernel's waits go through: one thread waits on an
 * mbarrier that nothing arrives at, gives up after limit_ns (0 < limit_ns <= 1e8) and ORs
 * DSA_FLAG_TIMEOUT into the status word of `ws` (enqueued on `stream`; no other effect: the
 * context stays usable).  DSA_ERR_WORKSPACE for a NULL or misaligned `ws`,
 * DSA_ERR_INVALID_ARG for a limit out of range. */
int dsa_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream);

/* Synchronise `stream`, then copy the workspace status word into *flags.
 * Returns DSA_ERR_TIMEOUT if DSA_FLAG_TIMEOUT is set, DSA_OK otherwise. */
int dsa_read_status(const void* ws, void* stream, uint32_t* flags);

/* Message of a dsa_status code (static storage). */
const char* dsa_status_str(int status);

/* Message of the last failing call on this thread ("" if none). */
const char* dsa_last_error(void);

/* DSA_ABI_VERSION of the loaded library. */
int dsa_abi_version(void);

/*
 * Launch tracing.  Between dsa_trace_begin(capacity) and dsa_trace_end(), every
 * kernel the library launches is bracketed by a pair of CUDA events recorded on
 * its stream (at most `capacity` launches are kept).  dsa_trace_get() returns
 * the kernel name and the elapsed milliseconds of launch i (it waits for that
 * launch's end event).  dsa_trace_count() gives the number recorded.
 */
int dsa_trace_begin(int capacity);
int dsa_trace_end(void);
int dsa_trace_count(void);
int dsa_trace_get(int i, char* name, int name_len, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
