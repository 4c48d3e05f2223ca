// Causal Top-K of a score row held entirely in shared memory (rows up to
// 40,960 keys): one CTA per query row.
//
// Top-K selection of the Lightning Indexer ("Day0 Inference Adaptation and
// Performance Optimization for New-Architecture LLMs", §4.1), with the same
// contract as topk_rows.cu: the n = min(top_k, pos+1) largest scores, ties to
// the smaller position, written in ascending position order, -1 padded.
// 1024 threads per row; every pass over the keys is warp-coalesced.
//
// When the indexer has also left a histogram of the row's scores by their top
// 12 key bits, the threshold bin comes straight from it and only that bin's keys
// are refined.  Otherwise:
// The row is read once from global memory into shared memory as
// order-preserving uint32 keys, with its min and max.  The radix select runs on
// the offsets v = key - min, whose top 8 significant bits already spread the
// row over up to 256 bins (on raw keys the first digit would be the float
// exponent, shared by almost every score), with per-warp histograms to keep
// shared-memory atomics uncontended.  Once the keys still in play fit a small buffer they
// are compacted and later digits scan only them.  A single block-wide prefix
// sum then places every selected position: each thread owns a contiguous run
// of keys, read in a lane-rotated order so the 32 lanes never share a bank.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kT = 1024;
constexpr int kW = kT / 32;
constexpr int kMaxKeys = 40960;
constexpr int kCandCap = 4096;
constexpr size_t kSmem = sizeof(uint32_t) * ((size_t)kMaxKeys + kW * 256 + 256 + kCandCap);

static_assert(kT * 4 == kHistBins, "one uint4 of histogram bins per thread");

__global__ void __launch_bounds__(kT, 1) topk_smem_kernel(TopkArgs a) {
  extern __shared__ uint32_t sm[];
  uint32_t* keys = sm;                  // [kMaxKeys]
  uint32_t* hist = keys + kMaxKeys;     // [kW][256]
  uint32_t* tot = hist + kW * 256;      // [256]
  uint32_t* cand = tot + 256;           // [kCandCap]
  __shared__ uint32_t red_min[kW], red_max[kW];
  __shared__ uint32_t s_digit, s_above, s_cnt, s_ncand;

  const int t = a.row0 + blockIdx.x;  // query row; its scores are row blockIdx.x
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;
  const float* row = a.scores + (int64_t)blockIdx.x * a.ld;
  const int n = r.pos + 1;
  const int k = min(a.top_k, n);
  int32_t* idx = a.idx + (int64_t)t * a.top_k;
  float* vals = a.vals ? a.vals + (int64_t)t * a.top_k : nullptr;
  for (int j = k + tid; j < a.top_k; j += kT) {
    idx[j] = -1;
    if (vals) vals[j] = -INFINITY;
  }
  // Histogram of this row's keys by their top 12 bits (filled by the indexer).
  uint32_t hb_bin = 0, hb_above = 0, hb_cnt = 0;
  const bool use_hist = a.hist != nullptr;
  if (use_hist) {
    const uint4* hrow = reinterpret_cast<const uint4*>(a.hist + (int64_t)blockIdx.x * kHistBins);
    const uint4 c4 = __ldcg(hrow + tid);  // bins 4*tid .. 4*tid+3
    if (k < n) {
      // keys in bins above this thread's: exclusive scan in descending bin order
      const uint32_t mine = c4.x + c4.y + c4.z + c4.w;
      uint32_t x = mine;
      // reverse: warp w' = kW-1-warp, lane' = 31-lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
      }
      if (lane == 0) red_min[warp] = x;  // warp total
      __syncthreads();
      uint32_t above = x - mine;         // within the warp, bins of higher lanes
      for (int w = warp + 1; w < kW; ++w) above += red_min[w];
      if (above < (uint32_t)k && above + mine >= (uint32_t)k) {
        const uint32_t c[4] = {c4.w, c4.z, c4.y, c4.x};  // descending bins
        uint32_t run = above;
        for (int i = 0; i < 4; ++i) {
          if (run + c[i] >= (uint32_t)k) {
            s_digit = 4 * tid + 3 - i;
            s_above = run;
            s_cnt = c[i];
            break;
          }
          run += c[i];
        }
      }
      if (tid == 0) s_ncand = 0;
      __syncthreads();
      hb_bin = s_digit; hb_above = s_above; hb_cnt = s_cnt;
    }
  }
  if (k == n) {
    for (int i = tid; i < n; i += kT) {
      idx[i] = i;
      if (vals) vals[i] = row[i];
    }
    return;
  }
  const bool hist_cand = use_hist && hb_cnt <= (uint32_t)kCandCap;

  // --- load the row as keys, with its min and max ----------------------------
  // Vector loads, several in flight per thread (the row usually sits in L2).
  uint32_t lmin = 0xffffffffu, lmax = 0u;
  int head = (int)(((16u - ((uintptr_t)row & 15u)) & 15u) >> 2);  // scalars before 16-B alignment
  if (((uintptr_t)row & 3u) != 0) head = n;                          // not even 4-B aligned
  head = min(head, n);
  for (int i = tid; i < head; i += kT) {
    const uint32_t key = order_key(row[i]);
    keys[i] = key;
    lmin = min(lmin, key);
    lmax = max(lmax, key);
  }
  const int nvec = (n - head) >> 2;
  const float4* rv = reinterpret_cast<const float4*>(row + head);
#pragma unroll 4
  for (int v = tid; v < nvec; v += kT) {
    const float4 f = __ldcg(rv + v);
    const int i = head + 4 * v;
    const uint32_t k0 = order_key(f.x), k1 = order_key(f.y), k2 = order_key(f.z),
                   k3 = order_key(f.w);
    keys[i] = k0; keys[i + 1] = k1; keys[i + 2] = k2; keys[i + 3] = k3;
    lmin = min(min(lmin, min(k0, k1)), min(k2, k3));
    lmax = max(max(lmax, max(k0, k1)), max(k2, k3));
  }
  for (int i = head + 4 * nvec + tid; i < n; i += kT) {
    const uint32_t key = order_key(row[i]);
    keys[i] = key;
    lmin = min(lmin, key);
    lmax = max(lmax, key);
  }
  lmin = __reduce_min_sync(0xffffffffu, lmin);
  lmax = __reduce_max_sync(0xffffffffu, lmax);
  __syncthreads();  // (red_min was used by the histogram scan)
  if (lane == 0) { red_min[warp] = lmin; red_max[warp] = lmax; }
  __syncthreads();
  uint32_t kmin = red_min[0], kmax = red_max[0];
  for (int w = 1; w < kW; ++w) { kmin = min(kmin, red_min[w]); kmax = max(kmax, red_max[w]); }

  // --- radix select of the exact n-th largest key -------------------------------
  // Without a histogram: on offsets v = key - kmin in [0, kmax - kmin], T = kmin +
  // (selected offset).  With one: the top 12 bits are already fixed by the threshold
  // bin, and only the keys of that bin (compacted here when they fit) are searched.
  uint32_t prefix, need, mask;
  int hb;
  const uint32_t* src = keys;
  int src_n = n;
  bool compacted = false, done = false;
  if (use_hist) {
    kmin = 0u;
    prefix = hb_bin << 20;
    mask = 0xfff00000u;
    need = (uint32_t)k - hb_above;
    hb = 19;
    if (hist_cand) {
      for (int i0 = 0; i0 < n; i0 += kT) {
        const int i = i0 + tid;
        const uint32_t key = i < n ? keys[i] : 0u;
        const bool hitk = i < n && (key & mask) == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, hitk);
        uint32_t wbase = 0;
        if (lane == 0 && bal) wbase = atomicAdd(&s_ncand, (uint32_t)__popc(bal));
        wbase = __shfl_sync(0xffffffffu, wbase, 0);
        if (hitk) cand[wbase + __popc(bal & ((1u << lane) - 1u))] = key;
      }
      __syncthreads();
      src = cand;
      src_n = (int)s_ncand;
      compacted = true;
    }
  } else {
    prefix = kmax - kmin;
    need = (uint32_t)k;
    mask = 0u;
    hb = 0;
    done = kmin == kmax;
    if (!done) {
      hb = 31 - __clz(kmax - kmin);                  // highest bit any offset uses
      mask = hb == 31 ? 0u : ~((2u << hb) - 1u);     // bits zero in every offset
      prefix = 0u;
    }
  }
  if (!done) {
    while (true) {
      const int shift = hb >= 7 ? hb - 7 : 0;
      const int nb = hb - shift + 1;
      const uint32_t dmask = (nb == 32) ? 0xffffffffu : ((1u << nb) - 1u);
      for (int i = tid; i < kW * 256; i += kT) hist[i] = 0;
      __syncthreads();
      uint32_t* h = hist + warp * 256;
      for (int i = tid; i < src_n; i += kT) {
        const uint32_t v = src[i] - kmin;
        if ((v & mask) == prefix) atomicAdd(&h[(v >> shift) & dmask], 1u);
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t c = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) c += hist[w * 256 + tid];
        tot[tid] = c;
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) { c[i] = tot[255 - 8 * lane - i]; sum += c[i]; }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - sum;
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= need && excl < need);
        if (hit && lane == __ffs(hit) - 1) {
          uint32_t run = excl;
          for (int i = 0; i < 8; ++i) {
            if (run + c[i] >= need) {
              s_digit = 255 - 8 * lane - i;
              s_above = run;
              s_cnt = c[i];
              break;
            }
            run += c[i];
          }
        }
      }
      __syncthreads();
      need -= s_above;
      prefix |= s_digit << shift;
      mask |= dmask << shift;
      const uint32_t cnt = s_cnt;
      if (shift == 0) break;
      hb = shift - 1;
      if (!compacted && cnt <= (uint32_t)kCandCap) {
        __syncthreads();
        if (tid == 0) s_ncand = 0;
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += kT) {  // one counter update per warp
          const int i = i0 + tid;
          const uint32_t key = i < n ? keys[i] : 0u;
          const bool hitk = i < n && ((key - kmin) & mask) == prefix;
          const unsigned bal = __ballot_sync(0xffffffffu, hitk);
          uint32_t wbase = 0;
          if (lane == 0 && bal) wbase = atomicAdd(&s_ncand, (uint32_t)__popc(bal));
          wbase = __shfl_sync(0xffffffffu, wbase, 0);
          if (hitk) cand[wbase + __popc(bal & ((1u << lane) - 1u))] = key;
        }
        __syncthreads();
        src = cand;
        src_n = (int)s_ncand;
        compacted = true;
      }
    }
  }
  const uint32_t T = kmin + prefix;  // the n-th largest key; `need` of the keys equal to it are kept

  // --- ordered write -------------------------------------------------------------------
  // Warp w owns the contiguous key range [w*seg, (w+1)*seg).  Pass A counts its keys
  // above / equal to T with ballots; a scan over the 16 warp totals gives each warp
  // its offsets; pass B places every selected key (ballot ranks within the warp).
  const int seg = ((n + kW - 1) / kW + 31) / 32 * 32;
  const int w0 = warp * seg, w1 = min(n, w0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  uint32_t cg = 0, ce = 0;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    cg += __popc(__ballot_sync(0xffffffffu, i < w1 && key > T));
    ce += __popc(__ballot_sync(0xffffffffu, i < w1 && key == T));
  }
  __shared__ uint32_t w_gt[kW], w_eq[kW];
  if (lane == 0) { w_gt[warp] = cg; w_eq[warp] = ce; }
  __syncthreads();
  uint32_t G = 0, E = 0;
  for (int w = 0; w < warp; ++w) { G += w_gt[w]; E += w_eq[w]; }
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < w1 ? keys[i] : 0u;
    const bool gt = i < w1 && key > T, eq = i < w1 && key == T;
    const unsigned bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    const uint32_t gb = G + __popc(bg & lt), eb = E + __popc(be & lt);
    int slot = -1;
    if (gt) slot = (int)(gb + min(eb, need));
    else if (eq && eb < need) slot = (int)(gb + eb);
    if (slot >= 0) {
      idx[slot] = i;
      if (vals) vals[slot] = key_to_float(key);
    }
    G += __popc(bg);
    E += __popc(be);
  }
}

__global__ void mask_tail_kernel(Seqs seqs, float* scores, int64_t ld, uint32_t* status) {
  RowInfo r;
  const int t = blockIdx.x;
  if (!query_row_info(seqs, t, r, status)) return;
  float* row = scores + (int64_t)t * ld;
  for (int64_t s = r.pos + 1 + threadIdx.x; s < ld; s += blockDim.x) row[s] = -INFINITY;
}

}  // namespace

int topk_smem_max_keys() { return kMaxKeys; }

int launch_topk_smem(const TopkArgs& a, cudaStream_t stream) {
  if (a.rows() <= 0) return DSA_OK;
  if (cudaFuncSetAttribute(topk_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmem) != cudaSuccess)
    return check_launch("topk_smem: smem attribute");
  DSA_LAUNCH("topk_smem", stream, topk_smem_kernel<<<a.rows(), kT, kSmem, stream>>>(a));
  return check_launch("topk_smem");
}

int launch_mask_tail(const Seqs& seqs, float* scores, int64_t ld, uint32_t* status,
                     cudaStream_t stream) {
  if (seqs.total_q == 0) return DSA_OK;
  DSA_LAUNCH("mask_tail", stream,
             mask_tail_kernel<<<seqs.total_q, 256, 0, stream>>>(seqs, scores, ld, status));
  return check_launch("mask_tail");
}

}  // namespace dsa
