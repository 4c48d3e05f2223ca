// Causal Top-K of materialised score rows, one thread-block cluster per row, for rows
// whose score histogram (top 12 bits of the order-preserving key) was built by the
// tensor-core indexer's epilogue and that fit in 8 segments.
//
// Top-K selection of the Lightning Indexer ("Day0 Inference Adaptation and
// Performance Optimization for New-Architecture LLMs", §4.1): row t keeps the
// n = min(top_k, pos+1) largest of scores[t, 0..pos]; equal scores go to the
// smaller position.
//
// The CTAs of a cluster are the row's segments (1024 threads x KPT keys each).  The
// histogram gives the bin B* that holds the n-th largest key and the count of keys
// above it; every CTA computes both, then reads its keys once and splits them into
// "definite" keys (bins above B*) and "candidates" (bin B*), in position order (block
// prefix sums).  The CTAs swap their two counts through distributed shared memory, so
// each one knows how many definite positions come before its own and writes them
// straight into the output row; their candidates (key, position) go into the first
// CTA's shared memory.  That CTA refines the candidates by exact radix select on the
// low 20 key bits (ties by position) and writes them after the definite ones.  The
// result is the same as the segmented kernel's: all definite positions ascending, then
// the selected candidates ascending.  Cross-CTA transfers are st.async writes counted
// on the receiver's mbarrier; every wait is bounded.
#include "dsa_internal.cuh"
#include "tc_sm100.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kT = 1024;
constexpr int kW = kT / 32;
constexpr int kMaxCluster = 8;
constexpr int kCap = 6144;  // candidates refined in the first CTA's shared memory

template <int KPT>
struct ShC {
  static constexpr int kSeg = KPT * kT;
  uint32_t warp_a[kW], warp_b[kW];
  uint64_t warp_s[kW];
  uint2 counts[kMaxCluster];          // (definite, candidate) count of every segment
  uint32_t hist[2048];
  uint64_t cnt_bar, cand_bar, done_bar;
  uint32_t s_bin, s_above, s_cnt, s_digit, s_ok;
  uint32_t lkey[kSeg];                // this segment's candidates, position order
  int32_t lpos[kSeg];
  uint2 gcand[kCap];                  // first CTA: every segment's (key, position), in order
};

__device__ __forceinline__ void st_async_u2(uint32_t cluster_addr, uint32_t x, uint32_t y,
                                            uint32_t cluster_mbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
          cluster_addr),
      "r"(x), "r"(y), "r"(cluster_mbar)
      : "memory");
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Block-wide exclusive prefix sum of a packed pair (low / high 16 bits).
__device__ __forceinline__ uint32_t scan_pair(uint32_t v, uint32_t* warp_a, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_a[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = warp_a[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_a[lane] = s;
  }
  __syncthreads();
  const uint32_t before = (warp ? warp_a[warp - 1] : 0u) + x - v;
  *total = warp_a[kW - 1];
  __syncthreads();
  return before;
}

// Block-wide exclusive prefix sum of a pair of 32-bit counts (low / high word).
__device__ __forceinline__ uint64_t scan_pair64(uint64_t v, uint64_t* warp_s, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_s[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t z = warp_s[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    __syncwarp();
    warp_s[lane] = z;
  }
  __syncthreads();
  const uint64_t before = (warp ? warp_s[warp - 1] : 0ull) + x - v;
  *total = warp_s[kW - 1];
  __syncthreads();
  return before;
}

// Block-wide count of everything held by higher threads (thread tid holds `mine`, threads
// above it hold larger keys): an exclusive suffix sum.  Two barriers.
__device__ __forceinline__ uint32_t suffix_above(uint32_t mine, uint32_t* warp_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = mine;  // inclusive suffix over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) warp_b[warp] = x;
  __syncthreads();
  if (warp == 0) {  // exclusive suffix over the warp totals
    const uint32_t v = warp_b[lane];
    uint32_t z = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, z, o);
      if (lane + o < 32) z += y;
    }
    __syncwarp();
    warp_b[lane] = z - v;
  }
  __syncthreads();
  return warp_b[warp] + x - mine;
}

// Bin of the n-th largest key, the number of keys in higher bins and in that bin.
template <int KPT>
__device__ __forceinline__ void threshold_bin(const uint32_t* hrow, uint32_t k, ShC<KPT>& S) {
  const int tid = threadIdx.x;
  const uint4 c4 = __ldcg(reinterpret_cast<const uint4*>(hrow) + tid);  // bins 4tid..4tid+3
  const uint32_t mine = c4.x + c4.y + c4.z + c4.w;
  const uint32_t above = suffix_above(mine, S.warp_b);
  if (above < k && above + mine >= k) {
    const uint32_t c[4] = {c4.w, c4.z, c4.y, c4.x};
    uint32_t run = above;
    for (int i = 0; i < 4; ++i) {
      if (run + c[i] >= k) {
        S.s_bin = 4 * tid + 3 - i;
        S.s_above = run;
        S.s_cnt = c[i];
        break;
      }
      run += c[i];
    }
  }
  __syncthreads();
}

// A bounded wait by one thread of the CTA, its outcome shared with the whole CTA.
template <int KPT>
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, ShC<KPT>& S,
                                         volatile int* abort_flag, uint32_t* status) {
  if (threadIdx.x == 0) S.s_ok = mbar_wait(bar, parity, abort_flag, status, DSA_FLAG_TIMEOUT);
  __syncthreads();
  return S.s_ok != 0;
}

template <int KPT>
__global__ void __launch_bounds__(kT, 1) topk_cluster_kernel(TopkArgs a, int csize) {
  constexpr int kSeg = ShC<KPT>::kSeg;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ShC<KPT>& S = *reinterpret_cast<ShC<KPT>*>(smem_raw);
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const uint32_t seg = cluster_ctarank();
  const int t = blockIdx.x / csize;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&S.cnt_bar, 1);
    mbar_init(&S.cand_bar, 1);
    mbar_init(&S.done_bar, 1);
    abort_word = 0;
    fence_barrier_init();
    // every CTA's counts land here (8 bytes each)
    mbar_arrive_expect_tx(&S.cnt_bar, (uint32_t)(8 * csize));
  }
  cluster_sync();  // barriers of every CTA initialised before any remote write

  RowInfo r;
  if (!query_row_info(a.seqs, t, r, a.status)) return;  // the same outcome in every CTA
  const int n = r.pos + 1;
  const int k = min(a.top_k, n);
  const int s0 = (int)seg * kSeg;
  griddep_wait();                  // the scores and histograms are complete
  if (tid == 0) griddep_launch();  // the attention kernel may be scheduled (it waits)
  const float* row = a.scores + (int64_t)t * a.ld;
  int32_t* irow = a.idx + (int64_t)t * a.top_k;
  float* vrow = a.vals ? a.vals + (int64_t)t * a.top_k : nullptr;

  if (k == n) {  // the whole history is kept (the same branch in every CTA; no remote access)
    for (int i = s0 + tid; i < min(n, s0 + kSeg); i += kT) {
      irow[i] = i;
      if (vrow) vrow[i] = row[i];
    }
    if (seg == 0)
      for (int j = n + tid; j < a.top_k; j += kT) {
        irow[j] = -1;
        if (vrow) vrow[j] = -INFINITY;
      }
    return;
  }

  // ---- this segment's keys: definite ones and candidates ----
  const int i0 = s0 + KPT * tid;  // this thread's KPT consecutive keys
  float f[KPT];
#pragma unroll
  for (int q = 0; q < KPT / 4; ++q) {
    const int i = i0 + 4 * q;
    if (i + 3 < n) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(row + i));
      f[4 * q] = v.x; f[4 * q + 1] = v.y; f[4 * q + 2] = v.z; f[4 * q + 3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) f[4 * q + e] = i + e < n ? row[i + e] : 0.f;
    }
  }
  threshold_bin(a.hist + (int64_t)t * kHistBins, (uint32_t)k, S);
  const uint32_t bstar = S.s_bin, above = S.s_above, nc = S.s_cnt;
  uint32_t dm = 0, cm = 0;  // KPT-bit masks
  uint32_t key[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    key[j] = order_key(f[j]);
    if (i0 + j < n) {
      const uint32_t b = key[j] >> 20;
      if (b > bstar) dm |= 1u << j;
      else if (b == bstar) cm |= 1u << j;
    }
  }
  uint32_t tot;
  const uint32_t pre = scan_pair((uint32_t)__popc(dm) | ((uint32_t)__popc(cm) << 16), S.warp_a, &tot);
  const uint32_t td = tot & 0xffffu, tcn = tot >> 16;
  {
    uint32_t pc = pre >> 16;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (cm >> j & 1u) { S.lkey[pc] = key[j]; S.lpos[pc] = i0 + j; ++pc; }
  }
  // our two counts to every CTA of the cluster (thread i writes to CTA i)
  if (tid < csize) {
    const uint32_t dst = mapa(smem_u32(&S.counts[seg]), (uint32_t)tid);
    st_async_u2(dst, td, tcn, mapa(smem_u32(&S.cnt_bar), (uint32_t)tid));
  }
  __syncthreads();  // local candidates written
  // the leader expects every candidate of the row
  const bool fast = nc <= (uint32_t)kCap;
  if (seg == 0 && tid == 0 && fast) mbar_arrive_expect_tx(&S.cand_bar, nc * 8u);
  if (!cta_wait(&S.cnt_bar, 0, S, abort_flag, a.status)) return;
  uint32_t def_off = 0, cand_off = 0, nc_sum = 0, def_sum = 0;
  for (int s = 0; s < csize; ++s) {
    const uint2 c = S.counts[s];
    if (s < (int)seg) { def_off += c.x; cand_off += c.y; }
    def_sum += c.x;
    nc_sum += c.y;
  }
  if (nc_sum != nc || def_sum != above) {  // histogram and scores disagree
    if (tid == 0) atomicOr(a.status, DSA_FLAG_BAD_SEQS);
    // keep the protocol going so that no CTA waits in vain
  }

  // definite positions, straight into the output row (segments in order)
  {
    uint32_t pd = def_off + (pre & 0xffffu);
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (dm >> j & 1u) {
        if (pd < (uint32_t)k) {
          irow[pd] = i0 + j;
          if (vrow) vrow[pd] = f[j];
        }
        ++pd;
      }
  }
  // candidates into the first CTA's shared memory
  if (fast) {
    const uint32_t gc = mapa(smem_u32(S.gcand), 0u);
    const uint32_t bar = mapa(smem_u32(&S.cand_bar), 0u);
    for (uint32_t j = tid; j < tcn; j += kT) {
      const uint32_t c = cand_off + j;
      if (c < (uint32_t)kCap) st_async_u2(gc + 8 * c, S.lkey[j], (uint32_t)S.lpos[j], bar);
    }
  }
  if (seg != 0) {
    // stay until the first CTA no longer needs this CTA's shared memory
    cta_wait(&S.done_bar, 0, S, abort_flag, a.status);
    return;
  }

  // ---- the first CTA: refine the candidates, write them, release the others ----
  auto release = [&]() {
    if (tid >= 1 && tid < csize) mbar_arrive_remote(mapa(smem_u32(&S.done_bar), (uint32_t)tid));
  };
  if (fast && !cta_wait(&S.cand_bar, 0, S, abort_flag, a.status)) { release(); return; }
  // candidate c: from shared memory, or (slow path) from its segment's CTA
  auto seg_of = [&](uint32_t c, uint32_t& local) -> int {
    int s = 0;
    uint32_t base = 0;
    while (s + 1 < csize && base + S.counts[s].y <= c) { base += S.counts[s].y; ++s; }
    local = c - base;
    return s;
  };
  auto cand_key = [&](uint32_t c) -> uint32_t {
    if (fast) return S.gcand[c].x;
    uint32_t l;
    const int s = seg_of(c, l);
    return ld_cluster_u32(mapa(smem_u32(&S.lkey[l]), (uint32_t)s));
  };
  auto cand_pos = [&](uint32_t c) -> int32_t {
    if (fast) return (int32_t)S.gcand[c].y;
    uint32_t l;
    const int s = seg_of(c, l);
    return (int32_t)ld_cluster_u32(mapa(smem_u32(&S.lpos[l]), (uint32_t)s));
  };

  // exact radix select among the candidates on the low 20 bits (11 + 9); thread tid
  // takes the candidates [tid * cpt, (tid + 1) * cpt), in position order
  const uint32_t cpt = (nc + kT - 1) / kT;
  const uint32_t c_lo = min(nc, tid * cpt), c_hi = min(nc, c_lo + cpt);
  uint32_t prefix = bstar << 20, need = (uint32_t)k - above;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 9 : 0;
    const uint32_t bits = pass == 0 ? 11u : 9u;
    const uint32_t dmask = (1u << bits) - 1u;
    const uint32_t pmask = pass == 0 ? 0xfff00000u : 0xfffffe00u;
    S.hist[2 * tid] = 0u;
    S.hist[2 * tid + 1] = 0u;
    __syncthreads();
    for (uint32_t c = c_lo; c < c_hi; ++c) {
      const uint32_t kk = cand_key(c);
      if ((kk & pmask) == prefix) atomicAdd(&S.hist[(kk >> shift) & dmask], 1u);
    }
    __syncthreads();
    // digit d (descending) where the need-th key falls: thread tid owns bins 2tid+1, 2tid
    const uint32_t h1 = S.hist[tid * 2 + 1], h0 = S.hist[tid * 2];
    const uint32_t mine = h0 + h1;
    const uint32_t ab = suffix_above(mine, S.warp_b);
    if (ab < need && ab + mine >= need) {
      if (ab + h1 >= need) { S.s_digit = tid * 2 + 1; S.s_cnt = ab; }
      else { S.s_digit = tid * 2; S.s_cnt = ab + h1; }
    }
    __syncthreads();
    need -= S.s_cnt;
    prefix |= S.s_digit << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // exact key of the n-th largest; `need` of the ties are kept

  // selected candidates, in position order, after the definite ones
  {
    uint32_t ng = 0, ne = 0;
    for (uint32_t c = c_lo; c < c_hi; ++c) {
      const uint32_t kk = cand_key(c);
      ng += kk > T;
      ne += kk == T;
    }
    uint64_t ttot;
    const uint64_t pr = scan_pair64((uint64_t)ng | ((uint64_t)ne << 32), S.warp_s, &ttot);
    uint32_t gb = (uint32_t)pr, eb = (uint32_t)(pr >> 32);
    for (uint32_t c = c_lo; c < c_hi; ++c) {
      const uint32_t kk = cand_key(c);
      int slot = -1;
      if (kk > T) { slot = (int)(above + gb + min(eb, need)); ++gb; }
      else if (kk == T) { if (eb < need) slot = (int)(above + gb + eb); ++eb; }
      if (slot >= 0 && slot < k) {
        irow[slot] = cand_pos(c);
        if (vrow) vrow[slot] = key_to_float(kk);
      }
    }
  }
  __syncthreads();
  release();
}

template <int KPT>
int launch(const TopkArgs& a, int csize, cudaStream_t stream) {
  const size_t smem = sizeof(ShC<KPT>);
  auto kern = topk_cluster_kernel<KPT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("topk_cluster: smem attribute");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(csize * a.seqs.total_q));
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaSuccess;
  DSA_LAUNCH("topk_cluster", stream, e = cudaLaunchKernelEx(&cfg, kern, a, csize));
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "topk_cluster: %s", cudaGetErrorString(e));
  return check_launch("topk_cluster");
}

}  // namespace

int topk_cluster_size(int max_k_len) {
  if (max_k_len <= kMaxCluster * 8 * kT) return (max_k_len + 8 * kT - 1) / (8 * kT);
  return (max_k_len + 16 * kT - 1) / (16 * kT);
}

// Few rows: when all clusters fit on the GPU at once, spreading a row over up to 8 SMs
// shortens the (latency-bound) step; beyond one wave the streaming kernel, one CTA per
// row and several rows per SM, does more work per SM and wins.
bool topk_cluster_eligible(const TopkArgs& a) {
  return a.hist != nullptr && a.seqs.max_k_len <= kMaxCluster * 16 * kT &&
         (int64_t)a.seqs.total_q * topk_cluster_size(a.seqs.max_k_len) <= num_sms();
}

int launch_topk_cluster(const TopkArgs& a, cudaStream_t stream) {
  if (a.seqs.total_q == 0) return DSA_OK;
  const int csize = topk_cluster_size(a.seqs.max_k_len);
  if (a.seqs.max_k_len <= kMaxCluster * 8 * kT) return launch<8>(a, csize, stream);
  return launch<16>(a, csize, stream);
}

}  // namespace dsa
