// The indexer's causal work schedule, shared by the kernel and a host-side check.
//
// Work item = (block of QB query rows of one sequence, 128-key tile); a block whose last
// row sits at position p has floor(p/128) + 1 tiles.  The items of all blocks are laid end
// to end (sequence by sequence, block by block, tile by tile) and each persistent CTA takes
// one contiguous, equal share.  Tile counts come in closed form:
//   QB = 1: per sequence F(L) - F(L - T), F(n) = Σ_{p<n} (floor(p/128) + 1)
//           = n + 64 q (q - 1) + r q  (q = n / 128, r = n % 128);
//   QB = 4: the first nb full blocks hold nb + G(a + nb) - G(a) tiles, a = (L - T + 3) / 4,
//           G(n) = Σ_{x<n} floor(x/32); a partial last block holds floor((L-1)/128) + 1.
// ("Day0 Inference Adaptation and Performance Optimization for New-Architecture LLMs" §6.2:
// index computation is causal, so later rows see longer histories and the work skews.)
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define DSA_HD_INLINE __host__ __device__ __forceinline__
#else
#define DSA_HD_INLINE inline
#endif

#ifndef INT64_MAX
#define INT64_MAX 9223372036854775807LL
#endif

namespace dsa {
namespace sched {

DSA_HD_INLINE int64_t ftiles(int64_t n) {  // Σ_{p<n} (floor(p/128) + 1)
  const int64_t q = n >> 7, r = n & 127;
  return n + 64 * q * (q - 1) + r * q;
}

// Σ_{x<n} floor(x / D)
DSA_HD_INLINE int64_t gsum(int64_t n, int64_t D) {
  const int64_t q = n / D, r = n % D;
  return D * q * (q - 1) / 2 + r * q;
}

// Tiles of the first nb blocks of a sequence with T queries over L keys (nb <= full blocks).
template <int QB>
DSA_HD_INLINE int64_t block_tiles(int T, int L, int nb) {
  if (QB == 1) return ftiles(L - T + nb) - ftiles(L - T);
  const int64_t a = (L - T + QB - 1) / QB;
  return nb + gsum(a + nb, 128 / QB) - gsum(a, 128 / QB);
}

// All tiles of a sequence.
template <int QB>
DSA_HD_INLINE int64_t seq_tiles(int T, int L) {
  if (QB == 1) return ftiles(L) - ftiles(L - T);
  const int nfull = T / QB;
  return block_tiles<QB>(T, L, nfull) + (T % QB ? (L - 1) / 128 + 1 : 0);
}

// A sequence's queries restricted to the packed rows [r0, r1): the rows it keeps are
// [q0, q0 + T) and, being the last T of the first L keys' positions, they sit where they
// sat in the whole sequence (the keys after the last kept row are simply not visible).
// T = 0 when the sequence has no row in the range.
DSA_HD_INLINE void clip_seq(int qa, int qe, int ka, int ke, int r0, int r1, int& q0, int& T,
                            int& L) {
  const int a = qa > r0 ? qa : r0, e = qe < r1 ? qe : r1;
  q0 = a;
  T = e > a ? e - a : 0;
  L = T > 0 ? (ke - ka) - (qe - qa) + (e - qa) : 0;
}

// Per-sequence tile table built in shared memory by every CTA.
struct SeqTab {
  const int32_t* st;  // [B+1] first tile of each sequence, then the total
  const int32_t* cq;  // [B+1] cu_q
  const int32_t* ck;  // [B+1] cu_k
  int B;
  int r0 = 0, r1 = 0x7fffffff;  // the packed query rows scored (all by default)
};

// Walks the CTA's items (block tile by block tile) in order; all roles run one.
template <int QB>
struct Cursor {
  int b, ib, T, L, q0, k0;   // sequence, block index in it, its sizes and offsets
  int t, pos, nrow, j, ntiles;  // first packed row of the block, its position, rows, tile

  DSA_HD_INLINE void load_seq(const SeqTab& s) {
    clip_seq(s.cq[b], s.cq[b + 1], s.ck[b], s.ck[b + 1], s.r0, s.r1, q0, T, L);
    k0 = s.ck[b];
  }
  DSA_HD_INLINE void set_block() {
    const int i0 = QB * ib;
    t = q0 + i0;
    pos = L - T + i0;
    nrow = QB < T - i0 ? QB : T - i0;
    ntiles = (pos + nrow - 1) / 128 + 1;
  }
  DSA_HD_INLINE void locate(const SeqTab& s, int g) {
    int lo = 0, hi = s.B - 1;  // last b with st[b] <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.st[mid] <= g) lo = mid; else hi = mid - 1;
    }
    b = lo;
    load_seq(s);
    const int64_t gl = g - s.st[b];
    const int nfull = T / QB, nblk = (T + QB - 1) / QB;
    int ilo = 0, ihi = nblk - 1;  // last block whose first tile is <= gl
    while (ilo < ihi) {
      const int mid = (ilo + ihi + 1) >> 1;
      const int64_t before = mid <= nfull ? block_tiles<QB>(T, L, mid) : INT64_MAX;
      if (before <= gl) ilo = mid; else ihi = mid - 1;
    }
    ib = ilo;
    set_block();
    j = (int)(gl - block_tiles<QB>(T, L, ib < nfull ? ib : nfull));
  }
  DSA_HD_INLINE void advance(const SeqTab& s) {
    if (++j < ntiles) return;
    j = 0;
    if (++ib * QB >= T) {
      ib = 0;
      do { ++b; } while (b < s.B - 1 && s.st[b + 1] == s.st[b]);  // skip tile-less sequences
      load_seq(s);
    }
    set_block();
  }
};

}  // namespace sched
}  // namespace dsa
