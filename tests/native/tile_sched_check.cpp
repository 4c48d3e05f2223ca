// Host check of the indexer's causal work schedule (csrc/tile_sched.cuh) against brute
// force: per-sequence and per-block tile counts in closed form, and the cursor that walks a
// CTA's items (locate at any item, advance item by item), on random problems with ragged
// sequences, tile-less sequences, T = L and T < L.  Prints "ok" or the first mismatch.
#include <cstdio>
#include <random>
#include <vector>

#include "tile_sched.cuh"

using namespace dsa::sched;

struct Item {
  int b, ib, j;
};

// Whole sequences (T0, L0) restricted to the packed query rows [r0, r1): brute force on
// the clipped sequences (T, L, first row q0) against the header's closed forms and cursor.
template <int QB>
static bool check(const std::vector<int>& T0, const std::vector<int>& L0, int r0 = 0,
                  int r1 = 0x7fffffff) {
  const int B = (int)T0.size();
  std::vector<int32_t> st(B + 1), cq(B + 1), ck(B + 1);
  std::vector<int> T(B), L(B), q0(B);
  cq[0] = ck[0] = st[0] = 0;
  for (int b = 0; b < B; ++b) {
    cq[b + 1] = cq[b] + T0[b];
    ck[b + 1] = ck[b] + L0[b];
    // brute-force clip: the rows of sequence b inside [r0, r1), their keys
    int first = -1, cnt = 0;
    for (int r = cq[b]; r < cq[b + 1]; ++r)
      if (r >= r0 && r < r1) { if (first < 0) first = r; ++cnt; }
    T[b] = cnt;
    q0[b] = cnt ? first : 0;
    L[b] = cnt ? L0[b] - T0[b] + (first - cq[b]) + cnt : 0;
  }
  std::vector<Item> items;
  for (int b = 0; b < B; ++b) {
    int64_t n = 0, full = 0;
    const int nfull = T[b] / QB;
    for (int ib = 0; ib * QB < T[b]; ++ib) {
      if (ib <= nfull && block_tiles<QB>(T[b], L[b], ib) != full) {
        std::printf("QB=%d block_tiles(T=%d, L=%d, nb=%d) = %lld, brute %lld\n", QB, T[b], L[b], ib,
                    (long long)block_tiles<QB>(T[b], L[b], ib), (long long)full);
        return false;
      }
      const int i0 = QB * ib, nrow = QB < T[b] - i0 ? QB : T[b] - i0;
      const int pos = L[b] - T[b] + i0;
      const int nt = (pos + nrow - 1) / 128 + 1;  // keys 0 .. pos + nrow - 1
      for (int j = 0; j < nt; ++j) items.push_back({b, ib, j});
      n += nt;
      if (nrow == QB) full += nt;
    }
    if (nfull * QB == T[b] && block_tiles<QB>(T[b], L[b], nfull) != full) {
      std::printf("QB=%d block_tiles(T=%d, L=%d, all) mismatch\n", QB, T[b], L[b]);
      return false;
    }
    if (seq_tiles<QB>(T[b], L[b]) != n) {
      std::printf("QB=%d seq_tiles(T=%d, L=%d) = %lld, brute %lld\n", QB, T[b], L[b],
                  (long long)seq_tiles<QB>(T[b], L[b]), (long long)n);
      return false;
    }
    st[b + 1] = st[b] + (int32_t)n;
  }
  if ((size_t)st[B] != items.size()) return false;
  SeqTab tab{st.data(), cq.data(), ck.data(), B};
  tab.r0 = r0;
  tab.r1 = r1;
  auto same = [&](const Cursor<QB>& c, int g) {
    const Item& it = items[g];
    const int i0 = QB * it.ib;
    return c.b == it.b && c.ib == it.ib && c.j == it.j && c.t == q0[it.b] + i0 &&
           c.pos == L[it.b] - T[it.b] + i0;
  };
  const int total = st[B];
  for (int g = 0; g < total; g += 1 + total / 3000) {
    Cursor<QB> c;
    c.locate(tab, g);
    if (!same(c, g)) {
      std::printf("QB=%d locate(%d) -> (%d, %d, %d), want (%d, %d, %d)\n", QB, g, c.b, c.ib, c.j,
                  items[g].b, items[g].ib, items[g].j);
      return false;
    }
  }
  if (total > 0) {
    Cursor<QB> c;
    c.locate(tab, 0);
    for (int g = 1; g < total; ++g) {
      c.advance(tab);
      if (!same(c, g)) {
        std::printf("QB=%d advance to %d -> (%d, %d, %d), want (%d, %d, %d)\n", QB, g, c.b, c.ib,
                    c.j, items[g].b, items[g].ib, items[g].j);
        return false;
      }
    }
  }
  return true;
}

int main() {
  std::mt19937 rng(12345);
  int cases = 0;
  for (int rep = 0; rep < 300; ++rep) {
    const int B = 1 + (int)(rng() % 9);
    std::vector<int> T(B), L(B);
    for (int b = 0; b < B; ++b) {
      L[b] = 1 + (int)(rng() % (rep % 3 == 0 ? 5000 : 700));
      const int kind = (int)(rng() % 5);
      T[b] = kind == 0 ? 0 : kind == 1 ? L[b] : kind == 2 ? 1 : (int)(rng() % (L[b] + 1));
    }
    if (!check<1>(T, L) || !check<4>(T, L)) return 1;
    // the same problem restricted to a random range of packed query rows
    int tq = 0;
    for (int b = 0; b < B; ++b) tq += T[b];
    const int a = tq ? (int)(rng() % tq) : 0;
    const int e = a + (tq ? (int)(rng() % (tq - a + 1)) : 0);
    if (!check<1>(T, L, a, e) || !check<4>(T, L, a, e)) {
      std::printf("  (rows %d..%d)\n", a, e);
      return 1;
    }
    ++cases;
  }
  // the first and last sequences tile-less, and exact 128 / 4 multiples
  if (!check<1>({0, 128, 0, 256, 0}, {7, 128, 3, 1024, 9}) ||
      !check<4>({0, 128, 0, 256, 0}, {7, 128, 3, 1024, 9}) || !check<4>({3, 5, 4}, {3, 130, 4}))
    return 1;
  std::printf("ok %d\n", cases);
  return 0;
}
