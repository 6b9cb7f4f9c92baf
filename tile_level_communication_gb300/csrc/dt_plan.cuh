// Rank-aware tile order (the distributed swizzle) as stateless position functions that run
// on the host and on the device.
//
// DITRON page, section 3.2 (论文 §3.2, Fig. 3): swizzle_func maps the original tile id to a
// new one with a rank-aware offset; rank r starts at r mod world_size.  Gather mode (AllGather
// GEMM) treats local HBM as a cache of remote memory: own rows first, remote chunks in the
// order they are fetched.  Scatter mode (GEMM ReduceScatter) computes first the rows that go
// to the farthest rank; here rank q sends to q+1 first and keeps its own block for last.
// Triton-distributed talk, "不完全なブロックスケジューリング": a tile that straddles ranks runs
// after the data it waits for (AllGather) or before the tiles other ranks do not need
// (ReduceScatter).  AutoOverlap page, section 5.4 / Fig. 6: across chunks the schedule follows
// chunk arrival, inside a chunk bands of G m-tiles are swept column by column for locality.
//
// Definition (the same one the oracle sorts by):
//   chunk (s, j) = rows [s*Ms + j*Cr, s*Ms + min((j+1)*Cr, Ms)),  nC = ceil(Ms / Cr)
//   AG: pos(s, j) = ((s - r) mod W) * nC + j;  key(i) = max pos of the chunks m-tile i reads;
//       order = sort (i, n) by (n / Nb, key(i), band(i), n, i): column bands of Nb tiles one
//       after another, each repeating the gather order (Nb = Tn: one band)
//   RS: dpos_q(s) = (s - q - 1) mod W;  key(q, i) = min over written chunks of dpos*nC + j;
//       order = sort (q, i, n) by (q, n / Nb, key, band, n, i): the virtual source ranks one
//       after another, each in its own scatter order, so every destination receives its
//       partials in source order q = 0 .. W-1; inside a rank's pass the column tiles go in
//       bands of Nb, each band repeating the scatter order over every destination, so only
//       one band of B_q is in use at a time (Nb = Tn: one band)
//   A2A (GEMM-AllToAll, rows local to each rank, columns split by destination h):
//       key(q, i, h) = dpos_q(h)*nC + (first chunk of m-tile i);
//       order = sort (q, i, h, c) by (q, key, band, c, i): the virtual source ranks one after
//       another, each in its own scatter order (each output is one product, so nothing but
//       L2 reuse depends on how they interleave: one rank's A_q and B columns stay in L2)
// Evaluation here does not sort.  Along the m-tiles rotated to start at the first m-tile of
// the own rank (AG) or of rank q+1 (RS) the key never decreases, so the key of an m-tile is
// read off one row of it, and the number of m-tiles with a smaller key is a binary search.
// A tile's position is then a closed expression of those counts.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DT_HD __host__ __device__ __forceinline__
#else
#define DT_HD inline
#endif

namespace dt {

struct Geom {
  int64_t M, N, Ms, Cr;
  int32_t W, rank, BM, BN, nC, Tm, Tn, G, swizzle;
  int64_t Nw;   // AllToAll: columns per destination (N / W); 0 otherwise
  int32_t Tnw;  // AllToAll: column tiles per destination; 0 otherwise
  int32_t Nb;   // AllGather / ReduceScatter: column tiles per column band (Tn: one band)
};

DT_HD int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
DT_HD int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
DT_HD int32_t min32(int32_t a, int32_t b) { return a < b ? a : b; }

DT_HD Geom make_geom(int32_t W, int32_t rank, int64_t M, int64_t N, int64_t Cr, int32_t BM,
                     int32_t BN, int32_t G, int32_t swizzle) {
  Geom g;
  g.M = M;
  g.N = N;
  g.W = W;
  g.rank = rank;
  g.Ms = M / W;
  g.Cr = Cr;
  g.BM = BM;
  g.BN = BN;
  g.G = G;
  g.swizzle = swizzle;
  g.nC = g.Ms > 0 ? static_cast<int32_t>(cdiv64(g.Ms, Cr)) : 0;
  g.Tm = static_cast<int32_t>(cdiv64(M, BM));
  g.Tn = static_cast<int32_t>(cdiv64(N, BN));
  g.Nw = 0;
  g.Tnw = 0;
  g.Nb = g.Tn;
  return g;
}

// GEMM-AllToAll: every rank's Ms rows are tiled on their own (Tm m-tiles per rank) and the N
// columns block by block, one block of Nw = N / W per destination (Tnw column tiles each).
DT_HD Geom make_geom_a2a(int32_t W, int64_t M, int64_t N, int64_t Cr, int32_t BM, int32_t BN,
                         int32_t G, int32_t swizzle) {
  Geom g = make_geom(W, 0, M, N, Cr, BM, BN, G, swizzle);
  g.Nw = N / W;
  g.Tm = static_cast<int32_t>(cdiv64(g.Ms, BM));
  g.Tnw = static_cast<int32_t>(cdiv64(g.Nw, BN));
  g.Tn = W * g.Tnw;
  g.Nb = g.Tn;
  return g;
}

// rank s and chunk j of global row `row`
DT_HD void row_chunk(const Geom& g, int64_t row, int32_t& s, int32_t& j) {
  s = static_cast<int32_t>(row / g.Ms);
  j = static_cast<int32_t>((row - static_cast<int64_t>(s) * g.Ms) / g.Cr);
}

// Offset of tile (u, n) inside its key group [ug, ue) of rotated m-tile indices: bands of
// G m-tiles, each swept column by column.
DT_HD int64_t band_offset(int32_t ug, int32_t ue, int32_t u, int32_t n, int32_t Tn, int32_t G) {
  const int32_t b = (u - ug) / G;
  const int32_t bs = ug + b * G;
  const int32_t bsz = min32(G, ue - bs);
  return static_cast<int64_t>(b) * G * Tn + static_cast<int64_t>(n) * bsz + (u - bs);
}

// ------------------------------------------------------------------ gather mode (AllGather)
DT_HD int32_t ag_chunk_pos(const Geom& g, int32_t s, int32_t j) {
  return ((s - g.rank + g.W) % g.W) * g.nC + j;
}
// first m-tile that lies wholly at or after the own rank's first row
DT_HD int32_t ag_rot0(const Geom& g) {
  return static_cast<int32_t>(cdiv64(static_cast<int64_t>(g.rank) * g.Ms, g.BM) % g.Tm);
}
// key of the m-tile at rotated index u
DT_HD int32_t ag_key(const Geom& g, int32_t rot0, int32_t u) {
  const int32_t i = (rot0 + u) % g.Tm;
  const int64_t first = static_cast<int64_t>(i) * g.BM;
  const int64_t last = min64(first + g.BM, g.M) - 1;
  const int64_t own0 = static_cast<int64_t>(g.rank) * g.Ms;
  // reads the last chunk of rank r-1: the latest chunk of the gather
  if (g.rank > 0 && first < own0 && last >= own0) return g.W * g.nC - 1;
  int32_t s, j;
  row_chunk(g, last, s, j);
  return ag_chunk_pos(g, s, j);
}
DT_HD int32_t ag_count_below(const Geom& g, int32_t rot0, int32_t k) {
  int32_t lo = 0, hi = g.Tm;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (ag_key(g, rot0, mid) < k) lo = mid + 1; else hi = mid;
  }
  return lo;
}
// execution position of AllGather tile (i, n): the full column bands before n's (Tm*Nb each),
// then n's band (nbw columns wide) laid out like a band-less order over those columns
DT_HD int64_t ag_position(const Geom& g, int32_t i, int32_t n) {
  if (!g.swizzle) return static_cast<int64_t>(i) * g.Tn + n;
  const int32_t rot0 = ag_rot0(g);
  const int32_t u = (i - rot0 + g.Tm) % g.Tm;
  const int32_t k = ag_key(g, rot0, u);
  const int32_t ug = ag_count_below(g, rot0, k);
  const int32_t ue = ag_count_below(g, rot0, k + 1);
  const int32_t b = n / g.Nb;
  const int32_t nbw = min32(g.Nb, g.Tn - b * g.Nb);
  return static_cast<int64_t>(b) * g.Tm * g.Nb + static_cast<int64_t>(ug) * nbw +
         band_offset(ug, ue, u, n - b * g.Nb, nbw, g.G);
}
// chunk moved at transfer step tc (own rank first, then r+1, r+2, ...)
DT_HD void ag_transfer_chunk(const Geom& g, int32_t tc, int32_t& s, int32_t& j) {
  const int32_t u = tc / g.nC;
  j = tc - u * g.nC;
  s = g.swizzle ? (g.rank + u) % g.W : u;
}

// ------------------------------------------------------------------ scatter mode (ReduceScatter)
// m-tile holding the first row of rank q+1
DT_HD int32_t rs_rot0(const Geom& g, int32_t q) {
  const int32_t d1 = (q + 1) % g.W;
  return static_cast<int32_t>((static_cast<int64_t>(d1) * g.Ms / g.BM) % g.Tm);
}
DT_HD int32_t rs_key(const Geom& g, int32_t q, int32_t rot0, int32_t u) {
  const int32_t i = (rot0 + u) % g.Tm;
  const int64_t first = static_cast<int64_t>(i) * g.BM;
  const int64_t last = min64(first + g.BM, g.M) - 1;
  const int64_t d1_first = static_cast<int64_t>((q + 1) % g.W) * g.Ms;
  // feeds the first chunk of rank q+1, the most urgent destination
  if (first < d1_first && last >= d1_first) return 0;
  int32_t s, j;
  row_chunk(g, first, s, j);
  return ((s - q - 1 + 2 * g.W) % g.W) * g.nC + j;
}
DT_HD int32_t rs_count_below(const Geom& g, int32_t q, int32_t rot0, int32_t k) {
  int32_t lo = 0, hi = g.Tm;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (rs_key(g, q, rot0, mid) < k) lo = mid + 1; else hi = mid;
  }
  return lo;
}
// execution position of ReduceScatter tile (q, i, n): rank q's block of Tm*Tn positions, the
// full column bands before n's (Tm*Nb each), then n's band (Nbw columns wide) laid out like a
// band-less order over those columns
DT_HD int64_t rs_position(const Geom& g, int32_t q, int32_t i, int32_t n) {
  if (!g.swizzle) return (static_cast<int64_t>(q) * g.Tm + i) * g.Tn + n;
  const int32_t rot0 = rs_rot0(g, q);
  const int32_t u = (i - rot0 + g.Tm) % g.Tm;
  const int32_t k = rs_key(g, q, rot0, u);
  const int32_t ug = rs_count_below(g, q, rot0, k);
  const int32_t ue = rs_count_below(g, q, rot0, k + 1);
  const int32_t b = n / g.Nb;
  const int32_t nbw = min32(g.Nb, g.Tn - b * g.Nb);
  return static_cast<int64_t>(q) * g.Tm * g.Tn + static_cast<int64_t>(b) * g.Tm * g.Nb +
         static_cast<int64_t>(ug) * nbw + band_offset(ug, ue, u, n - b * g.Nb, nbw, g.G);
}

// ------------------------------------------------------------------ all-to-all (GEMM-AllToAll)
// Scatter mode by columns: rank q sends column block h in the order dpos_q(h) = (h - q - 1)
// mod W (rank q+1 first, its own block last), and inside one destination its chunks in row
// order.  The key of m-tile i is dpos*nC + (first chunk it writes), so for one (q, d) the
// m-tiles keyed j are exactly those whose first row lies in chunk j: [first_mtile(j),
// first_mtile(j+1)).  Every (q, d) holds Tm m-tiles x Tnw column tiles; rank q's tiles fill
// positions [q*Tm*Tn, (q+1)*Tm*Tn).
DT_HD int32_t a2a_first_mtile(const Geom& g, int32_t j) {
  const int64_t t = cdiv64(static_cast<int64_t>(j) * g.Cr, g.BM);
  return static_cast<int32_t>(t < g.Tm ? t : g.Tm);
}
// execution position of AllToAll tile (q, i, n), n = h * Tnw + c
DT_HD int64_t a2a_position(const Geom& g, int32_t q, int32_t i, int32_t n) {
  if (!g.swizzle) return (static_cast<int64_t>(q) * g.Tm + i) * g.Tn + n;
  const int32_t h = n / g.Tnw;
  const int32_t c = n - h * g.Tnw;
  const int32_t d = (h - q - 1 + 2 * g.W) % g.W;
  const int32_t j = static_cast<int32_t>(static_cast<int64_t>(i) * g.BM / g.Cr);
  const int32_t ug = a2a_first_mtile(g, j);
  const int32_t ue = a2a_first_mtile(g, j + 1);
  return static_cast<int64_t>(g.Tnw) * g.Tm * (static_cast<int64_t>(q) * g.W + d) +
         static_cast<int64_t>(g.Tnw) * ug + band_offset(ug, ue, i, c, g.Tnw, g.G);
}
// stores counted on chunk j of one (destination, source) pair: the bm-row tiles (one CTA's
// rows) whose rows touch it, times Tnw
DT_HD int32_t a2a_chunk_tiles(const Geom& g, int32_t j, int32_t bm) {
  const int64_t lo = static_cast<int64_t>(j) * g.Cr;
  const int64_t hi = min64(lo + g.Cr, g.Ms);
  return static_cast<int32_t>((hi - 1) / bm - lo / bm + 1) * g.Tnw;
}

// Execution position of tile id t of an operation with the dt_op numbering (0 AllGather:
// t = i*Tn + n; 1 ReduceScatter, 2 AllReduce, 3 AllToAll: t = (q*Tm + i)*Tn + n).
DT_HD int64_t tile_position(const Geom& g, int op, int64_t t) {
  if (op == 0) return ag_position(g, static_cast<int32_t>(t / g.Tn), static_cast<int32_t>(t % g.Tn));
  const int64_t per_q = static_cast<int64_t>(g.Tm) * g.Tn;
  const int32_t q = static_cast<int32_t>(t / per_q);
  const int64_t rem = t - q * per_q;
  const int32_t i = static_cast<int32_t>(rem / g.Tn);
  const int32_t n = static_cast<int32_t>(rem - static_cast<int64_t>(i) * g.Tn);
  return op == 3 ? a2a_position(g, q, i, n) : rs_position(g, q, i, n);
}

// Most chunks that the rows of one m-tile touch: each (m-tile, chunk) piece times a column
// tile is one ReduceScatter reduction unit with its own arrival counter.
inline int32_t rs_pieces_max(const Geom& g) {
  int32_t best = 0;
  for (int32_t i = 0; i < g.Tm; ++i) {
    int32_t k = 0;
    const int64_t end = min64(static_cast<int64_t>(i + 1) * g.BM, g.M);
    for (int64_t r = static_cast<int64_t>(i) * g.BM; r < end; ++k) {
      int32_t s, j;
      row_chunk(g, r, s, j);
      r = static_cast<int64_t>(s) * g.Ms + min64(static_cast<int64_t>(j + 1) * g.Cr, g.Ms);
    }
    best = k > best ? k : best;
  }
  return best;
}

}  // namespace dt
