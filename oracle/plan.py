"""Reference tile orders of the distributed swizzle, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
* DITRON page, section 3.2 (论文 §3.2, Fig. 3): a stateless ``swizzle_func`` maps
  the original tile id to a new one with a rank-aware offset; rank r starts at
  ``r mod world_size``.  Gather mode (AllGather-GEMM): local HBM acts as a cache
  of remote memory, own data first while remote chunks are fetched.  Scatter
  mode (GEMM-ReduceScatter): first compute the tiles whose results go to the
  farthest rank.
* Triton-distributed talk, "不完全なブロックスケジューリング": with non-perfect
  tiling an AllGather tile that straddles ranks waits for the latest data it
  needs and runs last; in ReduceScatter the tiles that remote ranks depend on
  run first.
* AutoOverlap page, section 5.4 / Fig. 6: the tile scheduler follows chunk
  arrival order across chunks and keeps a locality-preserving traversal
  inside a chunk; chunks stay where they are.

The appendix that gives DITRON's exact transform is not available, so these
readings are fixed here (and implemented independently by the CUDA side):

Notation: W ranks, own rank r, M rows in total, Ms = M/W rows per rank, chunk
rows Cr, nC = ceil(Ms/Cr) chunks per rank, tiles BM x BN, Tm = ceil(M/BM),
Tn = ceil(N/BN); group width G (default 8).

* chunk (s, j) covers global rows [s*Ms + j*Cr, s*Ms + min((j+1)*Cr, Ms)).
* AllGather, swizzle on: pos(s, j) = ((s - r) mod W) * nC + j.  key(i) = max pos
  over the chunks that m-tile i reads.  Tiles (i, n) are sorted by
  (key(i), band(i), n, i), band(i) = (rank of i among the m-tiles that share its
  key, in ascending i) // G.  Chunks are transferred in ascending pos.
* AllGather column bands (col_band tiles wide; one band = all Tn when B fits the cache): the
  bands run one after another and each repeats the gather order over every chunk: sort by
  (n // col_band, key(i), band(i), n, i).  Only one band of B is in use at a time, so a wide B
  is not re-streamed from DRAM once per key group; the first band still follows the chunks'
  arrival, the later ones find every chunk landed.
* AllGather, swizzle off: tile order i-major (i * Tn + n); transfer order
  ascending (s, j); pos(s, j) = s * nC + j.
* ReduceScatter, swizzle on: source rank q sends to s in the order
  dpos_q(s) = (s - q - 1) mod W (next rank first, its own block last).
  key(q, i) = min over the chunks (s, j) that m-tile i writes of
  dpos_q(s) * nC + j.  Tiles (q, i, n) sorted by (q, key, band, n, i), band taken
  among the m-tiles of the same (q, key): the virtual source ranks run one after
  another, each in its own scatter order.  The pages fix only one rank's order;
  rank after rank is how W ranks that each own an SM array run on one GPU (one
  rank's B_q stays in L2 for all its send steps), and each destination then
  receives its partials in source order q = 0, 1, ..., W-1.
* ReduceScatter column bands (col_band tiles wide; one band = all Tn when B_q fits the
  cache): inside rank q's pass the column bands run one after another, and each band
  repeats the scatter order over all destinations: sort by (q, n // col_band, key, band,
  n, i).  A wide B_q no longer streams once per destination step: only one band of it
  is in use at a time (AutoOverlap section 5.4: the order inside the schedule keeps
  locality).  Destinations still receive their partials in source order.
* ReduceScatter, swizzle off: lexicographic (q, i, n).
* ReduceScatter arrivals: a unit is the part of chunk (s, j) that m-tile i covers, times
  column tile n (AutoOverlap section 4.1: a chunk is made of compute tiles; the reduction
  is done per tile-sized piece of it).  Exactly the W source tiles (q, i, n), q = 0..W-1,
  write its rows, so it is complete after W arrivals.
* AllToAll (GEMM-AllToAll, scatter mode by columns): rank q holds Ms rows of its own,
  m-tiles i = 0 .. ceil(Ms/BM)-1 of those rows, and Y_q's N = W * Nw columns are
  tiled per destination: Tnw = ceil(Nw/BN) column tiles c inside block h, tile column
  n = h * Tnw + c, tile id (q * Tm + i) * (W * Tnw) + n.  Chunk (q, j) = rows
  [j*Cr, min((j+1)*Cr, Ms)) of rank q; what goes to destination h is signalled per
  (h, q, j).  Swizzle on: key(q, i, h) = dpos_q(h) * nC + (first chunk m-tile i
  writes), dpos as in ReduceScatter (the next rank first, the own block last);
  tiles sorted by (key, q, band, c, i), band taken among the m-tiles of the same
  (q, key).  Swizzle off: lexicographic (q, i, n).  Chunk (h, q, j) is complete
  when every tile of source q, destination h whose rows touch it has been stored.
"""
from __future__ import annotations

from collections import defaultdict


def cdiv(a, b):
    return -(-a // b)


def geometry(world_size, m, n, chunk_rows, bm, bn):
    """Return (Ms, nC, Tm, Tn) for the given problem and tiling."""
    if world_size < 1 or m % world_size:
        raise ValueError("M must be a positive multiple of W")
    ms = m // world_size
    nc = cdiv(ms, chunk_rows) if ms > 0 else 0
    return ms, nc, cdiv(m, bm), cdiv(n, bn)


def chunk_of_row(g, ms, chunk_rows):
    """(rank, chunk) that holds global row g."""
    s = g // ms
    return s, (g - s * ms) // chunk_rows


def chunk_rows_range(s, j, ms, chunk_rows):
    """Global row range [lo, hi) of chunk (s, j)."""
    lo = s * ms + j * chunk_rows
    return lo, s * ms + min((j + 1) * chunk_rows, ms)


def tile_chunks(i, m, ms, chunk_rows, bm):
    """Set of chunks that m-tile i touches, by visiting every one of its rows."""
    return {chunk_of_row(g, ms, chunk_rows) for g in range(i * bm, min((i + 1) * bm, m))}


def ag_pos(s, j, world_size, rank, nc, swizzle=True):
    """Position of chunk (s, j) in rank `rank`'s gather (transfer and key) order."""
    if swizzle:
        return ((s - rank) % world_size) * nc + j
    return s * nc + j


def ag_transfer_order(world_size, rank, m, chunk_rows, swizzle=True):
    """Chunks (s, j) in the order the gather moves them."""
    ms = m // world_size
    nc = cdiv(ms, chunk_rows) if ms else 0
    chunks = [(s, j) for s in range(world_size) for j in range(nc)]
    return sorted(chunks, key=lambda c: ag_pos(c[0], c[1], world_size, rank, nc, swizzle))


def _bands(keys_by_tile, group):
    """band index of every m-tile: rank among same-key m-tiles (ascending i) // G."""
    members = defaultdict(list)
    for i in sorted(keys_by_tile):
        members[keys_by_tile[i]].append(i)
    band = {}
    for lst in members.values():
        for idx, i in enumerate(lst):
            band[i] = idx // group
    return band


def ag_keys(world_size, rank, m, chunk_rows, bm, swizzle=True):
    """key(i) = latest gather position among the chunks m-tile i reads."""
    ms = m // world_size
    nc = cdiv(ms, chunk_rows) if ms else 0
    tm = cdiv(m, bm)
    return {i: max(ag_pos(s, j, world_size, rank, nc, swizzle)
                   for (s, j) in tile_chunks(i, m, ms, chunk_rows, bm))
            for i in range(tm)}


def ag_order(world_size, rank, m, n, chunk_rows, bm, bn, swizzle=True, group=8, col_band=None):
    """Tile ids (i * Tn + n) of the AllGather-GEMM in execution order.

    col_band: column tiles per column band (None: all Tn, one band).  The bands run one after
    another and each repeats the gather order over every chunk: sort by
    (n // col_band, key, band, n, i)."""
    _, _, tm, tn = geometry(world_size, m, n, chunk_rows, bm, bn)
    if tm == 0 or tn == 0:
        return []
    if not swizzle:
        return [i * tn + c for i in range(tm) for c in range(tn)]
    nb = tn if col_band is None else col_band
    if nb < 1:
        raise ValueError("col_band must be >= 1")
    keys = ag_keys(world_size, rank, m, chunk_rows, bm, True)
    band = _bands(keys, group)
    entries = sorted((c // nb, keys[i], band[i], c, i) for i in range(tm) for c in range(tn))
    return [i * tn + c for (_, _, _, c, i) in entries]


def rs_dpos(q, s, world_size):
    """Send order of destination s for source rank q: q+1 first, q itself last."""
    return (s - q - 1) % world_size


def rs_keys(world_size, q, m, chunk_rows, bm):
    """key(q, i) = most urgent (smallest) send position among the chunks m-tile i writes."""
    ms = m // world_size
    nc = cdiv(ms, chunk_rows) if ms else 0
    tm = cdiv(m, bm)
    return {i: min(rs_dpos(q, s, world_size) * nc + j
                   for (s, j) in tile_chunks(i, m, ms, chunk_rows, bm))
            for i in range(tm)}


def rs_order(world_size, m, n, chunk_rows, bm, bn, swizzle=True, group=8, col_band=None):
    """Tile ids ((q * Tm + i) * Tn + n) of the GEMM-ReduceScatter in execution order.

    col_band: column tiles per column band (None: all Tn, one band).  Rank q's pass takes the
    bands one after another and repeats its scatter order inside each: sort by
    (q, n // col_band, key, band, n, i)."""
    _, _, tm, tn = geometry(world_size, m, n, chunk_rows, bm, bn)
    if tm == 0 or tn == 0:
        return []
    if not swizzle:
        return list(range(world_size * tm * tn))
    nb = tn if col_band is None else col_band
    if nb < 1:
        raise ValueError("col_band must be >= 1")
    entries = []
    for q in range(world_size):
        keys = rs_keys(world_size, q, m, chunk_rows, bm)
        band = _bands(keys, group)
        for i in range(tm):
            for c in range(tn):
                entries.append((q, c // nb, keys[i], band[i], c, i))
    entries.sort()
    return [(q * tm + i) * tn + c for (q, _, _, _, c, i) in entries]


def rs_expected_arrivals(world_size, m, n, chunk_rows, bm, bn):
    """{(i, s, j, n): partial tiles that must arrive before that unit is reduced}.

    A unit is (rows of m-tile i that lie in chunk (s, j)) x column tile n; the partial
    tiles that write any of its rows are counted over every source rank and m-tile."""
    ms, nc, tm, tn = geometry(world_size, m, n, chunk_rows, bm, bn)
    out = {}
    for s in range(world_size):
        for j in range(nc):
            lo, hi = chunk_rows_range(s, j, ms, chunk_rows)
            for i in sorted({g // bm for g in range(lo, hi)}):
                rows = set(range(max(lo, i * bm), min(hi, (i + 1) * bm)))
                for c in range(tn):
                    writers = [(q, i2) for q in range(world_size) for i2 in range(tm)
                               if rows & set(range(i2 * bm, min(m, (i2 + 1) * bm)))]
                    out[(i, s, j, c)] = len(writers)
    return out


def a2a_geometry(world_size, ms, n, chunk_rows, bm, bn):
    """Return (Nw, nC, Tm, Tnw): columns per destination, chunks per rank, m-tiles per
    rank, column tiles per destination."""
    if world_size < 1 or n % world_size:
        raise ValueError("N must be a positive multiple of W")
    nw = n // world_size
    nc = cdiv(ms, chunk_rows) if ms > 0 else 0
    return nw, nc, cdiv(ms, bm), cdiv(nw, bn)


def a2a_mtile_chunks(i, ms, chunk_rows, bm):
    """Chunks j of a rank that its m-tile i writes, by visiting every row."""
    return {r // chunk_rows for r in range(i * bm, min((i + 1) * bm, ms))}


def a2a_order(world_size, ms, n, chunk_rows, bm, bn, swizzle=True, group=8):
    """Tile ids ((q * Tm + i) * W * Tnw + h * Tnw + c) of the GEMM-AllToAll in execution
    order: source rank after source rank, each rank's tiles in its own scatter order
    (destination q+1 first, its own block last; chunk order inside a destination; grouped
    raster inside a chunk).  Reading: the pages fix each rank's order only; how W virtual
    ranks share one GPU is ours, and rank after rank keeps one rank's A_q and B columns in
    L2 the way separate GPUs would (no result depends on it: each output is one product)."""
    nw, nc, tm, tnw = a2a_geometry(world_size, ms, n, chunk_rows, bm, bn)
    tn = world_size * tnw
    if tm == 0 or tnw == 0:
        return []
    if not swizzle:
        return list(range(world_size * tm * tn))
    entries = []
    for q in range(world_size):
        for h in range(world_size):
            keys = {i: rs_dpos(q, h, world_size) * nc + min(a2a_mtile_chunks(i, ms, chunk_rows, bm))
                    for i in range(tm)}
            band = _bands(keys, group)
            for i in range(tm):
                for c in range(tnw):
                    entries.append((q, keys[i], band[i], c, i, h))
    entries.sort()
    return [(q * tm + i) * tn + h * tnw + c for (q, _, _, c, i, h) in entries]


def a2a_expected_counts(world_size, ms, n, chunk_rows, bm, bn):
    """{(h, q, j): tiles of source q, destination h whose rows touch chunk j}."""
    nw, nc, tm, tnw = a2a_geometry(world_size, ms, n, chunk_rows, bm, bn)
    out = {}
    for h in range(world_size):
        for q in range(world_size):
            for j in range(nc):
                rows = set(range(j * chunk_rows, min((j + 1) * chunk_rows, ms)))
                writers = [(i, c) for i in range(tm) for c in range(tnw)
                           if rows & set(range(i * bm, min(ms, (i + 1) * bm)))]
                out[(h, q, j)] = len(writers)
    return out
