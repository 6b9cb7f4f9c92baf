"""Pins of the tile-order oracle (distributed swizzle, gather and scatter modes).

Checked against: the hand-written worked orders in tests/golden (from the
DITRON Fig. 3 rule and the Triton-distributed non-perfect tiling rule),
bijection on tile ids including ragged edges, identity when the swizzle is
off, dependency safety of the gather order (simulated chunk arrival), the
own-rank-first / own-rank-last properties, the group raster inside a chunk,
and brute-force arrival counts.
"""
import itertools
import os

import pytest

from oracle import plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, order = line.split(":")
            rows.append((head.split(), [int(x) for x in order.split()]))
    return rows


def test_golden_rank_offset_orders():
    w, ms, bm, bn = 4, 128, 128, 256
    for head, order in _read_golden("ditron_fig3_rank_offset.txt"):
        kind, sw = head[0], bool(int(head[1]))
        if kind == "ag":
            r = int(head[2])
            assert plan.ag_order(w, r, w * ms, bn, ms, bm, bn, swizzle=sw) == order
        else:
            assert plan.rs_order(w, w * ms, bn, ms, bm, bn, swizzle=sw) == order


def test_golden_nonperfect_tiling():
    for head, order in _read_golden("nonperfect_tiling_w2.txt"):
        if head[0] == "ag":
            assert plan.ag_order(2, int(head[1]), 6, 1, 3, 2, 1) == order
        else:
            assert plan.rs_order(2, 6, 1, 3, 2, 1) == order


def test_golden_ag_column_bands():
    for head, order in _read_golden("ag_column_bands.txt"):
        r, ms, cr, tn, g, nb = (int(x) for x in head[1:])
        assert plan.ag_order(2, r, 2 * ms, tn, cr, 1, 1, group=g, col_band=nb) == order, head[0]


@pytest.mark.parametrize("w,r,m,n,cr,bm,bn", [(2, 1, 512, 2048, 128, 128, 256),
                                              (3, 2, 390, 520, 50, 128, 96),
                                              (8, 3, 8192, 3584, 1024, 256, 256),
                                              (5, 0, 35, 17, 3, 4, 1)])
@pytest.mark.parametrize("nb", [1, 2, 3, 7, 1000])
def test_ag_column_bands_keep_the_gather_order_inside_each_band(w, r, m, n, cr, bm, bn, nb):
    """AllGather column bands: a bijection; the bands come one after another; inside a band the
    order is the band-less order restricted to it (so every band follows the chunks' arrival)."""
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    o = plan.ag_order(w, r, m, n, cr, bm, bn, col_band=nb)
    assert sorted(o) == list(range(tm * tn))
    bands = [(t % tn) // nb for t in o]
    assert bands == sorted(bands)
    base = plan.ag_order(w, r, m, n, cr, bm, bn)
    for b in set(bands):
        assert [t for t in o if (t % tn) // nb == b] == [t for t in base if (t % tn) // nb == b]
    if nb >= tn:
        assert o == base


def test_golden_column_bands():
    for head, order in _read_golden("rs_column_bands.txt"):
        ms, cr, tn, g, nb = (int(x) for x in head[1:])
        assert plan.rs_order(2, 2 * ms, tn, cr, 1, 1, group=g, col_band=nb) == order, head[0]


@pytest.mark.parametrize("w,m,n,cr,bm,bn", [(2, 512, 2048, 128, 128, 256), (3, 390, 520, 50, 128, 96),
                                            (4, 2048, 4096, 256, 128, 256), (5, 35, 17, 3, 4, 1)])
@pytest.mark.parametrize("nb", [1, 2, 3, 5, 1000])
def test_column_bands_keep_each_rank_and_unit_in_order(w, m, n, cr, bm, bn, nb):
    """Column bands reorder tiles inside a rank's pass only: the order is a bijection, rank q's
    tiles still come as one block, inside a band the order is the band-less order restricted
    to it, the bands come one after another, and every unit still receives its partials in
    source order q = 0..W-1."""
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    o = plan.rs_order(w, m, n, cr, bm, bn, col_band=nb)
    assert sorted(o) == list(range(w * tm * tn))
    base = plan.rs_order(w, m, n, cr, bm, bn)
    per_q = tm * tn
    for q in range(w):
        mine = o[q * per_q:(q + 1) * per_q]
        assert all(t // per_q == q for t in mine)
        bands = [(t % tn) // nb for t in mine]
        assert bands == sorted(bands)
        for b in set(bands):
            assert [t for t in mine if (t % tn) // nb == b] == \
                [t for t in base[q * per_q:(q + 1) * per_q] if (t % tn) // nb == b]
    if nb >= tn:
        assert o == base


GRID = [
    # (W, M, N, Cr, BM, BN)
    (1, 100, 300, 64, 128, 256),
    (2, 512, 512, 128, 128, 256),
    (3, 390, 520, 50, 128, 256),
    (4, 2048, 4096, 256, 128, 256),
    (6, 6000, 3000, 192, 128, 256),
    (8, 80, 64, 4, 128, 256),
    (8, 1024, 1000, 7, 64, 96),
    (5, 35, 17, 3, 4, 8),
    (7, 700, 33, 1000, 96, 16),
]


@pytest.mark.parametrize("case", GRID)
@pytest.mark.parametrize("swizzle", [True, False])
def test_orders_are_bijections(case, swizzle):
    w, m, n, cr, bm, bn = case
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    for r in range(w):
        o = plan.ag_order(w, r, m, n, cr, bm, bn, swizzle)
        assert sorted(o) == list(range(tm * tn))
    o = plan.rs_order(w, m, n, cr, bm, bn, swizzle)
    assert sorted(o) == list(range(w * tm * tn))


@pytest.mark.parametrize("case", GRID)
def test_swizzle_off_is_identity(case):
    w, m, n, cr, bm, bn = case
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    for r in range(w):
        assert plan.ag_order(w, r, m, n, cr, bm, bn, False) == list(range(tm * tn))
    assert plan.rs_order(w, m, n, cr, bm, bn, False) == list(range(w * tm * tn))


def _rows_of_mtile(i, m, bm):
    return range(i * bm, min((i + 1) * bm, m))


@pytest.mark.parametrize("case", GRID)
@pytest.mark.parametrize("swizzle", [True, False])
def test_gather_order_is_dependency_monotone(case, swizzle):
    """Simulated arrival: chunks land one by one in transfer order; the index of the
    last chunk each tile needs never decreases along the tile order, so no tile is
    held up by a chunk later than the one the next tile needs."""
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    for r in range(w):
        arrival = {c: t for t, c in enumerate(plan.ag_transfer_order(w, r, m, cr, swizzle))}
        assert sorted(arrival) == [(s, j) for s in range(w) for j in range(nc)]
        needed = []
        for tile in plan.ag_order(w, r, m, n, cr, bm, bn, swizzle):
            i = tile // tn
            needed.append(max(arrival[plan.chunk_of_row(g, ms, cr)] for g in _rows_of_mtile(i, m, bm)))
        if swizzle:
            assert needed == sorted(needed)


@pytest.mark.parametrize("case", GRID)
def test_gather_own_rank_first(case):
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    for r in range(w):
        order = plan.ag_order(w, r, m, n, cr, bm, bn, True)
        own = [t for t in order
               if all(g // ms == r for g in _rows_of_mtile(t // tn, m, bm))]
        if own:
            # every tile that reads only its own rank's rows precedes all others
            assert order[:len(own)] == own
        # the first chunk transferred is the own rank's first chunk
        assert plan.ag_transfer_order(w, r, m, cr, True)[0] == (r, 0)


@pytest.mark.parametrize("case", GRID)
def test_gather_straddling_tile_last(case):
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    for r in range(1, w):
        i = (r * ms - 1) // bm  # m-tile holding the last row of rank r-1
        if (r * ms) // bm == i and i * bm < r * ms < min((i + 1) * bm, m):
            # it waits for the last chunk of rank r-1, the latest chunk of the gather,
            # so it runs after every tile that needs only earlier chunks
            keys = plan.ag_keys(w, r, m, cr, bm, True)
            assert keys[i] == w * nc - 1 == max(keys.values())
            order = plan.ag_order(w, r, m, n, cr, bm, bn, True)
            first = min(p for p, t in enumerate(order) if t // tn == i)
            assert all(keys[t // tn] == keys[i] for t in order[first:])


@pytest.mark.parametrize("case", GRID)
def test_scatter_next_rank_first_own_last(case):
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    order = plan.rs_order(w, m, n, cr, bm, bn, True)
    for q in range(w):
        mine = [(t // tn) % tm for t in order if t // (tm * tn) == q]
        dests = [{g // ms for g in _rows_of_mtile(i, m, bm)} for i in mine]
        nxt = (q + 1) % w
        assert nxt in dests[0]
        if w > 1:
            own_only = [k for k, d in enumerate(dests) if d == {q}]
            # tiles that feed only the own block come after every tile that feeds another rank
            assert own_only == list(range(len(dests) - len(own_only), len(dests)))


@pytest.mark.parametrize("case", GRID)
def test_scatter_ranks_one_after_another(case):
    """The virtual source ranks run one after another (q ascending) and, inside one
    rank, the send keys never decrease."""
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    keys = {q: plan.rs_keys(w, q, m, cr, bm) for q in range(w)}
    seq = []
    for t in plan.rs_order(w, m, n, cr, bm, bn, True):
        q, i = t // (tm * tn), (t // tn) % tm
        seq.append((q, keys[q][i]))
    assert seq == sorted(seq)


@pytest.mark.parametrize("case", GRID)
@pytest.mark.parametrize("swizzle", [True, False])
def test_scatter_units_receive_sources_in_rank_order(case, swizzle):
    """Executed one tile at a time, every reduction unit receives its W partials from
    sources 0, 1, ..., W-1 in that order, the order in which they are summed."""
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    seen = {}
    for t in plan.rs_order(w, m, n, cr, bm, bn, swizzle):
        q, i, c = t // (tm * tn), (t // tn) % tm, t % tn
        for u in {plan.chunk_of_row(g, ms, cr) for g in _rows_of_mtile(i, m, bm)}:
            got = seen.setdefault((i, u, c), [])
            assert len(got) == q
            got.append(q)


@pytest.mark.parametrize("case", GRID)
def test_group_raster_inside_chunk(case):
    """Inside one key group, bands of up to G m-tiles are swept column by column."""
    w, m, n, cr, bm, bn = case
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    g = 8
    order = plan.ag_order(w, 0, m, n, cr, bm, bn, True, group=g)
    keys = plan.ag_keys(w, 0, m, cr, bm, True)
    pos = 0
    while pos < len(order):
        k = keys[order[pos] // tn]
        grp = list(itertools.takewhile(lambda t: keys[t // tn] == k, order[pos:]))
        mt = sorted({t // tn for t in grp})
        assert len(grp) == len(mt) * tn
        for b0 in range(0, len(mt), g):
            band = mt[b0:b0 + g]
            seg = grp[b0 * tn:(b0 + len(band)) * tn]
            assert seg == [i * tn + c for c in range(tn) for i in band]
        pos += len(grp)


@pytest.mark.parametrize("case", GRID)
def test_arrival_counts_brute_force(case):
    w, m, n, cr, bm, bn = case
    ms, nc, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    counts = {}
    for t in plan.rs_order(w, m, n, cr, bm, bn, True):
        q, i, c = t // (tm * tn), (t // tn) % tm, t % tn
        for u in {plan.chunk_of_row(g, ms, cr) for g in _rows_of_mtile(i, m, bm)}:
            counts[(i, u[0], u[1], c)] = counts.get((i, u[0], u[1], c), 0) + 1
    want = plan.rs_expected_arrivals(w, m, n, cr, bm, bn)
    assert counts == want
    assert set(want.values()) == {w}  # only the W source tiles of the same m-tile write a unit


def test_chunk_map_covers_rows_once():
    for (w, m, n, cr, bm, bn) in GRID:
        ms, nc, _, _ = plan.geometry(w, m, n, cr, bm, bn)
        seen = []
        for s in range(w):
            for j in range(nc):
                lo, hi = plan.chunk_rows_range(s, j, ms, cr)
                assert lo < hi
                seen.extend(range(lo, hi))
                assert all(plan.chunk_of_row(g, ms, cr) == (s, j) for g in range(lo, hi))
        assert seen == list(range(m))


_ORIG_AG_ORDER = plan.ag_order


def _mut_ag_order_negative_offset(w, r, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    return _ORIG_AG_ORDER(w, (-r) % w, m, n, cr, bm, bn, swizzle, group, col_band)


def _mut_ag_order_min_key(w, r, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    ms = m // w
    nc = plan.cdiv(ms, cr)
    keys = {i: min(plan.ag_pos(s, j, w, r, nc) for (s, j) in plan.tile_chunks(i, m, ms, cr, bm))
            for i in range(tm)}
    ent = sorted((keys[i], c, i) for i in range(tm) for c in range(tn))
    return [i * tn + c for (_, c, i) in ent]


_ORIG_RS_ORDER = plan.rs_order


def _mut_rs_order_ranks_interleaved(w, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    """Steps interleaved across ranks (key before q) instead of rank after rank."""
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    ent = []
    for q in range(w):
        keys = plan.rs_keys(w, q, m, cr, bm)
        for i in range(tm):
            for c in range(tn):
                ent.append((keys[i], q, c, i))
    ent.sort()
    return [(q * tm + i) * tn + c for (_, q, c, i) in ent]


def _mut_rs_order_own_first(w, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    """Each rank keeps its own block first (dpos = (s - q) mod W)."""
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    ms = m // w
    nc = plan.cdiv(ms, cr)
    ent = []
    for q in range(w):
        for i in range(tm):
            key = min(((s - q) % w) * nc + j for (s, j) in plan.tile_chunks(i, m, ms, cr, bm))
            for c in range(tn):
                ent.append((q, key, c, i))
    ent.sort()
    return [(q * tm + i) * tn + c for (q, _, c, i) in ent]


def _mut_ag_order_bands_ignored(w, r, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    """AllGather column bands ignored."""
    return _ORIG_AG_ORDER(w, r, m, n, cr, bm, bn, swizzle, group)


def _mut_rs_order_bands_ignored(w, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    """Column bands ignored: the band-less order."""
    return _ORIG_RS_ORDER(w, m, n, cr, bm, bn, swizzle, group)


def _mut_rs_order_band_inside_key(w, m, n, cr, bm, bn, swizzle=True, group=8, col_band=None):
    """Column band taken inside each destination step instead of around the whole pass."""
    _, _, tm, tn = plan.geometry(w, m, n, cr, bm, bn)
    nb = col_band or tn
    ent = []
    for q in range(w):
        keys = plan.rs_keys(w, q, m, cr, bm)
        band = plan._bands(keys, group)
        for i in range(tm):
            for c in range(tn):
                ent.append((q, keys[i], c // nb, band[i], c, i))
    ent.sort()
    return [(q * tm + i) * tn + c for (q, _, _, _, c, i) in ent]


@pytest.mark.parametrize("name,mutant", [("ag_order", _mut_ag_order_negative_offset),
                                         ("ag_order", _mut_ag_order_min_key),
                                         ("rs_order", _mut_rs_order_ranks_interleaved),
                                         ("rs_order", _mut_rs_order_own_first),
                                         ("rs_order", _mut_rs_order_bands_ignored),
                                         ("ag_order", _mut_ag_order_bands_ignored),
                                         ("rs_order", _mut_rs_order_band_inside_key)])
def test_plan_pins_catch_planted_mistakes(name, mutant, monkeypatch):
    monkeypatch.setattr(plan, name, mutant)
    caught = False
    for fn in (test_golden_rank_offset_orders, test_golden_nonperfect_tiling,
               test_golden_column_bands, test_golden_ag_column_bands):
        try:
            fn()
        except AssertionError:
            caught = True
    assert caught
