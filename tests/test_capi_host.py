"""CPU checks of the C ABI library: it loads, exports every function include/dt.h declares,
its argument struct matches the binding, argument errors come back synchronously, and
its host evaluation of the tile order equals the oracle's bit for bit.

No call here launches GPU work.
"""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

from oracle import plan as oplan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dt():
    from tile_level_communication_gb300 import build
    build.build()
    import tile_level_communication_gb300 as t
    t.capi.lib()
    return t


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dt_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(dt):
    names = _declared_functions()
    assert len(names) >= 14
    h = ctypes.CDLL(dt.capi.LIB_PATH)
    missing = [n for n in names if not hasattr(h, n)]
    assert not missing, missing
    # and the binding knows the same set
    assert set(names) == set(dt.capi._SIGS)


def test_args_layout_matches(dt):
    assert dt.capi.lib().dt_sizeof_args() == ctypes.sizeof(dt.capi.DtArgs)
    assert dt.capi.lib().dt_sizeof_tune_point() == ctypes.sizeof(dt.capi.DtTunePoint)
    assert dt.capi.lib().dt_version() >= 100


@pytest.mark.parametrize("kw,status", [
    (dict(world_size=0, m=8, n=8, k=8), "DT_ERR_INVALID"),
    (dict(world_size=17, m=17, n=8, k=8), "DT_ERR_INVALID"),
    (dict(world_size=3, m=8, n=8, k=8), "DT_ERR_INVALID"),          # M % W
    (dict(world_size=2, m=8, n=12, k=8), "DT_ERR_UNSUPPORTED"),     # N % 8
    (dict(world_size=2, m=8, n=8, k=12), "DT_ERR_UNSUPPORTED"),     # AG K % 8
    (dict(world_size=2, m=8, n=8, k=8, rank=2), "DT_ERR_INVALID"),
    (dict(world_size=2, m=8, n=8, k=8, chunk_rows=0), "DT_ERR_INVALID"),
    (dict(world_size=2, m=8, n=8, k=8, lda=4), "DT_ERR_INVALID"),
    (dict(world_size=2, m=8, n=8, k=8, lda=12), "DT_ERR_INVALID"),  # 16-byte rows
    (dict(world_size=2, m=8, n=8, k=8, tile_m=512), "DT_ERR_UNSUPPORTED"),  # 512-row tiles gone
    (dict(world_size=2, m=2 * 100, n=8, k=8, backend="tma_tile"), "DT_ERR_UNSUPPORTED"),  # M/W % 128
    (dict(world_size=2, m=2 * 128, n=8, k=8, backend="tma_tile", copy_ctas=2), "DT_ERR_INVALID"),
    (dict(world_size=2, m=8, n=8, k=8, col_band=-1), "DT_ERR_INVALID"),
])
def test_argument_errors_are_synchronous(dt, kw, status):
    w = kw.pop("world_size")
    m, n, k = kw.pop("m"), kw.pop("n"), kw.pop("k")
    a = dt.make_args(w, m, n, k, **kw)
    with pytest.raises(dt.DtError):
        dt.workspace_size(a, dt.OP_AG)  # returns 0: invalid
    # the fused call rejects the same arguments, with the status, before touching a pointer
    with pytest.raises(dt.DtError) as ei:
        dt.ag_gemm([1] * max(1, min(w, 16)), 1, 1, 256, a, stream=0, ws_bytes=1 << 30)
    assert ei.value.status == getattr(dt.capi, status)


def test_workspace_errors(dt):
    a = dt.make_args(2, 512, 512, 512, chunk_rows=128)
    need = dt.workspace_size(a, dt.OP_AG)
    assert need >= 512 * 512 * 2
    with pytest.raises(dt.DtError) as ei:
        dt.ag_gemm([256, 512], 1024, 2048, 4096, a, stream=0, ws_bytes=need - 1)
    assert "DT_ERR_WORKSPACE" in str(ei.value)
    with pytest.raises(dt.DtError) as ei:
        dt.ag_gemm([256, 512], 1024, 2048, 4096 + 16, a, stream=0, ws_bytes=need)
    assert "DT_ERR_WORKSPACE" in str(ei.value)  # not 256-byte aligned
    with pytest.raises(dt.DtError) as ei:
        dt.ag_gemm([256, 8], 1024, 2048, 4096, a, stream=0, ws_bytes=need)
    assert "DT_ERR_INVALID" in str(ei.value)    # shard not 16-byte aligned
    r = dt.make_args(4, 2048, 4096, 2048, chunk_rows=256)
    assert dt.workspace_size(r, dt.OP_RS) >= 4 * 4 * 512 * 4096 * 4


@pytest.mark.parametrize("op", ["OP_RS", "OP_AR"])
@pytest.mark.parametrize("case", [(8, 8192, 8192, 3584), (4, 2048, 4096, 2048), (6, 6000, 5120, 3000),
                                  (2, 6, 8, 8)])
def test_reduce_workspace_does_not_grow_with_tile_rows(dt, op, case):
    """A larger tile needs no more workspace (only the tile order shrinks), and 512-row tiles
    are not built."""
    w, m, n, k = case
    for cr in (1, 64, 256, 1024):
        sizes = [dt.workspace_size(dt.make_args(w, m, n, k, chunk_rows=cr, tile_m=t),
                                   getattr(dt, op)) for t in (128, 256)]
        assert sizes[0] >= sizes[1] > 0
        assert dt.workspace_size(dt.make_args(w, m, n, k, chunk_rows=cr), getattr(dt, op)) >= sizes[1]
        with pytest.raises(dt.DtError, match="not built"):
            dt.workspace_size(dt.make_args(w, m, n, k, chunk_rows=cr, tile_m=512), getattr(dt, op))


# ----------------------------------------------------------------------------- plan parity

PLAN_GRID = [
    # (W, M, N, Cr) with the library's 128 x 256 tiles
    (1, 128, 256, 128), (1, 100, 264, 64), (2, 512, 512, 128), (2, 6, 8, 3),
    (3, 390, 520, 50), (4, 2048, 4096, 256), (6, 6000, 3000, 192), (6, 6000, 5120, 192),
    (8, 80, 64, 4), (8, 1024, 1000, 7), (5, 35, 16, 3), (7, 700, 40, 1000),
    (8, 8192, 3584, 256), (8, 8192, 8192, 256), (8, 16384, 8192, 64), (16, 4096, 512, 100),
    (3, 3 * 129, 8, 1), (4, 4 * 127, 8, 127), (2, 2 * 300, 264, 1000),
]


# the order's tile rows: one CTA (128) or a CTA pair (256); the oracle takes them as BM
TILE_M = [128, 256]


@pytest.mark.parametrize("case", PLAN_GRID)
@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("bm", TILE_M)
def test_host_plan_matches_oracle_ag(dt, case, swizzle, bm):
    w, m, n, cr = case
    for r in range(w):
        a = dt.make_args(w, m, n, 8, rank=r, chunk_rows=cr, swizzle=swizzle, tile_m=bm)
        got = dt.swizzle_plan(a, dt.OP_AG)
        want = oplan.ag_order(w, r, m, n, cr, bm, 256, swizzle)
        assert got.tolist() == want, (case, r)


@pytest.mark.parametrize("case", PLAN_GRID)
@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("bm", TILE_M)
def test_host_plan_matches_oracle_rs(dt, case, swizzle, bm):
    w, m, n, cr = case
    a = dt.make_args(w, m, n, 8, chunk_rows=cr, swizzle=swizzle, tile_m=bm)
    got = dt.swizzle_plan(a, dt.OP_RS)
    want = oplan.rs_order(w, m, n, cr, bm, 256, swizzle)
    assert got.tolist() == want, case


@pytest.mark.parametrize("case", PLAN_GRID)
@pytest.mark.parametrize("nb", [1, 2, 3, 7])
@pytest.mark.parametrize("bm", TILE_M)
def test_host_plan_matches_oracle_rs_column_bands(dt, case, nb, bm):
    w, m, n, cr = case
    for r in sorted({0, w - 1}):
        a = dt.make_args(w, m, n, 8, rank=r, chunk_rows=cr, tile_m=bm, col_band=nb)
        assert dt.swizzle_plan(a, dt.OP_AG).tolist() == oplan.ag_order(w, r, m, n, cr, bm, 256,
                                                                       col_band=nb), (case, r)
    for op in (dt.OP_RS, dt.OP_AR):
        a = dt.make_args(w, m, n, 8, chunk_rows=cr, tile_m=bm, col_band=nb)
        tn = -(-n // 256)
        assert dt.col_band(a, op) == min(nb, tn)
        assert dt.swizzle_plan(a, op).tolist() == oplan.rs_order(w, m, n, cr, bm, 256,
                                                                 col_band=nb), (case, nb)


@pytest.mark.parametrize("w,m,n,k,want", [
    (8, 8192, 8192, 3584, 16),    # B_q 56 MiB: two bands of 16 column tiles
    (4, 2048, 4096, 2048, 16),    # B_q 16 MiB: one band (all 16 column tiles)
    (6, 6000, 5120, 3000, 20),    # B_q 29.3 MiB: one band
    (2, 512, 8192, 16384, 4),     # B_q 256 MiB: eight bands of 4
    (2, 512, 2000, 16384, 4),     # 8 column tiles, B_q 62.5 MiB: two bands of 4
])
def test_automatic_column_bands(dt, w, m, n, k, want):
    a = dt.make_args(w, m, n, k, chunk_rows=128)
    assert dt.col_band(a, dt.OP_RS) == want
    assert dt.col_band(a, dt.OP_AR) == want
    assert dt.col_band(a, dt.OP_AG) == want   # the AllGather's B is K x N as well
    bm = dt.tile_rows(a, dt.OP_RS)
    assert dt.swizzle_plan(a, dt.OP_RS).tolist() == oplan.rs_order(w, m, n, 128, bm, 256,
                                                                   col_band=want)
    bm = dt.tile_rows(a, dt.OP_AG)
    assert dt.swizzle_plan(a, dt.OP_AG).tolist() == oplan.ag_order(w, 0, m, n, 128, bm, 256,
                                                                   col_band=want)


@pytest.mark.parametrize("group", [1, 3, 8, 64])
@pytest.mark.parametrize("bm", TILE_M)
def test_host_plan_group_width(dt, group, bm):
    for (w, m, n, cr) in [(4, 2048, 4096, 256), (6, 6000, 3000, 192)]:
        a = dt.make_args(w, m, n, 8, rank=w - 1, chunk_rows=cr, group=group, tile_m=bm)
        assert dt.swizzle_plan(a, dt.OP_AG).tolist() == oplan.ag_order(
            w, w - 1, m, n, cr, bm, 256, True, group)
        assert dt.swizzle_plan(a, dt.OP_RS).tolist() == oplan.rs_order(
            w, m, n, cr, bm, 256, True, group)


def test_host_plan_random_sweep(dt):
    rng = np.random.Generator(np.random.PCG64(5))
    for _ in range(60):
        w = int(rng.integers(1, 9))
        ms = int(rng.integers(1, 700))
        m = w * ms
        n = 8 * int(rng.integers(1, 80))
        cr = int(rng.integers(1, 2 * ms + 2))
        r = int(rng.integers(0, w))
        a = dt.make_args(w, m, n, 8, rank=r, chunk_rows=cr)
        bm = dt.tile_rows(a, dt.OP_AG)
        assert dt.swizzle_plan(a, dt.OP_AG).tolist() == oplan.ag_order(w, r, m, n, cr, bm, 256)
        bm = dt.tile_rows(a, dt.OP_RS)
        assert dt.swizzle_plan(a, dt.OP_RS).tolist() == oplan.rs_order(w, m, n, cr, bm, 256)
        nb = int(rng.integers(1, 12))
        a = dt.make_args(w, m, n, 8, chunk_rows=cr, col_band=nb, group=int(rng.integers(1, 9)))
        assert dt.swizzle_plan(a, dt.OP_RS).tolist() == oplan.rs_order(
            w, m, n, cr, dt.tile_rows(a, dt.OP_RS), 256, group=a.group, col_band=nb)


def test_tile_rows_auto_rule(dt):
    """tile_m = 0: a CTA pair (256 rows) when that leaves at least 76 tiles, else one CTA."""
    big = dt.make_args(8, 8192, 3584, 8192, chunk_rows=1024)   # 32 x 14 = 448 pair tiles
    small = dt.make_args(2, 512, 512, 512, chunk_rows=128)     # 2 x 2 = 4 pair tiles
    assert dt.tile_rows(big, dt.OP_AG) == 256 and dt.tile_rows(small, dt.OP_AG) == 128
    assert dt.tile_count(big, dt.OP_AG) == 32 * 14
    assert dt.tile_rows(dt.make_args(4, 2048, 4096, 2048, chunk_rows=256), dt.OP_RS) == 256
    for bm in TILE_M:
        a = dt.make_args(2, 512, 512, 512, chunk_rows=128, tile_m=bm)
        assert dt.tile_rows(a, dt.OP_AG) == bm
        assert dt.tile_count(a, dt.OP_AG) == (512 // bm) * 2


# ----------------------------------------------------------------------------- AllToAll

A2A_GRID = [
    # (W, Ms, Nw, Cr): each rank's Ms rows tiled on their own, Nw columns per destination
    (1, 100, 264, 64), (2, 256, 512, 128), (2, 3, 8, 1), (4, 300, 200, 96), (3, 130, 8, 1000),
    (8, 2048, 1280, 512), (8, 2048, 1280, 100), (5, 7, 520, 3), (16, 256, 16, 64),
]


@pytest.mark.parametrize("case", A2A_GRID)
@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("bm", TILE_M)
def test_host_plan_matches_oracle_a2a(dt, case, swizzle, bm):
    w, ms, nw, cr = case
    a = dt.make_args(w, w * ms, w * nw, 8, chunk_rows=cr, swizzle=swizzle, tile_m=bm)
    got = dt.swizzle_plan(a, dt.OP_A2A)
    assert got.tolist() == oplan.a2a_order(w, ms, w * nw, cr, bm, 256, swizzle), case


def test_host_plan_a2a_random_sweep(dt):
    rng = np.random.Generator(np.random.PCG64(6))
    for _ in range(40):
        w = int(rng.integers(1, 9))
        ms = int(rng.integers(1, 600))
        nw = 8 * int(rng.integers(1, 90))
        cr = int(rng.integers(1, 2 * ms + 2))
        g = int(rng.integers(1, 10))
        bm = 128 * int(rng.choice([1, 2]))
        a = dt.make_args(w, w * ms, w * nw, 8, chunk_rows=cr, group=g, tile_m=bm)
        assert dt.swizzle_plan(a, dt.OP_A2A).tolist() == \
            oplan.a2a_order(w, ms, w * nw, cr, bm, 256, True, g)


@pytest.mark.parametrize("kw,status", [
    (dict(world_size=3, m=9, n=16, k=8), "DT_ERR_INVALID"),        # N % W
    (dict(world_size=2, m=8, n=24, k=8), "DT_ERR_UNSUPPORTED"),    # N/W % 8
    (dict(world_size=2, m=7, n=16, k=8), "DT_ERR_INVALID"),        # M % W
    (dict(world_size=2, m=8, n=32, k=8, ldc=8), "DT_ERR_INVALID"),  # ldc < N/W
])
def test_a2a_argument_errors_are_synchronous(dt, kw, status):
    w = kw.pop("world_size")
    m, n, k = kw.pop("m"), kw.pop("n"), kw.pop("k")
    a = dt.make_args(w, m, n, k, **kw)
    assert dt.capi.lib().dt_workspace_size(ctypes.byref(a), dt.OP_A2A) == 0
    with pytest.raises(dt.DtError) as ei:
        dt.gemm_a2a([16] * w, [16] * w, [16] * w, 256, a, stream=0, ws_bytes=1 << 30)
    assert ei.value.status == getattr(dt.capi, status)


def test_a2a_workspace_holds_only_control(dt):
    # K is not restricted (lda pads the rows); the workspace is the control block alone
    a = dt.make_args(8, 16384, 10240, 8190, chunk_rows=512, lda=8192)
    need = dt.workspace_size(a, dt.OP_A2A)
    assert 0 < need < (1 << 20)
    assert dt.a2a_chunks(a) == 8 * 8 * 4


# ----------------------------------------------------------------------------- AllGather alone

@pytest.mark.parametrize("kw, status", [
    (dict(world_size=0, m=512, k=512), "DT_ERR_INVALID"),
    (dict(world_size=3, m=512, k=512), "DT_ERR_INVALID"),            # M % W
    (dict(world_size=2, m=512, k=500), "DT_ERR_UNSUPPORTED"),        # K % 8
    (dict(world_size=2, m=512, k=512, chunk_rows=0), "DT_ERR_INVALID"),
    (dict(world_size=2, m=512, k=512, ldc=504), "DT_ERR_INVALID"),   # out rows shorter than K
    (dict(world_size=2, m=512, k=512, ldc=516), "DT_ERR_INVALID"),   # not 16-byte rows
    (dict(world_size=2, m=512, k=512, ldc=520, backend="tma"), "DT_ERR_UNSUPPORTED"),
    (dict(world_size=2, m=512, k=512, ldc=520, backend="ldst"), "DT_ERR_UNSUPPORTED"),
    (dict(world_size=2, m=512, k=512, lda=500), "DT_ERR_INVALID"),
    (dict(world_size=2, m=512, k=512, backend="tma_tile"), "DT_ERR_INVALID"),  # not a transfer
])
def test_allgather_argument_errors_are_synchronous(dt, kw, status):
    w = kw.pop("world_size")
    m, k = kw.pop("m"), kw.pop("k")
    a = dt.make_args(w, m, 0, k, **kw)  # N plays no part
    with pytest.raises(dt.DtError) as ei:
        dt.allgather([256] * max(1, min(w, 16)), 4096, 8192, a, stream=0, ws_bytes=1 << 30)
    assert ei.value.status == getattr(dt.capi, status)


def test_allgather_pointer_and_workspace_errors(dt):
    a = dt.make_args(2, 512, 8, 512, chunk_rows=128, backend="tma")
    need = dt.workspace_size(a, dt.OP_AG)
    with pytest.raises(dt.DtError) as ei:
        dt.allgather([256, 8], 4096, 8192, a, stream=0, ws_bytes=need)     # shard misaligned
    assert ei.value.status == dt.capi.DT_ERR_INVALID
    with pytest.raises(dt.DtError) as ei:
        dt.allgather([256, 512], 4104, 8192, a, stream=0, ws_bytes=need)   # out misaligned
    assert ei.value.status == dt.capi.DT_ERR_INVALID
    with pytest.raises(dt.DtError) as ei:
        dt.allgather([256, 512], 4096, 8192, a, stream=0, ws_bytes=need - 1)
    assert ei.value.status == dt.capi.DT_ERR_WORKSPACE
    # N does not enter the workspace an AllGather needs
    b = dt.make_args(2, 512, 4096, 512, chunk_rows=128, backend="tma")
    assert dt.workspace_size(b, dt.OP_AG) >= need
    # nothing to move: no pointer is touched
    dt.allgather([0, 0], 0, 0, dt.make_args(2, 0, 8, 512), stream=0, ws_bytes=0)
    dt.allgather([0, 0], 0, 0, dt.make_args(2, 512, 8, 0), stream=0, ws_bytes=0)


def test_group_widths_that_reorder_nothing(dt):
    """The tuners time a group width only when it changes the tile order: with 256-row tiles
    and one chunk per rank, each key holds two m-tiles, so groups 4, 8 and 16 are one order."""
    w, m, n = 4, 2048, 4096
    orders = {g: tuple(dt.swizzle_plan(dt.make_args(w, m, n, 2048, chunk_rows=512, group=g),
                                       dt.OP_RS).tolist()) for g in (1, 4, 8, 16)}
    assert orders[4] == orders[8] == orders[16] != orders[1]


def test_tile_pull_needs_no_gather_buffer(dt):
    """The per-tile pull reads the shards in place: its workspace is the control block and the
    tile order only, and only the AllGather-GEMM takes it."""
    a = dt.make_args(8, 8192, 3584, 8192, chunk_rows=1024, backend="tma_tile")
    b = dt.make_args(8, 8192, 3584, 8192, chunk_rows=1024, backend="tma")
    assert dt.workspace_size(a, dt.OP_AG) < 1 << 20
    assert dt.workspace_size(b, dt.OP_AG) - dt.workspace_size(a, dt.OP_AG) >= 8192 * 8192 * 2
    with pytest.raises(dt.DtError) as ei:
        dt.workspace_size(a, dt.OP_RS)
    assert ei.value.status == dt.capi.DT_ERR_INVALID


def test_trace_bytes_and_attach(dt):
    a = dt.make_args(8, 8192, 3584, 8192, chunk_rows=1000)
    nc = -(-1024 // 1000)
    assert dt.trace_bytes(a) == (4 + 3 * 8 * nc) * 8
    dt.trace_attach(None)
    with pytest.raises(dt.DtError):
        dt.trace_attach(12, 64)  # not 8-byte aligned
    dt.trace_attach(None)


def test_trace_decode_marks_missing_events():
    from tile_level_communication_gb300 import capi
    a = capi.DtArgs()
    a.world_size, a.m, a.chunk_rows = 2, 4, 1   # two chunks per rank
    none = (1 << 64) - 1
    words = [1000, 9000, 700, 2] + [none] * 12
    words[4 + 3 * 2] = 3000   # chunk (1, 0): released at +2 us
    words[6 + 3 * 2] = 3500   # and first read at +2.5 us
    tr = capi.trace_decode(words, a)
    assert tr["kernel_us"] == 8.0 and tr["stall_us_total"] == 0.7 and tr["stalled_waits"] == 2
    assert tr["chunks"][(1, 0)] == {"released_us": 2.0, "first_miss_us": None, "first_read_us": 2.5}
    assert tr["chunks"][(0, 1)] == {"released_us": None, "first_miss_us": None, "first_read_us": None}
