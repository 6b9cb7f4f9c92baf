"""GPU parity of the fused AllGather-GEMM (through the C ABI) against the float64 oracle.

Covers the small W=2 workload for every transfer backend, swizzle on/off, both ranks and
both output types; the ragged W=6 workload (every tile edge ragged); bit-identity across
tile order, chunk size, backend and the kernel-level-overlap baseline; edge cases (W=1,
one-row shards, chunk of one row, chunks larger than a shard, K not a multiple of the
k-block, K=0, M=0, padded leading dimensions with canaries); the bounded-wait failure
path; and sampled entries at the full sizes in the benchmark's launch configuration.
"""
import numpy as np
import pytest

from gpu_helpers import (assert_close, bits_equal, dev_bf16, load_dt, need_gpu, out_tensor,
                         to_f64, torch, workspace)
from oracle import reference
from synth_inputs import WORKLOADS, f64_from_bf16_bits, make_ag_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def _oracle(inp):
    return reference.ag_gemm([f64_from_bf16_bits(s) for s in inp.shards], f64_from_bf16_bits(inp.b))


def _run(dt, inp, m, n, k, out_dtype="bf16", lda=0, ldb=0, ldc=0, fn=None, ws=None, **kw):
    w = inp.world_size
    args = dt.make_args(w, m, n, k, out_dtype=out_dtype, lda=lda, ldb=ldb, ldc=ldc, **kw)
    shards = [dev_bf16(s, lda) for s in inp.shards]
    b = dev_bf16(inp.b, ldb)
    c = out_tensor(m, n, out_dtype, ldc)
    if ws is None:
        ws = workspace(dt.workspace_size(args, dt.OP_AG))
    (fn or dt.ag_gemm)(shards, b, c, ws, args)
    st, info = dt.check(ws)
    assert st == 0, (dt.capi.status_string(st), info)
    return c


@pytest.fixture(scope="module")
def small():
    wl = WORKLOADS["ag_w2_m512_n512_k512"]
    inp = wl.make()
    return wl, inp, _oracle(inp)


@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst", "tma_tile"])
@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("rank", [0, 1])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_small_parity(dt, small, backend, swizzle, rank, out_dtype, tile_m):
    wl, inp, ref = small
    c = _run(dt, inp, wl.m, wl.n, wl.k, out_dtype, chunk_rows=wl.chunk_rows, backend=backend,
             swizzle=swizzle, rank=rank, tile_m=tile_m)
    assert_close(to_f64(c), ref, out_dtype, f"{backend} swz={swizzle} r={rank}")


def test_small_bit_identical_across_variants(dt, small):
    wl, inp, ref = small
    base = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=128, backend="tma", tile_m=128)
    for tile_m in [128, 256]:  # one CTA or a pair per tile: the same bits
        for backend in ["copy_engine", "tma", "ldst", "tma_tile"]:
            for swizzle in [True, False]:
                for cr in [1, 64, 100, 128, 256, 1000]:
                    c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=cr, backend=backend,
                             swizzle=swizzle, rank=1, tile_m=tile_m)
                    assert bits_equal(c, base), (tile_m, backend, swizzle, cr)
            for nb in (1, 2):  # column bands
                c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=64, backend=backend, rank=1,
                         tile_m=tile_m, col_band=nb)
                assert bits_equal(c, base), (tile_m, backend, nb)
        c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=128, fn=dt.ag_gemm_kernel_overlap,
                 tile_m=tile_m)
        assert bits_equal(c, base), tile_m


@pytest.fixture(scope="module")
def ragged():
    wl = WORKLOADS["ag_w6_m6000_n3000_k5120"]
    inp = wl.make()
    return wl, inp, _oracle(inp)


def test_tile_pull_needs_tile_aligned_shards(dt, ragged):
    """Shards of 1000 rows put m-tiles across two shards: the per-tile pull refuses them."""
    wl, inp, ref = ragged
    args = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows,
                        backend="tma_tile")
    with pytest.raises(dt.DtError) as ei:
        dt.workspace_size(args, dt.OP_AG)
    assert "multiple of 128" in ei.value.message


@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst"])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_ragged_parity_and_identity(dt, ragged, backend, tile_m):
    wl, inp, ref = ragged
    outs = []
    for rank, swizzle, cr in [(0, True, wl.chunk_rows), (5, True, wl.chunk_rows), (3, False, 77),
                              (2, True, 1000)]:
        c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=cr, backend=backend, swizzle=swizzle,
                 rank=rank, tile_m=tile_m)
        assert_close(to_f64(c), ref, "bf16", f"{backend} r={rank}")
        outs.append(c)
    assert all(bits_equal(outs[0], o) for o in outs[1:])
    c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, rank=4,
             fn=dt.ag_gemm_kernel_overlap, tile_m=tile_m)
    assert bits_equal(outs[0], c)


@pytest.mark.parametrize("case", [
    # (W, M, N, K, chunk_rows)
    (1, 128, 256, 64, 128),
    (1, 300, 264, 72, 64),
    (3, 3, 8, 8, 1),          # one row per shard, one 8-column tile
    (4, 4 * 33, 40, 136, 1),  # chunk of one row, K not a multiple of 64
    (2, 2 * 70, 24, 8, 500),  # chunk larger than a shard
    (8, 8 * 16, 520, 200, 5),
    (16, 16 * 9, 16, 16, 4),
])
@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst"])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_edge_shapes(dt, case, backend, tile_m):
    w, m, n, k, cr = case
    inp = make_ag_inputs(w, m, n, k, seed=31 + m)
    ref = _oracle(inp)
    for rank in sorted({0, w - 1}):
        c = _run(dt, inp, m, n, k, chunk_rows=cr, backend=backend, rank=rank, tile_m=tile_m)
        assert_close(to_f64(c), ref, "bf16", f"{case} {backend} r={rank}")


@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst"])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_padded_leading_dims_and_canaries(dt, backend, tile_m):
    w, m, n, k = 3, 3 * 50, 72, 96
    inp = make_ag_inputs(w, m, n, k, seed=77)
    ref = _oracle(inp)
    lda, ldb, ldc = 104, 80, 88
    for out_dtype in ["bf16", "f32"]:
        c = _run(dt, inp, m, n, k, out_dtype, lda=lda, ldb=ldb, ldc=ldc, chunk_rows=16,
                 backend=backend, rank=1, tile_m=tile_m)
        assert_close(to_f64(c, n), ref, out_dtype)
        # the padding columns of C were filled with NaN and must be untouched
        assert torch.isnan(c[:, n:].float()).all()


def test_k_zero_and_m_zero(dt):
    inp = make_ag_inputs(2, 8, 16, 8, seed=1)
    args = dt.make_args(2, 8, 16, 0, chunk_rows=4)
    c = out_tensor(8, 16, "bf16")
    ws = workspace(dt.workspace_size(args, dt.OP_AG))
    dt.ag_gemm([dev_bf16(s) for s in inp.shards], dev_bf16(inp.b), c, ws, args)
    torch.cuda.synchronize()
    assert (c.float() == 0).all()
    args0 = dt.make_args(2, 0, 16, 8, chunk_rows=4)
    dt.ag_gemm([dev_bf16(s) for s in inp.shards], dev_bf16(inp.b), c, ws, args0)
    torch.cuda.synchronize()


def test_workspace_reuse_across_problems(dt):
    """One workspace, alternating problems and backends: epochs and layouts stay coherent."""
    big = make_ag_inputs(4, 4 * 96, 264, 128, seed=5)
    small_ = make_ag_inputs(2, 2 * 40, 8, 64, seed=6)
    ref_big, ref_small = _oracle(big), _oracle(small_)
    a_big = dt.make_args(4, 4 * 96, 264, 128, chunk_rows=32)
    ws = workspace(dt.workspace_size(a_big, dt.OP_AG))
    for it in range(3):
        for backend in ["tma", "copy_engine", "ldst"]:
            c = _run(dt, big, 4 * 96, 264, 128, chunk_rows=32, backend=backend, rank=it % 4, ws=ws)
            assert_close(to_f64(c), ref_big, "bf16")
            c = _run(dt, small_, 2 * 40, 8, 64, chunk_rows=7, backend=backend, rank=1, ws=ws)
            assert_close(to_f64(c), ref_small, "bf16")


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst"])
def test_lost_chunk_times_out_and_context_survives(dt, small, tile_m, backend):
    """Host-made fault: one chunk's copy and flag are never issued (the host does not queue
    the copy, or tells the in-kernel transfer to skip the chunk); the consumer tiles' bounded
    waits run out, the error comes back through dt_check, and the next call works (with a CTA
    pair per tile too: the partner CTA's waits run out as well)."""
    wl, inp, ref = small
    args = dt.make_args(2, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, backend=backend,
                        rank=0, timeout_us=200_000, tile_m=tile_m)
    shards = [dev_bf16(s) for s in inp.shards]
    b = dev_bf16(inp.b)
    c = out_tensor(wl.m, wl.n, "bf16")
    ws = workspace(dt.workspace_size(args, dt.OP_AG))
    dt.debug_drop_transfer(3)  # the second chunk of rank 1
    dt.ag_gemm(shards, b, c, ws, args)
    st, info = dt.check(ws)
    assert st == dt.capi.DT_ERR_TIMEOUT, (st, info)
    assert info[0] == 1  # a chunk's ready flag did not flip
    c2 = out_tensor(wl.m, wl.n, "bf16")
    dt.ag_gemm(shards, b, c2, ws, args)
    st, info = dt.check(ws)
    assert st == 0, info
    assert_close(to_f64(c2), ref, "bf16")


def _sampled_indices(m, n, rng, count=1500):
    rows = np.concatenate([rng.integers(0, m, count), [0, m - 1, m // 2, 127, 128]])
    cols = np.concatenate([rng.integers(0, n, count), [0, n - 1, n // 2, 255, 256 % n]])
    return rows, cols


@pytest.mark.parametrize("name,backend,chunk", [
    ("ag_w8_m8192_n3584_k8192", "auto", 1024),   # the bench's launch configuration
    ("ag_w8_m8192_n3584_k8192", "tma", 256),
    ("ag_w8_m16384_n8192_k8192", "auto", 256),
    ("ag_w8_m16384_n8192_k8192", "copy_engine", 2048),
    ("ag_w8_m16384_n8192_k8192", "ldst", 64),
    ("ag_w8_m16384_n8192_k8192", "tma", -256),   # one CTA per tile (tile_m = 128)
])
def test_full_size_sampled(dt, name, backend, chunk):
    wl = WORKLOADS[name]
    inp = wl.make()
    tile_m = 128 if chunk < 0 else 0
    c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=abs(chunk), backend=backend, rank=3,
             tile_m=tile_m)
    rng = np.random.Generator(np.random.PCG64(9))
    rows, cols = _sampled_indices(wl.m, wl.n, rng)
    ref = reference.ag_gemm_entries([f64_from_bf16_bits(s) for s in inp.shards],
                                    f64_from_bf16_bits(inp.b), rows, cols)
    got = c.float()[torch.as_tensor(rows, device="cuda"), torch.as_tensor(cols, device="cuda")]
    # the tolerance scale is the largest |C| over the sample
    assert_close(got.cpu().numpy(), ref, "bf16", name)
    assert torch.isfinite(c.float()).all()


# dedicated CTAs come in whole clusters: a multiple of tile_m / 128
_DEDICATED = [(c, t) for c in (1, 8, 16) for t in (128, 256) if c % (t // 128) == 0]


@pytest.mark.parametrize("backend", ["tma", "ldst"])
@pytest.mark.parametrize("copy_ctas,tile_m", _DEDICATED)
def test_dedicated_transfer_ctas(dt, small, ragged, backend, copy_ctas, tile_m):
    """CTAs that only move chunks (dedicated SMs) give the same bits as co-located warps."""
    for wl, inp, ref in (small, ragged):
        base = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, backend=backend, rank=1,
                    tile_m=tile_m)
        c = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, backend=backend, rank=1,
                 copy_ctas=copy_ctas, tile_m=tile_m)
        assert_close(to_f64(c), ref, "bf16", f"{backend} dedicated {copy_ctas}")
        assert bits_equal(c, base)


def test_tuner_picks_a_measured_candidate_with_identical_output(dt, ragged):
    wl, inp, ref = ragged
    args = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, rank=2, chunk_rows=wl.chunk_rows)
    shards = [dev_bf16(s) for s in inp.shards]
    b = dev_bf16(inp.b)
    c = out_tensor(wl.m, wl.n, "bf16")
    probe = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, rank=2, chunk_rows=64)
    ws = workspace(max(dt.workspace_size(probe, dt.OP_AG), dt.workspace_size(args, dt.OP_AG)))
    pts = dt.tune_ag_gemm(shards, b, c, ws, args, reps=2)
    ran = [p for p in pts if p["status"] == 0 and p["ms"] > 0]
    assert len(ran) >= 10
    # the kept point: the largest chunk rows among the points within 1 % of the fastest (an
    # AllGather has no column bands)
    fastest = min(p["ms"] for p in ran)
    near = [p for p in ran if p["ms"] <= 1.01 * fastest]
    top = max(p["chunk_rows"] for p in near)
    best = min((p for p in near if p["chunk_rows"] == top), key=lambda p: p["ms"])
    assert (args.chunk_rows, args.copy_ctas, args.group) == (best["chunk_rows"], best["copy_ctas"],
                                                             best["group"])
    assert {p["backend"] for p in ran} >= {"tma", "ldst", "copy_engine"}
    assert any(p["copy_ctas"] > 0 for p in ran)
    tuned = out_tensor(wl.m, wl.n, "bf16")
    dt.ag_gemm(shards, b, tuned, ws, args)
    assert dt.check(ws)[0] == 0
    assert_close(to_f64(tuned), ref, "bf16", "tuned")
    default = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, rank=2)
    assert bits_equal(tuned, default)


def test_single_rank_reads_its_shard_in_place(dt):
    """W = 1: nothing to gather; a plain GEMM on the shard, padded rows included."""
    inp = make_ag_inputs(1, 200, 40, 96, seed=91)
    ref = _oracle(inp)
    for act in ("none",):
        c = _run(dt, inp, 200, 40, 96, lda=104, ldc=48, chunk_rows=64, backend="tma")
        assert_close(to_f64(c, 40), ref, "bf16", "W=1")
        assert torch.isnan(c[:, 40:].float()).all()


@pytest.mark.parametrize("backend", ["tma", "ldst", "copy_engine"])
def test_trace_records_release_before_first_read(dt, backend):
    """The debug timeline: every chunk the kernel transfers is released before any tile reads
    past its flag, chunks read in place are never released, and tracing changes no bit."""
    inp = make_ag_inputs(8, 8 * 512, 1024, 2048, seed=13)
    args = dt.make_args(8, 8 * 512, 1024, 2048, rank=2, chunk_rows=128, backend=backend)
    shards = [dev_bf16(s) for s in inp.shards]
    b = dev_bf16(inp.b)
    ws = workspace(dt.workspace_size(args, dt.OP_AG))
    base = out_tensor(8 * 512, 1024, "bf16")
    dt.ag_gemm(shards, b, base, ws, args)
    assert dt.check(ws)[0] == 0
    buf = torch.zeros(dt.trace_bytes(args) // 8, dtype=torch.int64, device="cuda")
    dt.trace_attach(buf)
    try:
        c = out_tensor(8 * 512, 1024, "bf16")
        dt.ag_gemm(shards, b, c, ws, args)
        assert dt.check(ws)[0] == 0
    finally:
        dt.trace_attach(None)
    assert bits_equal(c, base)
    tr = dt.trace_decode(buf.cpu().tolist(), args)
    assert tr["kernel_us"] is not None and tr["kernel_us"] > 0
    for (s, j), ev in tr["chunks"].items():
        if s == 2:   # the own block is tile-aligned: read in place, never transferred
            assert ev["released_us"] is None and ev["first_read_us"] is None, (s, j, ev)
            continue
        assert ev["first_read_us"] is not None, (s, j, ev)
        if backend == "copy_engine":
            assert ev["released_us"] is None   # the copy's stream writes the flag
        else:
            assert ev["released_us"] is not None
            assert 0 <= ev["released_us"] <= ev["first_read_us"] <= tr["kernel_us"], (s, j, ev)
        if ev["first_miss_us"] is not None:
            assert ev["first_miss_us"] <= ev["first_read_us"]
    assert tr["stall_us_total"] >= 0 and tr["stalled_waits"] >= 0
