"""GPU parity of the fused GEMM-AllToAll (through the C ABI) against the float64 oracle.

Small ragged case (300 rows per rank, 200 columns per destination, K = 520, chunk 96): every
output entry against the oracle, padding columns of out_h untouched; bf16 and fp32 outputs;
per-rank and shared B; W = 1; K = 0.  Swizzle on / off, chunk sizes, group widths and the
kernel-level-overlap baseline agree bit for bit (each output entry is one product, computed
by the same MMA sequence whatever the order).  After a call every chunk's ready flag holds
the call's epoch and every counter is back to 0.  The Llama-70B-like sequence-parallel QKV
projection (W = 8, 2048 rows per rank, K = 8192, N = 10240) is checked on sampled entries
and against the baseline bit for bit.
"""
import numpy as np
import pytest

from gpu_helpers import (assert_close, bits_equal, dev_bf16, load_dt, need_gpu, out_tensor,
                         to_f64, torch, workspace)
from oracle import reference
from synth_inputs import WORKLOADS, f64_from_bf16_bits, make_a2a_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def _f64(inp):
    return [f64_from_bf16_bits(a) for a in inp.a], [f64_from_bf16_bits(b) for b in inp.b]


def _upload(inp, lda=0):
    a = [dev_bf16(x, lda) for x in inp.a]
    cache = {}
    b = []
    for x in inp.b:  # a replicated B is uploaded once and passed W times
        if id(x) not in cache:
            cache[id(x)] = dev_bf16(x)
        b.append(cache[id(x)])
    return a, b


def _run(dt, inp, m, n, k, out_dtype="bf16", ldc=0, baseline=False, dev=None, ws=None, **kw):
    w = inp.world_size
    nw = n // w
    args = dt.make_args(w, m, n, k, out_dtype=out_dtype, ldc=ldc, **kw)
    a, b = dev if dev is not None else _upload(inp, kw.get("lda", 0))
    outs = [out_tensor(m, nw, out_dtype, ld=ldc) for _ in range(w)]
    if ws is None:
        ws = workspace(dt.workspace_size(args, dt.OP_A2A))
    if baseline:
        y = [out_tensor(m // w, n, out_dtype) for _ in range(w)]
        dt.gemm_a2a_kernel_overlap(a, b, y, outs, ws, args)
    else:
        dt.gemm_a2a(a, b, outs, ws, args)
    st, info = dt.check(ws)
    assert st == 0, (dt.capi.status_string(st), info)
    return outs, args, ws


@pytest.fixture(scope="module")
def small():
    wl = WORKLOADS["a2a_w4_m1200_n800_k520"]
    inp = wl.make()
    return wl, inp, reference.gemm_a2a(*_f64(inp))


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_small_parity_and_padding_untouched(dt, small, out_dtype, tile_m):
    wl, inp, ref = small
    nw = wl.n // wl.world_size
    ldc = nw + 24
    outs, _, _ = _run(dt, inp, wl.m, wl.n, wl.k, out_dtype, ldc=ldc, chunk_rows=wl.chunk_rows,
                      tile_m=tile_m)
    for h, o in enumerate(outs):
        assert_close(to_f64(o, nw), ref[h], out_dtype, f"out_{h}")
        assert torch.isnan(o[:, nw:].float()).all(), f"out_{h}: padding written"


def test_small_bit_identical_across_orders_chunks_groups_and_baseline(dt, small):
    wl, inp, _ = small
    dev = _upload(inp)
    base, _, _ = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, dev=dev, tile_m=128)
    variants = [dict(swizzle=False), dict(chunk_rows=1), dict(chunk_rows=64),
                dict(chunk_rows=300), dict(chunk_rows=1000), dict(group=1),
                dict(group=3, chunk_rows=128), dict(num_sms=7), dict(tile_m=256),
                dict(tile_m=256, chunk_rows=1), dict(tile_m=256, swizzle=False),
                dict(tile_m=256, num_sms=7)]
    for kw in variants:
        kw.setdefault("chunk_rows", wl.chunk_rows)
        outs, _, _ = _run(dt, inp, wl.m, wl.n, wl.k, dev=dev, **kw)
        assert all(bits_equal(x, y) for x, y in zip(outs, base)), kw
    outs, _, _ = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, dev=dev, baseline=True)
    assert all(bits_equal(x, y) for x, y in zip(outs, base)), "baseline"


@pytest.mark.parametrize("chunk_rows", [96, 1, 300])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_signals_after_each_call(dt, small, chunk_rows, tile_m):
    wl, inp, _ = small
    dev = _upload(inp)
    outs, args, ws = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=chunk_rows, dev=dev,
                          tile_m=tile_m)
    flags, counts, e1 = dt.a2a_signals(args, ws)
    assert e1 > 0 and (flags == e1).all() and (counts == 0).all()
    _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=chunk_rows, dev=dev, ws=ws, tile_m=tile_m)
    flags, counts, e2 = dt.a2a_signals(args, ws)
    assert e2 == e1 + 1 and (flags == e2).all() and (counts == 0).all()


def test_per_rank_b_parity(dt):
    inp = make_a2a_inputs(3, 3 * 200, 3 * 264, 136, seed=41, shared_b=False)
    ref = reference.gemm_a2a(*_f64(inp))
    outs, _, _ = _run(dt, inp, 600, 792, 136, "f32", chunk_rows=64)
    for h, o in enumerate(outs):
        assert_close(to_f64(o), ref[h], "f32", f"out_{h}")


@pytest.mark.parametrize("tile_m", [128, 256])
def test_sixteen_ranks_tiny_blocks(dt, tile_m):
    # the largest world size: 9 rows per rank, 16 columns per destination, K not a multiple of 8
    inp = make_a2a_inputs(16, 16 * 9, 16 * 16, 20, seed=44)
    ref = reference.gemm_a2a(*_f64(inp))
    a = [dev_bf16(x, 24) for x in inp.a]
    b0 = dev_bf16(inp.b[0])
    for swizzle in (True, False):
        outs, _, _ = _run(dt, inp, 16 * 9, 16 * 16, 20, "f32", chunk_rows=4, lda=24,
                          dev=(a, [b0] * 16), tile_m=tile_m, swizzle=swizzle)
        for h, o in enumerate(outs):
            assert_close(to_f64(o), ref[h], "f32", f"out_{h}")


def test_w1_is_a_plain_gemm(dt):
    inp = make_a2a_inputs(1, 257, 264, 200, seed=42)
    ref = reference.gemm_a2a(*_f64(inp))
    outs, _, _ = _run(dt, inp, 257, 264, 200, chunk_rows=100)
    assert_close(to_f64(outs[0]), ref[0], "bf16", "W=1")


def test_k0_writes_zeros_and_m0_is_a_no_op(dt):
    inp = make_a2a_inputs(2, 256, 32, 0, seed=43)
    args = dt.make_args(2, 256, 32, 0, chunk_rows=64)
    outs = [out_tensor(256, 16, "bf16") for _ in range(2)]
    ws = workspace(dt.workspace_size(args, dt.OP_A2A))
    a = [torch.zeros(128, 8, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dt.gemm_a2a(a, a, outs, ws, args)
    torch.cuda.synchronize()
    assert all((o.float() == 0).all() for o in outs)
    args0 = dt.make_args(2, 0, 32, 64, chunk_rows=64)
    dt.gemm_a2a(a, a, outs, ws, args0)  # nothing to do
    torch.cuda.synchronize()
    del inp


@pytest.fixture(scope="module")
def big(dt):
    wl = WORKLOADS["a2a_w8_m16384_n10240_k8192"]
    inp = wl.make()
    return wl, inp, _upload(inp)


def test_large_sampled_entries_and_baseline(dt, big):
    wl, inp, dev = big
    w, nw = wl.world_size, wl.n // wl.world_size
    outs, _, _ = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, dev=dev)
    rng = np.random.Generator(np.random.PCG64(7))
    dest = rng.integers(0, w, 160)
    rows = rng.integers(0, wl.m, 160)
    cols = rng.integers(0, nw, 160)
    # the corners of the first and last blocks too
    dest = np.concatenate([dest, [0, w - 1, w - 1, 0]])
    rows = np.concatenate([rows, [0, wl.m - 1, 0, wl.m - 1]])
    cols = np.concatenate([cols, [0, nw - 1, nw - 1, 0]])
    a64, b64 = [f64_from_bf16_bits(x) for x in inp.a], [f64_from_bf16_bits(inp.b[0])] * w
    want = reference.gemm_a2a_entries(a64, b64, dest, rows, cols)
    got = np.array([float(outs[h][r, c].float()) for h, r, c in zip(dest, rows, cols)])
    scale = max(float(np.max(np.abs(want))), 1e-30)
    assert np.max(np.abs(got - want)) <= 1e-2 * scale
    base, _, _ = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=wl.chunk_rows, dev=dev, baseline=True)
    assert all(bits_equal(x, y) for x, y in zip(outs, base))
