"""GPU parity of the fused GEMM-AllReduce (through the C ABI) against the float64 oracle.

Every rank's output must hold the whole sum; its row block s must equal, bit for bit, the
GEMM-ReduceScatter's out_s (same schedule and fixed-order folding); one shared output buffer
gives the same bits as W copies; swizzle on/off, chunk sizes and the kernel-level-overlap
baseline agree bit for bit.
"""
import numpy as np
import pytest

from gpu_helpers import (assert_close, bits_equal, dev_bf16, load_dt, need_gpu, out_tensor,
                         to_f64, torch, workspace)
from oracle import reference
from synth_inputs import WORKLOADS, f64_from_bf16_bits, make_rs_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def _oracle(inp):
    return reference.gemm_ar([f64_from_bf16_bits(a) for a in inp.a],
                             [f64_from_bf16_bits(b) for b in inp.b])


def _run(dt, inp, m, n, k, out_dtype="bf16", shared=False, fn=None, rs=False, lda=0, **kw):
    w = inp.world_size
    args = dt.make_args(w, m, n, k, out_dtype=out_dtype, lda=lda, **kw)
    a = [dev_bf16(x, lda) for x in inp.a]
    b = [dev_bf16(x) for x in inp.b]
    if rs:
        outs = [out_tensor(m // w, n, out_dtype) for _ in range(w)]
    elif shared:
        one = out_tensor(m, n, out_dtype)
        outs = [one] * w
    else:
        outs = [out_tensor(m, n, out_dtype) for _ in range(w)]
    ws = workspace(dt.workspace_size(args, dt.OP_RS if rs else dt.OP_AR))
    (fn or (dt.gemm_rs if rs else dt.gemm_ar))(a, b, outs, ws, args)
    st, info = dt.check(ws)
    assert st == 0, (dt.capi.status_string(st), info)
    return outs


@pytest.fixture(scope="module")
def w4():
    wl = WORKLOADS["rs_w4_m2048_n4096_k2048"]
    inp = wl.make()
    return wl, inp, _oracle(inp)


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_w4_parity_and_rs_identity(dt, w4, out_dtype):
    wl, inp, ref = w4
    outs = _run(dt, inp, wl.m, wl.n, wl.k, out_dtype, chunk_rows=wl.chunk_rows)
    for r, o in enumerate(outs):
        assert_close(to_f64(o), ref[r], out_dtype, f"rank {r}")
        if r:
            assert bits_equal(o, outs[0])
    rs = _run(dt, inp, wl.m, wl.n, wl.k, out_dtype, chunk_rows=wl.chunk_rows, rs=True)
    ms = wl.m // wl.world_size
    for s in range(wl.world_size):
        assert bits_equal(outs[0][s * ms:(s + 1) * ms], rs[s])


def test_w4_variants_bit_identical(dt, w4):
    wl, inp, ref = w4
    base = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=256)[0]
    for shared, swizzle, cr in [(True, True, 256), (False, False, 256), (False, True, 100),
                                (True, True, 512)]:
        o = _run(dt, inp, wl.m, wl.n, wl.k, shared=shared, chunk_rows=cr, swizzle=swizzle)
        assert all(bits_equal(x, base) for x in o), (shared, swizzle, cr)
    o = _run(dt, inp, wl.m, wl.n, wl.k, chunk_rows=256, fn=dt.gemm_ar_kernel_overlap)
    assert all(bits_equal(x, base) for x in o)


@pytest.mark.parametrize("case", [(6, 6000, 5120, 3000, 192), (3, 3 * 70, 24, 20, 9),
                                  (1, 200, 264, 72, 64), (16, 16 * 9, 16, 16, 4)])
def test_ragged_and_edges(dt, case):
    w, m, n, k, cr = case
    inp = make_rs_inputs(w, m, n, k, seed=51 + m)
    ref = _oracle(inp)
    lda = -(-k // 8) * 8
    outs = _run(dt, inp, m, n, k, chunk_rows=cr, lda=lda)
    for r, o in enumerate(outs):
        assert_close(to_f64(o), ref[r], "bf16", f"{case} rank {r}")
    shared = _run(dt, inp, m, n, k, chunk_rows=cr, lda=lda, shared=True, swizzle=False)
    assert bits_equal(shared[0], outs[0])


def test_k_zero(dt):
    w = 2
    args = dt.make_args(w, 8, 16, 0, chunk_rows=4)
    outs = [out_tensor(8, 16, "bf16") for _ in range(w)]
    a = [torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda") for _ in range(w)]
    b = [torch.zeros((8, 16), dtype=torch.bfloat16, device="cuda") for _ in range(w)]
    ws = workspace(dt.workspace_size(args, dt.OP_AR))
    dt.gemm_ar(a, b, outs, ws, args)
    torch.cuda.synchronize()
    assert all((o.float() == 0).all() for o in outs)
