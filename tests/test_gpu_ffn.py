"""GPU parity of the chained tensor-parallel feed-forward block (dt_ffn_ag_rs): the fused
AllGather-GEMM with the activation in its epilogue writes H, the fused GEMM-ReduceScatter
reads H's rank blocks.  Checked against the float64 oracle (H rounded to bf16 as the kernel
stores it) for GELU, SiLU and no activation, on an aligned and a ragged shape, and against
the two fused calls made one after the other."""
import numpy as np
import pytest

from gpu_helpers import (assert_close, bits_equal, dev_bf16, load_dt, need_gpu, out_tensor,
                         to_f64, torch, workspace)
from oracle import reference
from synth_inputs import f64_from_bf16_bits, make_ffn_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def _run(dt, inp, m, k, fr, n, act, cr_ag, cr_rs, backend="auto"):
    w = inp.world_size
    ag = dt.make_args(w, m, w * fr, k, chunk_rows=cr_ag, act=act, backend=backend)
    rs = dt.make_args(w, m, n, fr, chunk_rows=cr_rs, lda=w * fr)
    x = [dev_bf16(s) for s in inp.x_shards]
    w1 = dev_bf16(inp.w1)
    w2 = [dev_bf16(t) for t in inp.w2]
    h = out_tensor(m, w * fr, "bf16")
    outs = [out_tensor(m // w, n, "bf16") for _ in range(w)]
    ws_ag = workspace(dt.workspace_size(ag, dt.OP_AG))
    ws_rs = workspace(dt.workspace_size(rs, dt.OP_RS))
    dt.ffn_ag_rs(x, w1, w2, h, outs, ws_ag, ws_rs, ag, rs)
    assert dt.check(ws_ag)[0] == 0 and dt.check(ws_rs)[0] == 0
    return h, outs, (x, w1, w2, ag, rs)


@pytest.mark.parametrize("act", ["gelu_tanh", "silu", "none"])
@pytest.mark.parametrize("case", [(4, 512, 256, 128, 256, 64, 128), (6, 600, 200, 48, 72, 37, 50)])
def test_ffn_block_parity(dt, case, act):
    w, m, k, fr, n, cr_ag, cr_rs = case
    inp = make_ffn_inputs(w, m, k, fr, n, seed=61 + m, dist_x="normal(1.0)", dist_w="normal(0.1)")
    h, outs, _ = _run(dt, inp, m, k, fr, n, act, cr_ag, cr_rs)
    h_ref, out_ref = reference.ffn_tp([f64_from_bf16_bits(s) for s in inp.x_shards],
                                      f64_from_bf16_bits(inp.w1),
                                      [f64_from_bf16_bits(t) for t in inp.w2], act)
    assert_close(to_f64(h), h_ref, "bf16", f"H {act}")
    for s, (o, r) in enumerate(zip(outs, out_ref)):
        assert_close(to_f64(o), r, "bf16", f"out rank {s} {act}")


def test_ffn_block_equals_the_two_calls(dt):
    w, m, k, fr, n = 4, 512, 256, 128, 256
    inp = make_ffn_inputs(w, m, k, fr, n, seed=7)
    h, outs, (x, w1, w2, ag, rs) = _run(dt, inp, m, k, fr, n, "gelu_tanh", 64, 128, "tma")
    h2 = out_tensor(m, w * fr, "bf16")
    ws = workspace(max(dt.workspace_size(ag, dt.OP_AG), dt.workspace_size(rs, dt.OP_RS)))
    dt.ag_gemm(x, w1, h2, ws, ag)
    outs2 = [out_tensor(m // w, n, "bf16") for _ in range(w)]
    dt.gemm_rs([h2[:, q * fr:(q + 1) * fr] for q in range(w)], w2, outs2, ws, rs)
    assert dt.check(ws)[0] == 0
    assert bits_equal(h, h2)
    assert all(bits_equal(a, b) for a, b in zip(outs, outs2))
