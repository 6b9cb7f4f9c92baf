"""GPU parity of the AllGather alone (the fused AllGather-GEMM's chunk transfer, through the C
ABI) against the oracle's row concatenation: a copy, so bit for bit.

Every backend (copy engine, in-kernel TMA bulk copies, in-kernel vector ld/st) over world sizes
1, 3, 8 and 16, ragged chunks (1 row, 96 rows, 1000 rows against 300-row shards), padded source
rows, padded destination rows (copy engine; the padding stays untouched), few SMs, swizzle off
and a nonzero rank; then the FFN pair's shards (W = 8, 1024 x 8192 each) on every backend.
"""
import numpy as np
import pytest

from gpu_helpers import dev_bf16, load_dt, need_gpu, torch, workspace
from oracle import reference
from synth_inputs import WORKLOADS, make_ag_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def _bits(t, cols=None):
    x = t.view(torch.int16).cpu().numpy().view(np.uint16)
    return x if cols is None else x[:, :cols]


def _gather(dt, shards_dev, m, k, ldc=0, **kw):
    w = len(shards_dev)
    args = dt.make_args(w, m, 8, k, ldc=ldc, **kw)
    ws = workspace(dt.workspace_size(args, dt.OP_AG))
    out = torch.full((m, ldc or k), float("nan"), dtype=torch.bfloat16, device="cuda")
    dt.allgather(shards_dev, out, ws, args)
    st, info = dt.check(ws)
    assert st == 0, (dt.capi.status_string(st), info)
    return out


CASES = [  # (W, Ms, K)
    (1, 300, 136), (3, 300, 520), (8, 128, 8192 + 64), (16, 9, 64),
]


@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst"])
@pytest.mark.parametrize("w, ms, k", CASES)
@pytest.mark.parametrize("chunk_rows", [1, 96, 1000])
def test_allgather_is_the_concatenation(dt, backend, w, ms, k, chunk_rows):
    inp = make_ag_inputs(w, w * ms, 8, k, seed=51 + w)
    want = reference.allgather(inp.shards)
    out = _gather(dt, [dev_bf16(s) for s in inp.shards], w * ms, k, chunk_rows=chunk_rows,
                  backend=backend)
    assert np.array_equal(_bits(out), want)


@pytest.mark.parametrize("backend", ["copy_engine", "tma", "ldst"])
def test_padded_sources_few_sms_rank_and_order(dt, backend):
    w, ms, k = 4, 200, 264
    inp = make_ag_inputs(w, w * ms, 8, k, seed=57)
    want = reference.allgather(inp.shards)
    dev = [dev_bf16(s, k + 40) for s in inp.shards]  # lda = k + 40
    for kw in (dict(), dict(num_sms=5), dict(rank=3), dict(swizzle=False), dict(chunk_rows=7)):
        kw.setdefault("chunk_rows", 64)
        out = _gather(dt, dev, w * ms, k, lda=k + 40, backend=backend, **kw)
        assert np.array_equal(_bits(out), want), kw


def test_copy_engine_writes_strided_rows_and_leaves_padding(dt):
    w, ms, k = 3, 128, 200
    inp = make_ag_inputs(w, w * ms, 8, k, seed=58)
    want = reference.allgather(inp.shards)
    for backend in ("copy_engine", "auto"):  # auto takes the copy engine for strided rows
        out = _gather(dt, [dev_bf16(s) for s in inp.shards], w * ms, k, ldc=k + 24,
                      chunk_rows=50, backend=backend)
        assert np.array_equal(_bits(out, k), want)
        assert torch.isnan(out[:, k:].float()).all(), "padding written"


def test_ffn_pair_shards_every_backend(dt):
    wl = WORKLOADS["ag_w8_m8192_n3584_k8192"]
    inp = wl.make()
    dev = [dev_bf16(s) for s in inp.shards]
    want = torch.cat(dev, dim=0)
    for backend in ("copy_engine", "tma", "ldst"):
        for cr in (wl.chunk_rows or 256, 256):
            out = _gather(dt, dev, wl.m, wl.k, chunk_rows=cr, backend=backend)
            assert torch.equal(out.view(torch.int16), want.view(torch.int16)), (backend, cr)
    # and the oracle on sampled rows
    rows = np.random.Generator(np.random.PCG64(5)).integers(0, wl.m, 24)
    full = reference.allgather(inp.shards)
    got = _bits(out)
    assert np.array_equal(got[rows], full[rows])
