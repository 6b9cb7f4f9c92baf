"""The fixed-scratch AllGather-GEMM entry point, for callers that cannot allocate device
memory (a plugin whose framework owns all device memory and passes no workspace, a process
whose allocator reserved the whole GPU, a path that cannot afford cudaMalloc's
synchronisation).  It must give the same results as dt_ag_gemm with a caller workspace, on
consecutive calls that share its one scratch array, and reject problems that do not fit.

This file is collected last so that a stop at the first failure has run every other test.
"""
import pytest

from gpu_helpers import (assert_close, bits_equal, dev_bf16, load_dt, need_gpu, out_tensor,
                         to_f64, workspace)
from synth_inputs import WORKLOADS, make_ag_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def _reference_call(dt, inp, args, m, n):
    c = out_tensor(m, n, "bf16")
    ws = workspace(dt.workspace_size(args, dt.OP_AG))
    dt.ag_gemm([dev_bf16(s) for s in inp.shards], dev_bf16(inp.b), c, ws, args)
    st, info = dt.check(ws)
    assert st == 0, info
    return c


def test_static_scratch_matches_workspace_entry_on_consecutive_calls(dt):
    import gc

    import torch

    wl = WORKLOADS["ag_w2_m512_n512_k512"]
    small = wl.make()
    ragged = make_ag_inputs(6, 6 * 100, 264, 1024, seed=12)
    cases = [
        (small, dt.make_args(2, wl.m, wl.n, wl.k, rank=1, chunk_rows=wl.chunk_rows, backend="tma"),
         wl.m, wl.n),
        (ragged, dt.make_args(6, 600, 264, 1024, rank=4, chunk_rows=37, backend="ldst"), 600, 264),
        (small, dt.make_args(2, wl.m, wl.n, wl.k, rank=0, chunk_rows=64, backend="auto"),
         wl.m, wl.n),
    ]
    for inp, args, m, n in cases:
        want = _reference_call(dt, inp, args, m, n)
        shards = [dev_bf16(s) for s in inp.shards]
        b = dev_bf16(inp.b)
        outs = [out_tensor(m, n, "bf16") for _ in range(3)]
        dt.ag_gemm_static_scratch(shards, b, outs[0], args)  # first call: set-up, kernel loads
        torch.cuda.synchronize()
        gc.collect()
        free0, _ = torch.cuda.mem_get_info()
        torch.cuda.reset_peak_memory_stats()
        torch_bytes0 = torch.cuda.memory_allocated()
        # two calls in a row on the shared scratch: nothing is allocated on the device, by the
        # driver or through torch's allocator (its peak stays where it was)
        for c in outs[1:]:
            dt.ag_gemm_static_scratch(shards, b, c, args)
            torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert torch.cuda.max_memory_allocated() == torch_bytes0
        assert dt.static_scratch_check() == (0, [0, 0, 0, 0])
        for c in outs:
            assert_close(to_f64(c), to_f64(want), "bf16", "fixed scratch vs workspace entry")
            assert bits_equal(c, want)


@pytest.mark.parametrize("backend", ["tma", "ldst"])
def test_static_scratch_reports_a_lost_chunk(dt, backend):
    """A chunk the host drops never lands: the bounded waits run out, the error stays in the
    fixed scratch until dt_static_scratch_check reads and clears it, and the next call on the
    same scratch gives the exact result."""
    import torch

    wl = WORKLOADS["ag_w2_m512_n512_k512"]
    inp = wl.make()
    args = dt.make_args(2, wl.m, wl.n, wl.k, rank=0, chunk_rows=wl.chunk_rows, backend=backend,
                        timeout_us=200_000)
    want = _reference_call(dt, inp, args, wl.m, wl.n)
    shards = [dev_bf16(s) for s in inp.shards]
    b = dev_bf16(inp.b)
    c = out_tensor(wl.m, wl.n, "bf16")
    dt.debug_drop_transfer(3)  # the second chunk of rank 1
    dt.ag_gemm_static_scratch(shards, b, c, args)
    st, info = dt.static_scratch_check()
    assert st == dt.capi.DT_ERR_TIMEOUT, (st, info)
    assert info[0] == 1  # a chunk's ready flag did not flip
    assert dt.static_scratch_check() == (0, [0, 0, 0, 0])  # read once, then cleared
    c2 = out_tensor(wl.m, wl.n, "bf16")
    dt.ag_gemm_static_scratch(shards, b, c2, args)
    torch.cuda.synchronize()
    assert dt.static_scratch_check()[0] == 0
    assert bits_equal(c2, want)


def test_static_scratch_rejects_problems_that_do_not_fit(dt):
    args = dt.make_args(8, 8192, 3584, 8192, chunk_rows=256, backend="tma")  # 128 MiB gather
    assert dt.workspace_size(args, dt.OP_AG) > dt.capi.STATIC_SCRATCH_BYTES
    with pytest.raises(dt.DtError) as ei:
        dt.ag_gemm_static_scratch([0] * 8, 0, 0, args)
    assert ei.value.status == dt.capi.DT_ERR_WORKSPACE
    assert "32 MiB" in ei.value.message
    ce = dt.make_args(2, 512, 512, 512, chunk_rows=128, backend="copy_engine")
    inp = WORKLOADS["ag_w2_m512_n512_k512"].make()
    with pytest.raises(dt.DtError) as ei:
        dt.ag_gemm_static_scratch([dev_bf16(s) for s in inp.shards], dev_bf16(inp.b),
                                  out_tensor(512, 512, "bf16"), ce)
    assert ei.value.status == dt.capi.DT_ERR_UNSUPPORTED
