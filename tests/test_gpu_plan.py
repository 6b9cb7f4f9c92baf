"""The tile order evaluated by the device plan kernel equals the oracle's, bit for bit."""
import pytest

from gpu_helpers import load_dt, need_gpu, torch
from oracle import plan as oplan

pytestmark = pytest.mark.gpu

CASES = [(2, 512, 512, 128), (4, 2048, 4096, 256), (6, 6000, 3000, 192), (6, 6000, 5120, 192),
         (8, 8192, 3584, 256), (8, 8192, 8192, 256), (8, 16384, 8192, 64), (3, 390, 520, 50),
         (8, 80, 64, 4), (16, 4096, 512, 100)]


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("bm", [128, 256])
def test_device_plan_matches_oracle(dt, case, swizzle, bm):
    w, m, n, cr = case
    for r in sorted({0, 1 % w, w - 1}):
        a = dt.make_args(w, m, n, 8, rank=r, chunk_rows=cr, swizzle=swizzle, tile_m=bm)
        t = dt.tile_count(a, dt.OP_AG)
        buf = torch.full((t,), -1, dtype=torch.int32, device="cuda")
        dt.swizzle_plan_device(a, dt.OP_AG, buf)
        assert buf.cpu().tolist() == oplan.ag_order(w, r, m, n, cr, bm, 256, swizzle)
    a = dt.make_args(w, m, n, 8, chunk_rows=cr, swizzle=swizzle, tile_m=bm)
    t = dt.tile_count(a, dt.OP_RS)
    buf = torch.full((t,), -1, dtype=torch.int32, device="cuda")
    dt.swizzle_plan_device(a, dt.OP_RS, buf)
    assert buf.cpu().tolist() == oplan.rs_order(w, m, n, cr, bm, 256, swizzle)
    for nb in (1, 3, 5):  # column bands
        a = dt.make_args(w, m, n, 8, chunk_rows=cr, swizzle=swizzle, tile_m=bm, col_band=nb)
        buf.fill_(-1)
        dt.swizzle_plan_device(a, dt.OP_RS, buf)
        assert buf.cpu().tolist() == oplan.rs_order(w, m, n, cr, bm, 256, swizzle, col_band=nb)
        r = w - 1
        a = dt.make_args(w, m, n, 8, rank=r, chunk_rows=cr, swizzle=swizzle, tile_m=bm,
                         col_band=nb)
        t = dt.tile_count(a, dt.OP_AG)
        abuf = torch.full((t,), -1, dtype=torch.int32, device="cuda")
        dt.swizzle_plan_device(a, dt.OP_AG, abuf)
        assert abuf.cpu().tolist() == oplan.ag_order(w, r, m, n, cr, bm, 256, swizzle, col_band=nb)
    if n % (8 * w) == 0:  # the AllToAll over the same rows, each rank's M/W of them
        a = dt.make_args(w, m, n, 8, chunk_rows=cr, swizzle=swizzle, tile_m=bm)
        t = dt.tile_count(a, dt.OP_A2A)
        buf = torch.full((t,), -1, dtype=torch.int32, device="cuda")
        dt.swizzle_plan_device(a, dt.OP_A2A, buf)
        assert buf.cpu().tolist() == oplan.a2a_order(w, m // w, n, cr, bm, 256, swizzle)
