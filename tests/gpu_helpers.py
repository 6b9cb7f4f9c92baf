"""Helpers of the GPU parity tests: device upload of the seeded bf16 inputs, oracle values
as float64, and the tolerance checks.

Tolerances: max |GPU - oracle| <= 1e-2 * max |oracle| for bf16 outputs and
<= 2e-3 * max |oracle| for fp32 outputs.  The bf16 bound covers the final round to bf16
(relative 2^-9 of each entry) plus fp32 accumulation over K of products that are exact in
fp32; the fp32 bound covers the accumulation alone with a wide margin.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

TOL = {"bf16": 1e-2, "f32": 2e-3}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def load_dt():
    from tile_level_communication_gb300 import build
    build.build()
    import tile_level_communication_gb300 as dt
    dt.capi.lib()
    return dt


def dev_bf16(bits: np.ndarray, ld: int = 0):
    """Upload uint16 bf16 patterns as a CUDA bf16 tensor; pad rows to `ld` elements."""
    rows, cols = bits.shape
    ld = ld or cols
    host = np.zeros((rows, ld), dtype=np.uint16)
    host[:, :cols] = bits
    t = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).cuda()
    return t


def to_f64(t, cols=None):
    x = t.float().cpu().numpy().astype(np.float64)
    return x if cols is None else x[:, :cols]


def assert_close(got, ref, out_dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err <= TOL[out_dtype] * max(scale, 1e-30), \
        f"{what}: max err {err:.4g} > {TOL[out_dtype]} * {scale:.4g}"


def bits_equal(x, y):
    """Bitwise equality of two CUDA tensors of the same dtype."""
    if x.dtype == torch.bfloat16:
        return torch.equal(x.view(torch.int16), y.view(torch.int16))
    return torch.equal(x.view(torch.int32), y.view(torch.int32))


def out_tensor(rows, cols, out_dtype, ld=0, fill=None):
    ld = ld or cols
    dt_ = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    t = torch.empty((rows, ld), dtype=dt_, device="cuda")
    t.fill_(float("nan") if fill is None else fill)
    return t


def workspace(nbytes):
    # 256-byte aligned by the CUDA caching allocator
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
