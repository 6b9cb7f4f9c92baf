"""Full-size parity at the benchmark shapes, through the C ABI.

The FFN pair's GEMM-ReduceScatter (W=8, M=8192, N=8192, K=3584 per rank) and the largest
AllGather-GEMM (W=8, M=16384, N=8192, K=8192):

* every output entry is bit-identical across chunk rows, tile rows (one CTA or a CTA pair),
  swizzle on / off, for the ReduceScatter column bands and for the AllGather every transfer
  backend (DITRON page, section 6: the adapted kernels give bit-identical results);
* whole 128-row strips of every destination (ReduceScatter) or source block (AllGather), and
  one strip that crosses a block boundary, match the float64 oracle element by element within
  the bf16 tolerance.
"""
import numpy as np
import pytest

from gpu_helpers import assert_close, bits_equal, dev_bf16, load_dt, need_gpu, to_f64, torch
from oracle import reference
from synth_inputs import WORKLOADS, f64_from_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


# ----------------------------------------------------------------------------- ReduceScatter

RS_NAME = "rs_w8_m8192_n8192_k3584"
RS_VARIANTS = ([dict(chunk_rows=c, tile_m=t, swizzle=s)
                for c in (128, 256, 1024) for t in (128, 256) for s in (True, False)] +
               [dict(chunk_rows=c, col_band=nb) for c in (256, 1024) for nb in (3, 32)])


@pytest.fixture(scope="module")
def rs_full(dt):
    wl = WORKLOADS[RS_NAME]
    inp = wl.make()
    a = [dev_bf16(x) for x in inp.a]
    b = [dev_bf16(x) for x in inp.b]
    need = max(dt.workspace_size(dt.make_args(wl.world_size, wl.m, wl.n, wl.k, **v), dt.OP_RS)
               for v in RS_VARIANTS)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")

    def run(**kw):
        args = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, **kw)
        outs = [torch.full((wl.m // wl.world_size, wl.n), float("nan"), dtype=torch.bfloat16,
                           device="cuda") for _ in range(wl.world_size)]
        dt.gemm_rs(a, b, outs, ws, args)
        st, info = dt.check(ws)
        assert st == 0, info
        return outs

    base = run(chunk_rows=1024)
    return wl, inp, run, base


@pytest.mark.parametrize("variant", RS_VARIANTS,
                         ids=[f"c{v['chunk_rows']}-t{v.get('tile_m', 0)}-"
                              f"{'sw' if v.get('swizzle', True) else 'nosw'}-b{v.get('col_band', 0)}"
                              for v in RS_VARIANTS])
def test_rs_full_size_bit_identical_across_variants(rs_full, variant):
    wl, inp, run, base = rs_full
    outs = run(**variant)
    for s, (o, want) in enumerate(zip(outs, base)):
        assert bits_equal(o, want), (variant, s)


def _rs_strip(inp, rows):
    """Rows `rows` (global) of sum_q A_q @ B_q, from the oracle's definition: the ReduceScatter
    of the strip's rows over W ranks, its W destination blocks stacked back."""
    a = [f64_from_bf16_bits(x[rows]) for x in inp.a]
    b = [f64_from_bf16_bits(x) for x in inp.b]
    return np.vstack(reference.gemm_rs(a, b))


def test_rs_full_size_strips_match_oracle(rs_full):
    wl, inp, run, base = rs_full
    w, ms = wl.world_size, wl.m // wl.world_size
    rng = np.random.Generator(np.random.PCG64(21))
    got_all = [to_f64(o) for o in base]
    for s in range(w):
        r0 = int(rng.integers(0, ms // 128)) * 128  # a whole 128-row strip of destination s
        rows = np.arange(s * ms + r0, s * ms + r0 + 128)
        ref = _rs_strip(inp, rows)
        assert_close(got_all[s][r0:r0 + 128], ref, "bf16", f"destination {s} rows {r0}..")
    # a strip across the boundary of destinations 3 and 4 (64 rows of each)
    rows = np.arange(4 * ms - 64, 4 * ms + 64)
    ref = _rs_strip(inp, rows)
    got = np.vstack([got_all[3][ms - 64:], got_all[4][:64]])
    assert_close(got, ref, "bf16", "strip across destinations 3 / 4")


# ----------------------------------------------------------------------------- AllGather

AG_NAME = "ag_w8_m16384_n8192_k8192"
AG_VARIANTS = ([dict(chunk_rows=c, backend=be, tile_m=256, swizzle=True)
                for c in (128, 256, 1024) for be in ("copy_engine", "tma", "ldst")] +
               [dict(chunk_rows=c, backend="tma", tile_m=t, swizzle=s)
                for c in (256, 1024) for t in (128, 256) for s in (True, False)
                if (t, s) != (256, True)] +
               [dict(chunk_rows=c, backend="tma_tile", tile_m=t, swizzle=True)
                for c in (256, 2048) for t in (128, 256)] +
               [dict(chunk_rows=1024, backend=be, tile_m=256, swizzle=True, col_band=nb)
                for be in ("tma_tile", "copy_engine") for nb in (3, 32)])


@pytest.fixture(scope="module")
def ag_full(dt):
    wl = WORKLOADS[AG_NAME]
    inp = wl.make()
    shards = [dev_bf16(x) for x in inp.shards]
    b = dev_bf16(inp.b)
    need = max(dt.workspace_size(dt.make_args(wl.world_size, wl.m, wl.n, wl.k, **v), dt.OP_AG)
               for v in AG_VARIANTS)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")

    def run(rank=3, **kw):
        args = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, rank=rank, **kw)
        c = torch.full((wl.m, wl.n), float("nan"), dtype=torch.bfloat16, device="cuda")
        dt.ag_gemm(shards, b, c, ws, args)
        st, info = dt.check(ws)
        assert st == 0, info
        return c

    base = run(chunk_rows=2048, backend="copy_engine")
    return wl, inp, run, base


@pytest.mark.parametrize("variant", AG_VARIANTS,
                         ids=[f"c{v['chunk_rows']}-{v['backend']}-t{v['tile_m']}-"
                              f"{'sw' if v['swizzle'] else 'nosw'}-b{v.get('col_band', 0)}"
                              for v in AG_VARIANTS])
def test_ag_full_size_bit_identical_across_variants(ag_full, variant):
    wl, inp, run, base = ag_full
    assert bits_equal(run(**variant), base), variant


def test_ag_full_size_other_rank_views_identical(ag_full):
    """Every rank's view gathers the same rows into the same C."""
    wl, inp, run, base = ag_full
    for r in (0, 7):
        assert bits_equal(run(rank=r, chunk_rows=512, backend="tma"), base), r


def test_ag_full_size_strips_match_oracle(ag_full):
    wl, inp, run, base = ag_full
    w, ms = wl.world_size, wl.m // wl.world_size
    rng = np.random.Generator(np.random.PCG64(22))
    b = f64_from_bf16_bits(inp.b)
    strips = [(s * ms + int(rng.integers(0, ms // 128)) * 128, 128) for s in range(w)]
    strips.append((5 * ms - 64, 128))  # across the blocks of ranks 4 and 5
    for g0, nrows in strips:
        rows = np.arange(g0, g0 + nrows)
        # the oracle's definition on the strip's rows: concat of the row pieces, times B
        pieces, s0 = [], int(rows[0]) // ms
        for s in range(s0, int(rows[-1]) // ms + 1):
            lo = max(int(rows[0]), s * ms) - s * ms
            hi = min(int(rows[-1]) + 1, (s + 1) * ms) - s * ms
            pieces.append(f64_from_bf16_bits(inp.shards[s][lo:hi]))
        ref = reference.ag_gemm(pieces, b)
        got = to_f64(base[g0:g0 + nrows])
        assert_close(got, ref, "bf16", f"rows {g0}..{g0 + nrows}")
