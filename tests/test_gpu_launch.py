"""Launch mode of the fused kernel, and the AllGather's debug timeline, through the C ABI.

* Programmatic dependent launch (the fused kernel's launch and set-up overlap the prepare
  kernel before it; the kernel waits for that grid before it touches global memory) and the
  ReduceScatter's fold path (a middle source's TMA reduce-add into the running sum, or a load,
  an add and a store) and schedule (the rotation of the CTA pairs' slots per wave) change no
  bit: every op gives the same outputs by default, with DT_PDL=0 (plain stream order), with
  DT_RS_REDUCE=0 and with DT_ROT=0 or 7: the AllGather-GEMM on each transfer
  backend and on one CTA or a CTA pair per tile, the GEMM-ReduceScatter and GEMM-AllReduce
  (bf16 and fp32 outputs; six ranks whose tiles are cut by destination and chunk boundaries),
  the GEMM-AllToAll, the fixed-scratch AllGather-GEMM and dt_allgather.  The settings are read
  once per process, so each mode runs in a child process.  The DITRON page, section 6, asks for
  bit-identical results from the adapted kernels whatever their schedule.
* dt_allgather on an in-kernel backend records the timeline: every chunk is released inside
  the kernel's span, and no GEMM word is written.
"""
import json
import os
import subprocess
import sys

import pytest

from gpu_helpers import bits_equal, dev_bf16, load_dt, need_gpu, torch
from synth_inputs import make_ag_inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs every op once on seeded inputs and prints one JSON object: op name -> sha256 of its
# outputs' bytes (and the workspace status after the call).
CHILD = r"""
import hashlib, json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import tile_level_communication_gb300 as dt
from synth_inputs import make_ag_inputs, make_rs_inputs, make_a2a_inputs

def up(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

def digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.view(torch.int16).cpu().numpy().tobytes())
    return h.hexdigest()

res = {}
w, m, n, k = 4, 4 * 512, 1024, 1024
ag = make_ag_inputs(w, m, n, k, seed=71)
shards, b = [up(s) for s in ag.shards], up(ag.b)
for be in ("copy_engine", "tma", "ldst", "tma_tile"):
    for tm in (128, 256):
        a = dt.make_args(w, m, n, k, rank=1, chunk_rows=128, backend=be, tile_m=tm)
        ws = torch.zeros(dt.workspace_size(a, dt.OP_AG), dtype=torch.uint8, device="cuda")
        c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        for _ in range(2):
            dt.ag_gemm(shards, b, c, ws, a)
        res[f"ag/{be}/{tm}"] = [digest([c]), dt.check(ws)[0]]
a = dt.make_args(w, m, n, k, chunk_rows=128, backend="tma")
c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
dt.ag_gemm_static_scratch(shards, b, c, a)
res["ag/static"] = [digest([c]), dt.static_scratch_check()[0]]
for be in ("tma", "ldst"):
    a = dt.make_args(w, m, 8, k, chunk_rows=128, backend=be)
    ws = torch.zeros(dt.workspace_size(a, dt.OP_AG), dtype=torch.uint8, device="cuda")
    g = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    dt.allgather(shards, g, ws, a)
    res[f"allgather/{be}"] = [digest([g]), dt.check(ws)[0]]

rs = make_rs_inputs(w, 2048, 1024, 512, seed=72)
A, B = [up(x) for x in rs.a], [up(x) for x in rs.b]
for op, fn, rows in (("rs", dt.gemm_rs, 512), ("ar", dt.gemm_ar, 2048)):
    for odt in ("bf16", "f32"):
        a = dt.make_args(w, 2048, 1024, 512, chunk_rows=256, out_dtype=odt)
        opid = dt.OP_RS if op == "rs" else dt.OP_AR
        ws = torch.zeros(dt.workspace_size(a, opid), dtype=torch.uint8, device="cuda")
        tdt = torch.bfloat16 if odt == "bf16" else torch.float32
        outs = [torch.full((rows, 1024), float("nan"), dtype=tdt, device="cuda") for _ in range(w)]
        for _ in range(2):
            fn(A, B, outs, ws, a)
        res[f"{op}/{odt}"] = [digest([o.view(torch.int16) for o in outs]), dt.check(ws)[0]]
# six ranks, 200 rows each: 128-row tiles cut by destination and chunk boundaries, a ragged
# last tile, ragged columns
w6, m6, n6, k6 = 6, 1200, 600, 384
rs6 = make_rs_inputs(w6, m6, n6, k6, seed=75)
A6, B6 = [up(x) for x in rs6.a], [up(x) for x in rs6.b]
for tm in (128, 256):
    a = dt.make_args(w6, m6, n6, k6, chunk_rows=96, tile_m=tm)
    ws = torch.zeros(dt.workspace_size(a, dt.OP_RS), dtype=torch.uint8, device="cuda")
    outs = [torch.full((m6 // w6, n6), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(w6)]
    for _ in range(2):
        dt.gemm_rs(A6, B6, outs, ws, a)
    res[f"rs6/{tm}"] = [digest(outs), dt.check(ws)[0]]

a2 = make_a2a_inputs(w, 4 * 256, 4 * 256, 512, seed=73)
A, B = [up(x) for x in a2.a], [up(x) for x in a2.b]
a = dt.make_args(w, 1024, 1024, 512, chunk_rows=128)
ws = torch.zeros(dt.workspace_size(a, dt.OP_A2A), dtype=torch.uint8, device="cuda")
outs = [torch.full((1024, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        for _ in range(w)]
for _ in range(2):
    dt.gemm_a2a(A, B, outs, ws, a)
res["a2a"] = [digest(outs), dt.check(ws)[0]]
print(json.dumps(res))
"""


def _child(pdl, reduce=1, rot=1):
    env = dict(os.environ, DT_PDL=str(pdl), DT_RS_REDUCE=str(reduce), DT_ROT=str(rot))
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def dt():
    need_gpu()
    return load_dt()


def test_launch_mode_fold_path_and_schedule_change_no_bit(dt):
    base = _child(1)
    assert len(base) == 18
    for name, (_, st) in base.items():
        assert st == 0, (name, st)
    for other in (_child(0), _child(1, reduce=0), _child(1, rot=0), _child(1, rot=7)):
        assert other.keys() == base.keys()
        for name in base:
            assert other[name][1] == 0, (name, other[name])
            assert other[name][0] == base[name][0], name


@pytest.mark.parametrize("backend", ["tma", "ldst"])
def test_allgather_trace(dt, backend):
    w, ms, k = 8, 384, 1024
    inp = make_ag_inputs(w, w * ms, 8, k, seed=74)
    shards = [dev_bf16(s) for s in inp.shards]
    args = dt.make_args(w, w * ms, 8, k, chunk_rows=128, backend=backend)
    ws = torch.zeros(dt.workspace_size(args, dt.OP_AG), dtype=torch.uint8, device="cuda")
    base = torch.empty((w * ms, k), dtype=torch.bfloat16, device="cuda")
    dt.allgather(shards, base, ws, args)
    buf = torch.zeros(dt.trace_bytes(args) // 8, dtype=torch.int64, device="cuda")
    dt.trace_attach(buf)
    try:
        out = torch.empty((w * ms, k), dtype=torch.bfloat16, device="cuda")
        dt.allgather(shards, out, ws, args)
        assert dt.check(ws)[0] == 0
    finally:
        dt.trace_attach(None)
    assert bits_equal(out, base)
    assert bits_equal(out, torch.cat(shards))
    words = buf.cpu().tolist()
    tr = dt.trace_decode(words, args)
    assert tr["kernel_us"] is not None and tr["kernel_us"] > 0
    assert tr["stall_us_total"] == 0 and tr["stalled_waits"] == 0  # no GEMM waits
    assert len(tr["chunks"]) == w * 3
    for (s, j), ev in tr["chunks"].items():
        assert ev["released_us"] is not None, (s, j)
        assert 0 <= ev["released_us"] <= tr["kernel_us"], (s, j, ev)
        assert ev["first_read_us"] is None and ev["first_miss_us"] is None, (s, j, ev)
