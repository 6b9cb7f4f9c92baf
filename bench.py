#!/usr/bin/env python
"""Benchmark of the chunk-centric fused AllGather-GEMM + GEMM-ReduceScatter on GB300.

One step is one pass of the whole hot path over one batch of synthetic input: the
Llama-70B-like tensor-parallel (W=8) FFN pair -- a fused AllGather-GEMM (gathered M=8192,
K=8192, N=3584; chunk transfer, ready flags, swizzled persistent tcgen05 GEMM) followed by
a fused GEMM-ReduceScatter over all 8 virtual ranks (M=8192, K=3584 per rank, N=8192;
the ranks one after another in their scatter order, each tile's fp32 partial folded into its
unit's running sum in source order).  Other workloads: --workload <name> from
synth_inputs.WORKLOADS (one operation per step); --allgather-only times the chunk transfer
alone; --sweep and --ffn-crossover print one line per point.

Prints one JSON line (rank 0).  --impl reference times the float64 CPU oracle on a bounded
row sample of the same workload instead.  Under torchrun every GPU runs an independent
replica (weak scaling); there is no data-path collective.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# one hardware work queue per stream (the default of 8 is shared out round robin, and a copy
# stream that shares a queue with the compute stream waits behind its kernels); read when the
# CUDA context is created, so set before any CUDA call
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

import numpy as np  # noqa: E402

from synth_inputs import WORKLOADS, f64_from_bf16_bits  # noqa: E402

METRIC = "fused AG-GEMM / GEMM-RS TFLOP/s and % of GB300 bf16 tensor peak (1 GPU)"

# Recorded DRAM bytes (read + write) of one launch of the dominant kernel: figures copied from
# earlier `ncu` captures (the profile named beside each workload), not measured by this run.
# They hold only for the kernel sources they were taken on (csrc hash) and the knobs
# "chunk_rows/group/tile_rows"; otherwise the roofline's traffic is null.
NCU_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (one pass), one launch after two
    # warm-up launches, 256-row tiles; keys "chunk_rows/tile_rows/col_band/l2_hints" (the
    # group width gives the same order at these chunk sizes: a key holds at most 4 m-tiles)
    "rs_w8_m8192_n8192_k3584": {"csrc": "719259b6f03ac510",
                                "profile": "profiles/fused_gemm_rs_w8_m8192_n8192_k3584.md",
                                "points": {
        "1024/256/16/3": 3936388352 + 1991550720, "1024/256/32/3": 5236883968 + 1993030400,
        "512/256/16/3": 3808375552 + 1991179008, "512/256/32/3": 5351156736 + 1995966976,
        "256/256/16/3": 4036418816 + 1993510144, "256/256/32/3": 5534166784 + 1998488832,
        "128/256/16/3": 4168581376 + 1993465600, "128/256/32/3": 5486107904 + 1998518016,
        "64/256/16/3": 3797574400 + 1990460160, "64/256/32/3": 5485989632 + 1996728320,
    }},
}


# the sources that make up the fused kernel and its launch (device code, plan, launchers); the
# host-side API, tuner and workspace code are not part of what an ncu capture measures
KERNEL_SOURCES = ("dt_kernel.cuh", "dt_ptx.cuh", "dt_plan.cuh", "dt_internal.h", "dt_ag.cu",
                  "dt_rs.cu", "dt_a2a.cu")


def csrc_hash():
    """Hash of the kernel sources' code: comments and whitespace do not count."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        with open(os.path.join(ROOT, "tile_level_communication_gb300", "csrc", name)) as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]
FFN_PAIR = ("ag_w8_m8192_n3584_k8192", "rs_w8_m8192_n8192_k3584")
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000,
                    help="timed steps; >= 2 s of them is measured against the sustained peak")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fused", choices=["fused", "reference"])
    ap.add_argument("--workload", default="ffn_pair")
    ap.add_argument("--backend", default="auto", choices=["auto", "copy_engine", "tma", "ldst", "tma_tile"])
    ap.add_argument("--chunk-rows", type=int, default=0, help="0 = the workload's")
    ap.add_argument("--no-swizzle", action="store_true")
    ap.add_argument("--group", type=int, default=0, help="m-tiles per band of the in-chunk "
                    "raster (0 = the library's 8; fixed, not tuned, when given)")
    ap.add_argument("--tile-m", type=int, default=0, choices=[0, 128, 256],
                    help="tile rows: 128 (one CTA), 256 (a CTA pair), 0 = the library's choice")
    ap.add_argument("--col-band", type=int, default=0,
                    help="ReduceScatter / AllReduce column tiles per column band (0 = the "
                         "library's automatic choice)")
    ap.add_argument("--rank-view", type=int, default=0, help="AllGather rank whose view is computed")
    ap.add_argument("--skip-extras", action="store_true",
                    help="skip the baselines, e2e, CPU oracle and clock sampling")
    ap.add_argument("--no-tune", action="store_true",
                    help="skip the enumerate-and-measure tuner and use the workload's knobs")
    ap.add_argument("--sweep", action="store_true",
                    help="AllGather chunk x backend x swizzle sweep of --workload (default: the "
                         "largest AllGather); one JSON line per point")
    ap.add_argument("--sweep-chunks", default="64,128,256,512,2048")
    ap.add_argument("--sweep-rounds", type=int, default=5,
                    help="rounds over all sweep points (each point's median is reported)")
    ap.add_argument("--allgather-only", action="store_true",
                    help="time the AllGather's chunk transfer alone (dt_allgather) on the shards "
                         "of --workload's AllGather, per backend (or --backend), L2 flushed by "
                         "reading before each call; one JSON line per backend")
    ap.add_argument("--ffn-crossover", action="store_true",
                    help="time the feed-forward block in AllGather+ReduceScatter form and in "
                         "AllReduce form over a range of token counts M (one JSON line per M)")
    return ap.parse_args()


def workload_ops(name):
    if name == "ffn_pair":
        return [WORKLOADS[FFN_PAIR[0]], WORKLOADS[FFN_PAIR[1]]]
    return [WORKLOADS[name]]


def workload_desc(name, ops, chunk_override):
    d = {"workload": name if name != "ffn_pair" else
         "llama70b_like_tp8_ffn_pair (AG-GEMM then GEMM-RS, W=8 virtual ranks)"}
    for wl in ops:
        if wl.op == "ffn":
            d["ffn"] = {"name": wl.name, "world_size": wl.world_size, "m": wl.m, "k": wl.k,
                        "f_per_rank": wl.f_rank, "n": wl.n, "act": wl.act, "seed": wl.seed,
                        "chunk_rows": chunk_override or wl.chunk_rows, "gflop": wl.flops / 1e9,
                        "dist_x": wl.dist_a, "dist_w": wl.dist_b}
            continue
        d[wl.op] = {"name": wl.name, "world_size": wl.world_size, "m": wl.m, "n": wl.n,
                    "k" if wl.op in ("ag", "a2a") else "k_per_rank": wl.k,
                    "chunk_rows": chunk_override or wl.chunk_rows, "seed": wl.seed,
                    "dist_a": wl.dist_a, "dist_b": wl.dist_b, "gflop": wl.flops / 1e9}
    return d


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as tdist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group("gloo", rank=rank, world_size=world)
        pg = tdist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(ops, ag_rows, rs_rows, inputs):
    """Time the float64 oracle on a row sample: returns (flops, seconds, description)."""
    from oracle import reference
    flops = 0.0
    secs = 0.0
    desc = []
    for wl, inp in zip(ops, inputs):
        ms = wl.m // wl.world_size
        if wl.op == "ffn":
            # the block is row-independent: run it on the first rows, split over W ranks
            w = wl.world_size
            rows = max(w, min(rs_rows, wl.m) // w * w)
            x = np.concatenate([f64_from_bf16_bits(sh) for sh in inp.x_shards])[:rows]
            pieces = [x[q * rows // w:(q + 1) * rows // w] for q in range(w)]
            w1 = f64_from_bf16_bits(inp.w1)
            w2 = [f64_from_bf16_bits(t) for t in inp.w2]
            t0 = time.perf_counter()
            reference.ffn_tp(pieces, w1, w2, wl.act)
            secs += time.perf_counter() - t0
            flops += 2.0 * rows * w * wl.f_rank * (wl.k + wl.n)
            desc.append(f"FFN block on rows 0..{rows}")
            continue
        if wl.op == "a2a":
            # the first r rows of every rank, all W destinations
            w = wl.world_size
            r = max(1, min(rs_rows, wl.m) // w)
            a = [f64_from_bf16_bits(x[:r]) for x in inp.a]
            b = [f64_from_bf16_bits(inp.b[0])] * w
            t0 = time.perf_counter()
            reference.gemm_a2a(a, b)
            secs += time.perf_counter() - t0
            flops += 2.0 * w * r * wl.n * wl.k
            desc.append(f"A2A rows 0..{r} of every rank, all destinations")
            continue
        if wl.op == "ag":
            rows = min(ag_rows, wl.m)
            nsh = -(-rows // ms)
            shards = [f64_from_bf16_bits(inp.shards[s]) for s in range(nsh)]
            b = f64_from_bf16_bits(inp.b)
            t0 = time.perf_counter()
            reference.ag_gemm(shards, b)
            secs += time.perf_counter() - t0
            flops += 2.0 * nsh * ms * wl.n * wl.k
            desc.append(f"AG rows 0..{nsh * ms} of C")
        else:
            rows = min(rs_rows, wl.m)
            rows = max(wl.world_size, rows - rows % wl.world_size)
            a = [f64_from_bf16_bits(x[:rows]) for x in inp.a]
            b = [f64_from_bf16_bits(x) for x in inp.b]
            t0 = time.perf_counter()
            reference.gemm_rs(a, b)
            secs += time.perf_counter() - t0
            flops += 2.0 * rows * wl.n * wl.k * wl.world_size
            desc.append(f"RS rows 0..{rows} of sum_q A_q B_q ({wl.world_size} partials)")
    return flops, secs, "; ".join(desc)


def run_reference(args):
    world, rank, local, pg = dist_setup(args.gpus)
    if rank != 0:
        return 0
    ops = workload_ops(args.workload)
    inputs = [wl.make() for wl in ops]
    ag_rows, rs_rows = 256, 128
    for _ in range(args.warmup):
        oracle_sample(ops, ag_rows, rs_rows, inputs)
    flops = secs = 0.0
    desc = ""
    for _ in range(args.steps):
        f, s, desc = oracle_sample(ops, ag_rows, rs_rows, inputs)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_desc(args.workload, ops, args.chunk_rows),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id):
        self.device_id = device_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.device_id), "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:], float(parts[4])))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed region"
        if len(inside) < 3:  # short region: widen to the samples around it (under load)
            inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 0.2]
            window = "timed region +-1 s (region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in inside:
            for nm, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window,
                "power_w_max": max(r[4] for r in inside)}


# ----------------------------------------------------------------------------- peaks
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p["bf16_tflops_sustained"],
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- sweep
def run_sweep(args):
    """Chunk rows x transfer backend x swizzle on one AllGather workload (config 5 of the
    benchmark plan): inputs generated and uploaded once, every point warmed up, then timed
    (--steps calls back to back) once in each of --sweep-rounds interleaved rounds."""
    import torch

    import tile_level_communication_gb300 as dt
    name = args.workload if args.workload != "ffn_pair" else "ag_w8_m16384_n8192_k8192"
    wl = WORKLOADS[name]
    if wl.op != "ag":
        raise SystemExit("--sweep takes an AllGather workload")
    inp = wl.make()
    up = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    shards = [up(x) for x in inp.shards]
    b = up(inp.b)
    c = torch.empty((wl.m, wl.n), dtype=torch.bfloat16, device="cuda")
    peak = peaks()["bf16_tflops"]
    chunks = [int(x) for x in args.sweep_chunks.split(",")]
    ws = None
    backends = ["copy_engine", "tma", "ldst"]
    if (wl.m // wl.world_size) % 128 == 0:
        backends.append("tma_tile")  # the per-tile pull needs tile-aligned shards
    # every point is timed once per round and the rounds interleave the points, so that the
    # GPU's drift in clock and power over the sweep falls on every point alike; each point
    # reports the median of its rounds
    points = []
    for cr in chunks:
        for backend in backends:
            for swizzle in [True, False]:
                a = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, rank=args.rank_view,
                                 chunk_rows=cr, swizzle=swizzle, backend=backend)
                need = dt.workspace_size(a, dt.OP_AG)
                if ws is None or ws.numel() < need:
                    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
                points.append(dict(chunk_rows=cr, backend=backend, swizzle=swizzle, args=a, ms=[]))
    for p in points:
        for _ in range(max(3, args.warmup)):
            dt.ag_gemm(shards, b, c, ws, p["args"])
    for _ in range(args.sweep_rounds):
        for p in points:
            dt.ag_gemm(shards, b, c, ws, p["args"])  # its order and flags in the workspace
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(args.steps):
                dt.ag_gemm(shards, b, c, ws, p["args"])
            e1.record()
            torch.cuda.synchronize()
            p["ms"].append(e0.elapsed_time(e1) / args.steps)
    st, info = dt.check(ws)
    if st != 0:
        raise RuntimeError(f"device error in the sweep {info}")
    for p in points:
        ms = statistics.median(p["ms"])
        tf = wl.flops / (ms * 1e-3) / 1e12
        print(json.dumps({"sweep": name, "chunk_rows": p["chunk_rows"], "backend": p["backend"],
                          "swizzle": p["swizzle"], "ms": ms, "ms_rounds": p["ms"], "tflops": tf,
                          "frac_of_burst_peak": tf / peak}), flush=True)
    return 0


# ----------------------------------------------------------------------------- FFN forms
def run_ffn_crossover(args):
    """The Llama-70B-like TP=8 feed-forward block (K=8192, F=8x3584, N=8192, GELU) for several
    token counts M, in its two tensor-parallel forms (DITRON page, section 5.1, FFN module):
    AG+RS: sequence-sharded X is gathered, out is reduce-scattered (dt_ffn_ag_rs);
    AR:    X is replicated, H = act(X W1) needs no communication, out is all-reduced
           (GEMM then dt_gemm_ar), with W output copies, or one shared output buffer."""
    import torch

    import tile_level_communication_gb300 as dt
    from synth_inputs import make_ffn_inputs
    w, k, fr, n = 8, 8192, 3584, 8192
    ms_list = [1024, 2048, 4096, 8192, 16384]
    inp = make_ffn_inputs(w, max(ms_list), k, fr, n, seed=2)
    up = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    x_all = up(np.concatenate(inp.x_shards))
    w1 = up(inp.w1)
    w2 = [up(t) for t in inp.w2]
    peak = peaks()["bf16_tflops_sustained"]

    def timed(fn, reps):
        for _ in range(max(3, args.warmup)):  # order and tensor maps prepared, clocks up
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    # the GPU sat idle while the inputs were drawn: bring its clocks up before the first size
    spin = torch.empty((8192, 8192), dtype=torch.bfloat16, device="cuda").normal_()
    t_end = time.time() + 0.3
    while time.time() < t_end:
        torch.matmul(spin, spin)
        torch.cuda.synchronize()
    del spin
    for m in ms_list:
        x = x_all[:m]
        ms_ = m // w
        flops = 2.0 * m * w * fr * (k + n)
        cr = max(ms_ // 1, 1)
        h = torch.empty((m, w * fr), dtype=torch.bfloat16, device="cuda")
        # AG + RS
        ag = dt.make_args(w, m, w * fr, k, chunk_rows=cr, act="gelu_tanh")
        rs = dt.make_args(w, m, n, fr, chunk_rows=cr, lda=w * fr)
        ws_ag = torch.zeros(dt.workspace_size(ag, dt.OP_AG), dtype=torch.uint8, device="cuda")
        ws_rs = torch.zeros(dt.workspace_size(rs, dt.OP_RS), dtype=torch.uint8, device="cuda")
        shards = [x[q * ms_:(q + 1) * ms_] for q in range(w)]
        outs_rs = [torch.empty((ms_, n), dtype=torch.bfloat16, device="cuda") for _ in range(w)]
        t_agrs = timed(lambda: dt.ffn_ag_rs(shards, w1, w2, h, outs_rs, ws_ag, ws_rs, ag, rs),
                       args.steps)
        # AR: replicated X, plain GEMM with the activation, then GEMM-AllReduce
        g1 = dt.make_args(1, m, w * fr, k, chunk_rows=m, act="gelu_tanh")
        ws_g1 = torch.zeros(dt.workspace_size(g1, dt.OP_AG), dtype=torch.uint8, device="cuda")
        ar = dt.make_args(w, m, n, fr, chunk_rows=cr, lda=w * fr)
        ws_ar = torch.zeros(dt.workspace_size(ar, dt.OP_AR), dtype=torch.uint8, device="cuda")
        a_blocks = [h[:, q * fr:(q + 1) * fr] for q in range(w)]
        outs_ar = [torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(w)]
        shared = [outs_ar[0]] * w

        def ar_form(outs):
            dt.ag_gemm([x], w1, h, ws_g1, g1)
            dt.gemm_ar(a_blocks, w2, outs, ws_ar, ar)
        t_ar = timed(lambda: ar_form(outs_ar), args.steps)
        t_ar1 = timed(lambda: ar_form(shared), args.steps)
        for ws in (ws_ag, ws_rs, ws_g1, ws_ar):
            if dt.check(ws)[0] != 0:
                raise RuntimeError("device error in the crossover run")
        print(json.dumps({"ffn_crossover_m": m, "gflop": flops / 1e9,
                          "ag_rs_ms": t_agrs, "ar_copies_ms": t_ar, "ar_shared_ms": t_ar1,
                          "ag_rs_tflops": flops / t_agrs / 1e9,
                          "ar_shared_tflops": flops / t_ar1 / 1e9,
                          "ag_rs_frac_of_sustained_peak": flops / t_agrs / 1e9 / peak}),
              flush=True)
        del h, ws_ag, ws_rs, ws_g1, ws_ar, outs_rs, outs_ar, shared, a_blocks
        torch.cuda.empty_cache()
    return 0


def run_allgather_only(args):
    """The copy path alone: every shard of the AllGather's workload gathered into one [M, K]
    buffer by dt_allgather; 2 x bytes (read + write) over the time per call."""
    import statistics

    import torch

    import tile_level_communication_gb300 as dt
    ag = [wl for wl in workload_ops(args.workload) if wl.op in ("ag", "ffn")]
    if not ag:
        raise SystemExit("--allgather-only takes a workload with an AllGather")
    wl = ag[0]
    inp = wl.make()
    up = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    shards = [up(x) for x in (inp.x_shards if wl.op == "ffn" else inp.shards)]
    m, k = sum(t.shape[0] for t in shards), shards[0].shape[1]
    out = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    flush = torch.zeros(2 * L2_BYTES // 8, dtype=torch.int64, device="cuda")
    hbm = peaks()["hbm_gbs"]
    cr = args.chunk_rows or wl.chunk_rows
    for be in ([args.backend] if args.backend != "auto" else ["copy_engine", "tma", "ldst"]):
        a = dt.make_args(wl.world_size, m, 8, k, chunk_rows=cr, backend=be)
        ws = torch.zeros(dt.workspace_size(a, dt.OP_AG), dtype=torch.uint8, device="cuda")
        for _ in range(max(3, args.warmup)):
            dt.allgather(shards, out, ws, a)
        times = []
        for _ in range(args.steps):
            torch.amax(flush)  # reads twice L2's size: evicts the shards, leaves clean lines
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            dt.allgather(shards, out, ws, a)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        st, info = dt.check(ws)
        if st != 0:
            raise RuntimeError(f"AllGather device error {info}")
        if not torch.equal(out.view(torch.int16), torch.cat(shards).view(torch.int16)):
            raise RuntimeError("AllGather result differs from the shards")
        ms = statistics.median(times)
        gbs = 2 * m * k * 2 / (ms * 1e-3) / 1e9
        print(json.dumps({"allgather": wl.name, "bytes": m * k * 2, "chunk_rows": cr,
                          "backend": be, "ms": ms, "gbs": gbs, "frac_of_hbm_copy": gbs / hbm}),
              flush=True)
    return 0


# ----------------------------------------------------------------------------- fused arm
class Arena:
    """One flat device buffer handing out consecutive 256-byte-aligned bf16 tensors: the
    step's inputs (or outputs) then cross the host link as one copy."""
    ALIGN = 256

    def __init__(self, capacity, dev):
        import torch
        self.buf = torch.empty(capacity, dtype=torch.uint8, device=dev)
        self.used = 0

    def take(self, shape):
        import torch
        n = int(np.prod(shape)) * 2
        if self.used + n > self.buf.numel():
            raise RuntimeError("arena too small")
        t = self.buf[self.used:self.used + n].view(torch.bfloat16).view(*shape)
        self.used += -(-n // self.ALIGN) * self.ALIGN
        return t

    def put(self, bits):
        import torch
        t = self.take(bits.shape)
        t.copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
        return t

    def span(self, t):
        """Byte range of tensor `t` (one of this arena's) inside the buffer."""
        lo = t.data_ptr() - self.buf.data_ptr()
        return lo, lo + t.numel() * t.element_size()

    @staticmethod
    def capacity(arrays):
        return sum(-(-a.nbytes // Arena.ALIGN) * Arena.ALIGN for a in arrays)


def _input_arrays(inp):
    """Every array a workload's inputs hold (an upper bound on what the step uploads)."""
    out = []
    for v in vars(inp).values():
        if isinstance(v, np.ndarray):
            out.append(v)
        elif isinstance(v, (list, tuple)):
            out.extend(x for x in v if isinstance(x, np.ndarray))
    return out


def _output_bytes(wl):
    """Bytes of a step's outputs for one workload, padded per output tensor."""
    w = wl.world_size
    pad = Arena.ALIGN * (w + 1)
    if wl.op == "ar":
        return w * wl.m * wl.n * 2 + pad
    return wl.m * wl.n * 2 + pad  # ag: C; rs: the W row blocks; a2a: the W column blocks; ffn: out_s


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.ffn_crossover:
        return run_ffn_crossover(args)
    if args.allgather_only:
        return run_allgather_only(args)
    import torch

    import tile_level_communication_gb300 as dt

    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ops = workload_ops(args.workload)
    inputs = [wl.make() for wl in ops]

    # device-resident inputs, outputs, workspaces, argument structs
    knobs = {"tile_m": args.tile_m, "col_band": args.col_band}
    if args.group:
        knobs["group"] = args.group
    in_capacity = sum(Arena.capacity(_input_arrays(inp)) for inp in inputs)
    out_capacity = sum(_output_bytes(wl) for wl in ops)

    def build_calls():
        """One set of device-resident inputs, outputs, workspaces and argument structs; the
        inputs sit back to back in one arena and the outputs in another (`arenas`)."""
        in_arena, out_arena = Arena(in_capacity, dev), Arena(out_capacity, dev)
        up = in_arena.put
        out = out_arena.take
        calls = []
        in_bytes = out_bytes = 0
        for wl, inp in zip(ops, inputs):
            cr = args.chunk_rows or wl.chunk_rows
            if wl.op == "ffn":
                # chained block: AllGather-GEMM (+ activation) into H, GEMM-ReduceScatter reads H
                import dataclasses
                w, fr = wl.world_size, wl.f_rank
                ag_wl = dataclasses.replace(wl, name=wl.name + "/ag", op="ag", n=w * fr)
                rs_wl = dataclasses.replace(wl, name=wl.name + "/rs", op="rs", k=fr)
                x = [up(s_) for s_ in inp.x_shards]
                w1 = up(inp.w1)
                h = torch.empty((wl.m, w * fr), dtype=torch.bfloat16, device=dev)
                a_ag = dt.make_args(w, wl.m, w * fr, wl.k, chunk_rows=cr, act=wl.act,
                                    swizzle=not args.no_swizzle, backend=args.backend, **knobs)
                probe = dt.make_args(w, wl.m, w * fr, wl.k, chunk_rows=64)
                ws_ag = torch.zeros(max(dt.workspace_size(a_ag, dt.OP_AG),
                                        dt.workspace_size(probe, dt.OP_AG)), dtype=torch.uint8, device=dev)
                calls.append(dict(op="ag", wl=ag_wl, args=a_ag, ins=x + [w1], acts=x, shards=x, b=w1, outs=[h],
                                  ws=ws_ag, act=wl.act))
                w2 = [up(t) for t in inp.w2]
                a_rs = dt.make_args(w, wl.m, wl.n, fr, chunk_rows=cr, lda=w * fr,
                                    swizzle=not args.no_swizzle, **knobs)
                probe = dt.make_args(w, wl.m, wl.n, fr, chunk_rows=64, lda=w * fr)
                ws_rs = torch.zeros(max(dt.workspace_size(a_rs, dt.OP_RS),
                                        dt.workspace_size(probe, dt.OP_RS)), dtype=torch.uint8, device=dev)
                outs = [out((wl.m // w, wl.n)) for _ in range(w)]
                calls.append(dict(op="rs", wl=rs_wl, args=a_rs, ins=w2, acts=[],
                                  A=[h[:, q * fr:(q + 1) * fr] for q in range(w)], B=w2, outs=outs,
                                  ws=ws_rs))
                in_bytes += sum(t.numel() * 2 for t in x + [w1] + w2)
                out_bytes += sum(t.numel() * 2 for t in outs)
                continue
            if wl.op == "ag":
                a = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, rank=args.rank_view, chunk_rows=cr,
                                 swizzle=not args.no_swizzle, backend=args.backend, **knobs)
                shards = [up(s) for s in inp.shards]
                b = up(inp.b)
                c = out((wl.m, wl.n))
                probe = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, chunk_rows=64)
                need = max(dt.workspace_size(a, dt.OP_AG), dt.workspace_size(probe, dt.OP_AG))
                ws = torch.zeros(need, dtype=torch.uint8, device=dev)
                calls.append(dict(op="ag", wl=wl, args=a, ins=shards + [b], acts=shards, shards=shards, b=b,
                                  outs=[c], ws=ws))
            elif wl.op == "a2a":
                w = wl.world_size
                a = dt.make_args(w, wl.m, wl.n, wl.k, chunk_rows=cr, swizzle=not args.no_swizzle,
                                 **knobs)
                A = [up(x) for x in inp.a]
                b = up(inp.b[0])  # the replicated weight, held once
                outs = [out((wl.m, wl.n // w)) for _ in range(w)]
                y = [torch.empty((wl.m // w, wl.n), dtype=torch.bfloat16, device=dev)
                     for _ in range(w)]  # the baseline's per-rank GEMM outputs
                probe = dt.make_args(w, wl.m, wl.n, wl.k, chunk_rows=64)
                need = max(dt.workspace_size(a, dt.OP_A2A), dt.workspace_size(probe, dt.OP_A2A))
                ws = torch.zeros(need, dtype=torch.uint8, device=dev)
                calls.append(dict(op="a2a", wl=wl, args=a, ins=A + [b], acts=A, A=A, B=[b] * w, outs=outs,
                                  y=y, ws=ws))
            else:
                a = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, chunk_rows=cr,
                                 swizzle=not args.no_swizzle, **knobs)
                A = [up(x) for x in inp.a]
                B = [up(x) for x in inp.b]
                rows = wl.m // wl.world_size if wl.op == "rs" else wl.m  # AllReduce: every rank all rows
                outs = [out((rows, wl.n)) for _ in range(wl.world_size)]
                op_id = dt.OP_RS if wl.op == "rs" else dt.OP_AR
                probe = dt.make_args(wl.world_size, wl.m, wl.n, wl.k, chunk_rows=64)
                need = max(dt.workspace_size(a, op_id), dt.workspace_size(probe, op_id))
                ws = torch.zeros(need, dtype=torch.uint8, device=dev)
                calls.append(dict(op=wl.op, wl=wl, args=a, ins=A + B, acts=A, A=A, B=B, outs=outs, ws=ws))
            in_bytes += sum(t.numel() * 2 for t in calls[-1]["ins"])
            out_bytes += sum(t.numel() * 2 for t in calls[-1]["outs"])
        return calls, in_bytes, out_bytes, (in_arena, out_arena)

    calls, in_bytes, out_bytes, arenas = build_calls()

    def run_call(cl, fused=True):
        if cl["op"] == "ag":
            fn = dt.ag_gemm if fused else dt.ag_gemm_kernel_overlap
            fn(cl["shards"], cl["b"], cl["outs"][0], cl["ws"],
               cl["args"] if fused else cl.get("base_args", cl["args"]))
        elif cl["op"] == "rs":
            fn = dt.gemm_rs if fused else dt.gemm_rs_kernel_overlap
            fn(cl["A"], cl["B"], cl["outs"], cl["ws"], cl["args"])
        elif cl["op"] == "a2a":
            if fused:
                dt.gemm_a2a(cl["A"], cl["B"], cl["outs"], cl["ws"], cl["args"])
            else:
                dt.gemm_a2a_kernel_overlap(cl["A"], cl["B"], cl["y"], cl["outs"], cl["ws"],
                                           cl["args"])
        else:
            fn = dt.gemm_ar if fused else dt.gemm_ar_kernel_overlap
            fn(cl["A"], cl["B"], cl["outs"], cl["ws"], cl["args"])

    flops_step = sum(cl["wl"].flops for cl in calls)
    stream = torch.cuda.current_stream(dev)

    # enumerate-and-measure tuning of every call's knobs (not timed)
    tuned = {}
    if not args.no_tune and args.chunk_rows == 0 and args.backend == "auto" and not args.group:
        for cl in calls:
            if cl["op"] == "ag":
                pts = dt.tune_ag_gemm(cl["shards"], cl["b"], cl["outs"][0], cl["ws"], cl["args"],
                                      reps=8)
            else:
                op_id = {"rs": dt.OP_RS, "ar": dt.OP_AR, "a2a": dt.OP_A2A}[cl["op"]]
                pts = dt.tune_reduce(op_id, cl["A"], cl["B"], cl["outs"], cl["ws"], cl["args"],
                                     reps=16)
            a = cl["args"]
            tuned[cl["op"]] = {"chunk_rows": int(a.chunk_rows),
                               "backend": [k for k, v in dt.BACKENDS.items() if v == a.backend][0],
                               "copy_ctas": int(a.copy_ctas), "group": int(a.group),
                               "tile_m": int(a.tile_m), "col_band": int(a.col_band),
                               "candidates": len(pts),
                               "fastest": sorted(({k: p[k] for k in ("chunk_rows", "backend",
                                                                     "group", "col_band", "ms")}
                                                  for p in pts if p["status"] == 0 and p["ms"] > 0),
                                                 key=lambda x: x["ms"])[:4]}

    # warm-up (also writes each workspace's tile order once)
    for _ in range(max(3, args.warmup)):
        for cl in calls:
            run_call(cl)
    for cl in calls:
        st, info = dt.check(cl["ws"])
        if st != 0:
            raise RuntimeError(f"device error during warm-up: {info}")

    sampler = None if args.skip_extras else ClockSampler(local)
    if sampler:
        sampler.start()
        time.sleep(0.3)
        for _ in range(3):  # keep the GPU loaded while the sampler starts
            for cl in calls:
                run_call(cl)
    # per-call events: [start, end] per op per step on the launching stream
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in calls] for _ in range(args.steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize(dev)
    gc.disable()  # a collector pause on the host would leave the GPU idle (as timeit does)
    w0 = time.time()
    ev0.record(stream)
    for s in range(args.steps):
        for j, cl in enumerate(calls):
            evs[s][j][0].record(stream)
            run_call(cl)
            evs[s][j][1].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    gc.enable()
    barrier(pg)
    if sampler:
        sampler.stop()
    for cl in calls:
        st, info = dt.check(cl["ws"])
        if st != 0:
            raise RuntimeError(f"device error in the timed region: {info}")
    t_ms = ev0.elapsed_time(ev1)
    t_max = max_over_ranks(pg, t_ms)
    per_call_ms = [statistics.mean(evs[s][j][0].elapsed_time(evs[s][j][1]) for s in range(args.steps))
                   for j in range(len(calls))]
    value = world * flops_step * args.steps / (t_max * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_desc(args.workload, ops, args.chunk_rows),
        # per call: the prepare kernel and the fused kernel
        "gpu_launches": 2 * len(calls) * args.steps,
    }
    line["config"].update({
        "parallelism": f"{ops[0].world_size} virtual ranks in one GPU's HBM; "
                       f"{world} independent replica(s)",
        "backend": args.backend, "swizzle": not args.no_swizzle, "rank_view": args.rank_view,
        "l2": f"inputs larger than L2: {in_bytes / 2**20:.0f} MiB read per step vs "
              f"{L2_BYTES / 2**20:.0f} MiB L2",
        "accumulate": "fp32", "out_dtype": "bf16",
        "tuned": tuned or None,
    })
    for op_name, t in tuned.items():
        if op_name in line["config"]:
            line["config"][op_name]["chunk_rows"] = t["chunk_rows"]
    pk = peaks()
    # the timed region's own regime: seconds of back-to-back steps settle under the power cap
    # (the sustained cuBLAS figure); a short region runs at boost clocks (the burst figure)
    regime = "sustained" if (w1 - w0) >= 2.0 else "burst"
    peak = pk["bf16_tflops_sustained"] if regime == "sustained" else pk["bf16_tflops"]
    line["frac_of_peak"] = value / world / peak
    line["per_op"] = {cl["op"]: {"ms": ms, "tflops": cl["wl"].flops / (ms * 1e-3) / 1e12,
                                 "frac_of_peak": cl["wl"].flops / (ms * 1e-3) / 1e12 / peak}
                      for cl, ms in zip(calls, per_call_ms)}
    dom = max(range(len(calls)), key=lambda j: per_call_ms[j])
    dom_achieved = calls[dom]["wl"].flops / (per_call_ms[dom] * 1e-3) / 1e12
    tr = NCU_TRAFFIC.get(calls[dom]["wl"].name)
    used = calls[dom]["args"]  # the knobs actually timed (after tuning)
    op_id = {"ag": dt.OP_AG, "rs": dt.OP_RS, "ar": dt.OP_AR, "a2a": dt.OP_A2A}[calls[dom]["op"]]
    hints = int(os.environ.get("DT_L2_HINTS", "3")) & 3  # the library's L2 policies
    knob_key = (f"{used.chunk_rows}/{dt.tile_rows(used, op_id)}/{dt.col_band(used, op_id)}/"
                f"{hints}")
    traffic = tr["points"].get(knob_key) if tr and tr["csrc"] == csrc_hash() else None
    line["roofline"] = {
        "bound": "tensor", "kernel": f"fused_gemm_kernel ({calls[dom]['op']})",
        "achieved": dom_achieved, "peak": peak, "unit": "TFLOP/s", "frac": dom_achieved / peak,
        "regime": regime,
        "traffic": traffic, "traffic_unit": "bytes per launch (ncu dram read + write)",
        "traffic_source": (f"recorded ncu capture of these kernel sources ({tr['profile']}), not "
                           "measured in this run" if traffic is not None else
                           "none recorded for these kernel sources and knobs"),
        "knobs": knob_key,
        "peak_source": (f"{pk['source']} bf16 sustained (cuBLAS back to back for seconds, under the "
                        f"power cap): the timed region ran {w1 - w0:.2f} s"
                        if regime == "sustained" else
                        f"{pk['source']} bf16 burst (cuBLAS best of 10): the timed region ran "
                        f"{w1 - w0:.2f} s, too short to settle under the power cap"),
        "algorithmic_flops_per_launch": calls[dom]["wl"].flops,
    }

    if not args.skip_extras and rank == 0:
        line["clocks"] = sampler.summary(w0, w1)
        line.update(extras(args, dt, torch, dev, calls, run_call, flops_step, in_bytes, out_bytes,
                           ops, inputs, value, world, pk, build_calls, arenas))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def extras(args, dt, torch, dev, calls, run_call, flops_step, in_bytes, out_bytes, ops, inputs,
           value, world, pk, build_calls, arenas):
    out = {}
    stream = torch.cuda.current_stream(dev)
    k_side = max(3, min(args.steps, 20))

    def timed(fn, k):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / k

    # kernel-level-overlap baseline: same GEMM kernel, per-chunk / per-destination launches.
    # Its AllGather launches one GEMM per chunk, so it runs at its own best chunk size rather
    # than the fused kernel's.
    base_chunks = {}
    for cl in calls:
        if cl["op"] != "ag":
            continue
        ms_rank = cl["wl"].m // cl["wl"].world_size
        best = None
        for cr in sorted({int(cl["args"].chunk_rows), 256, 512, 1024, 2048, ms_rank}):
            if cr > ms_rank:
                continue
            a = dt.DtArgs.from_buffer_copy(cl["args"])
            a.chunk_rows = cr
            if dt.workspace_size(a, dt.OP_AG) > cl["ws"].numel():
                continue
            cl["base_args"] = a
            t = timed(lambda: run_call(cl, fused=False), 3)
            if best is None or t < best[0]:
                best = (t, a)
        cl["base_args"] = best[1]
        base_chunks[cl["op"]] = int(best[1].chunk_rows)
    ms_b = timed(lambda: [run_call(cl, fused=False) for cl in calls], k_side)
    for cl in calls:
        st, info = dt.check(cl["ws"])
        if st != 0:
            raise RuntimeError(f"baseline device error {info}")
    out["kernel_overlap_baseline"] = {
        "value": flops_step / (ms_b * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_b,
        "fused_speedup": ms_b / (flops_step / (value / world * 1e12) * 1e3),
        "chunk_rows": base_chunks or None}

    # the copy path on its own: the AllGather's chunk transfer of every shard into one [M, K]
    # buffer, per backend; 2 x bytes (read + write) over the time, against the measured HBM
    # copy rate; L2 flushed before each timed copy (the shards fit in L2 otherwise) by READING a
    # buffer of twice its size: a flush that writes leaves up to 129 MB of dirty lines whose
    # write-back then lands inside the timed copy
    hbm = peaks()["hbm_gbs"]

    def copy_path(shards, name, tuned_cr):
        w = len(shards)
        m, k = sum(t.shape[0] for t in shards), shards[0].shape[1]
        gathered = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
        flush = torch.zeros(2 * L2_BYTES // 8, dtype=torch.int64, device=dev)
        nbytes = m * k * 2
        res = {}

        def point(t):
            return {"ms": t, "gbs": 2 * nbytes / (t * 1e-3) / 1e9,
                    "frac": 2 * nbytes / (t * 1e-3) / 1e9 / hbm}
        for be in ("copy_engine", "tma", "ldst"):
            pts = {}
            for cr in sorted({tuned_cr, 512, 1024, m // w}):
                ga = dt.make_args(w, m, 8, k, chunk_rows=cr, backend=be)
                gws = torch.zeros(dt.workspace_size(ga, dt.OP_AG), dtype=torch.uint8, device=dev)
                dt.allgather(shards, gathered, gws, ga)
                times = []
                for _ in range(k_side):
                    torch.amax(flush)  # reads 258 MiB: evicts the shards, leaves clean lines
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    dt.allgather(shards, gathered, gws, ga)
                    e1.record(stream)
                    torch.cuda.synchronize(dev)
                    times.append(e0.elapsed_time(e1))
                code, info = dt.check(gws)
                if code != 0:
                    raise RuntimeError(f"AllGather device error {info}")
                pts[cr] = statistics.median(times)
            best = min(pts, key=pts.get)
            res[be] = dict(point(pts[tuned_cr]), chunk_rows=tuned_cr,
                           best=dict(point(pts[best]), chunk_rows=best))
        if not torch.equal(gathered.view(torch.int16), torch.cat(shards, dim=0).view(torch.int16)):
            raise RuntimeError("AllGather result differs from the shards")
        del gathered, flush
        return {
            "what": f"AllGather alone of {name}'s {w} shards ({nbytes / 2**20:.0f} MiB) at the "
                    "fused call's chunk rows and, under `best`, at the fastest of 512, 1024 and "
                    "one chunk per rank; L2 flushed before each copy by reading a 258 MiB "
                    "buffer; gbs = 2 x bytes / time (read + write)",
            "unit": "GB/s", "peak": hbm, "peak_source": "measured HBM copy" if
            peaks()["source"] == "measured" else "fallback", "backends": res}

    ag_calls = [cl for cl in calls if cl["op"] == "ag"]
    if ag_calls:
        cl = ag_calls[0]
        out["copy_path"] = copy_path(cl["shards"], cl["wl"].name, int(cl["args"].chunk_rows))
        # the same on the largest AllGather's shards (the chunk sweep's workload, 256 MiB):
        # the copy does not depend on the values, so they are drawn on the device
        big = WORKLOADS["ag_w8_m16384_n8192_k8192"]
        if big.name != cl["wl"].name:
            g = torch.Generator(device=dev).manual_seed(big.seed)
            shards = [torch.randn((big.m // big.world_size, big.k), generator=g, device=dev)
                      .to(torch.bfloat16) for _ in range(big.world_size)]
            out["copy_path_largest_ag"] = copy_path(shards, big.name, 2048)
            del shards

    # context: non-overlapped gather + cuBLAS (AG); cuBLAS partial products + sum (RS)
    def cublas_step():
        for cl in calls:
            if cl["op"] == "ag":
                a = torch.cat(cl["shards"], dim=0)
                torch.matmul(a, cl["b"])
            elif cl["op"] == "a2a":
                w = len(cl["A"])
                ms, nw = cl["A"][0].shape[0], cl["outs"][0].shape[1]
                for q, a_ in enumerate(cl["A"]):
                    y = torch.mm(a_, cl["B"][q])
                    for h in range(w):
                        cl["outs"][h][q * ms:(q + 1) * ms].copy_(y[:, h * nw:(h + 1) * nw])
            else:
                acc = None
                for a_, b_ in zip(cl["A"], cl["B"]):
                    p = torch.mm(a_, b_).float()
                    acc = p if acc is None else acc + p
                acc.to(torch.bfloat16)
    ms_c = timed(cublas_step, max(3, k_side // 2))
    out["cublas_nonoverlapped_context"] = {
        "value": flops_step / (ms_c * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_c,
        "note": "torch.cat gather + torch.matmul (AG); per-rank torch.mm, fp32 sum (RS); "
                "per-rank torch.mm then block copies (A2A)"}

    # spot check of the fused result against cuBLAS on a row sample
    for cl in calls:
        run_call(cl)
    torch.cuda.synchronize(dev)
    errs = []
    for cl in calls:
        if cl["op"] == "ag":
            a = torch.cat(cl["shards"], dim=0)[:256].float()
            ref = a @ cl["b"].float()
            if cl.get("act") == "gelu_tanh":
                ref = torch.nn.functional.gelu(ref, approximate="tanh")
            elif cl.get("act") == "silu":
                ref = torch.nn.functional.silu(ref)
            got = cl["outs"][0][:256].float()
        elif cl["op"] == "a2a":  # out_0 rows 0..127: source 0's rows, destination 0's columns
            nw = cl["outs"][0].shape[1]
            ref = cl["A"][0][:128].float() @ cl["B"][0][:, :nw].float()
            got = cl["outs"][0][:128].float()
        else:  # ReduceScatter out_0 / AllReduce rank 0: rows 0..127 of the sum
            ref = sum(a_[:128].float() @ b_.float() for a_, b_ in zip(cl["A"], cl["B"]))
            got = cl["outs"][0][:128].float()
        errs.append(float((got - ref).abs().max() / ref.abs().max()))
    out["spot_check_vs_cublas_max_rel_err"] = max(errs)

    # The same step run back to back for ~2.5 s, long enough to settle under the power cap,
    # against the sustained cuBLAS figure (the timed region above is a short burst when the
    # step count is small); outside the timed region, for context
    if world == 1:
        ms_step = flops_step / (value / world * 1e12) * 1e3
        n_sus = max(10, int(2500.0 / ms_step))
        dom_call = max(calls, key=lambda c: c["wl"].flops)
        evs_s = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(n_sus)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        gc.disable()
        e0.record(stream)
        for s_ in range(n_sus):
            for cl in calls:
                if cl is dom_call:
                    evs_s[s_][0].record(stream)
                run_call(cl)
                if cl is dom_call:
                    evs_s[s_][1].record(stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        gc.enable()
        for cl in calls:
            code, info = dt.check(cl["ws"])
            if code != 0:
                raise RuntimeError(f"device error in the sustained run {info}")
        t_s = e0.elapsed_time(e1)
        # the second half of the run: settled under the cap
        half = [evs_s[i][0].elapsed_time(evs_s[i][1]) for i in range(n_sus // 2, n_sus)]
        dom_ms = statistics.mean(half)
        sus_peak = pk["bf16_tflops_sustained"]
        out["sustained"] = {
            "steps": n_sus, "seconds": t_s / 1e3,
            "value": flops_step * n_sus / (t_s * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": t_s / n_sus,
            "dominant_kernel_frac_of_sustained_peak":
                dom_call["wl"].flops / (dom_ms * 1e-3) / 1e12 / sus_peak,
            "peak": sus_peak,
            "note": "the step back to back for ~2.5 s after the timed region; the dominant "
                    "kernel's fraction uses the mean of its second half, against the measured "
                    "sustained cuBLAS bf16 figure"}

    # How much of the AllGather's transfer the GEMM hid: one call with the debug timeline
    # attached (the kernel's own global-timer records of each chunk's release and first read,
    # and of the time its producers spent waiting for flags), at the tuned knobs and with the
    # in-kernel TMA transfer at the same chunk rows (whose releases are timed on the device)
    ag_calls = [cl for cl in calls if cl["op"] == "ag"]
    if ag_calls:
        cl = ag_calls[0]
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        res = {}
        variants = {"as_tuned": cl["args"]}
        if cl["args"].backend != dt.BACKENDS["tma"]:
            t = dt.DtArgs.from_buffer_copy(cl["args"])
            t.backend, t.copy_ctas = dt.BACKENDS["tma"], 0
            if dt.workspace_size(t, dt.OP_AG) <= cl["ws"].numel():
                variants["tma"] = t
        for name, a in variants.items():
            if a.backend == dt.BACKENDS["tma_tile"]:
                res[name] = {"backend": "tma_tile", "chunk_rows": int(a.chunk_rows),
                             "note": "no separate transfer: each tile pulls its own rows into "
                                     "shared memory behind the operand ring's mbarriers, so "
                                     "no flag is waited for"}
                continue
            buf = torch.zeros(dt.trace_bytes(a) // 8, dtype=torch.int64, device=dev)
            dt.ag_gemm(cl["shards"], cl["b"], cl["outs"][0], cl["ws"], a)  # warm
            dt.trace_attach(buf)
            try:
                dt.ag_gemm(cl["shards"], cl["b"], cl["outs"][0], cl["ws"], a)
                code, info = dt.check(cl["ws"])
            finally:
                dt.trace_attach(None)
            if code != 0:
                raise RuntimeError(f"traced AllGather device error {info}")
            tr = dt.trace_decode(buf.cpu().tolist(), a)
            rel = [c["released_us"] for c in tr["chunks"].values() if c["released_us"] is not None]
            seen = [c["first_read_us"] for c in tr["chunks"].values()
                    if c["first_read_us"] is not None]
            span = max(rel) if rel else (max(seen) if seen else 0.0)
            exposed = tr["stall_us_total"] / sms  # per SM: the producers' flag waits
            res[name] = {
                "backend": [k for k, v in dt.BACKENDS.items() if v == a.backend][0],
                "chunk_rows": int(a.chunk_rows), "kernel_us": tr["kernel_us"],
                "transfer_span_us": span,
                "transfer_span_source": "last in-kernel release" if rel else
                                        "last first-read of a chunk (copy-engine flags are "
                                        "written by the copy's stream, not timed)",
                "stall_us_total": tr["stall_us_total"], "stalled_waits": tr["stalled_waits"],
                "exposed_us_per_sm": exposed,
                "hidden_frac": (1.0 - exposed / span) if span > 0 else None}
        out["ag_overlap"] = dict(res, note="one traced call each; hidden_frac = 1 - (flag-wait "
                                 "time per SM) / (time from the kernel's start until the last "
                                 "chunk was released or first read)")

    # End to end through the public API with host buffers: every step copies its inputs in
    # from pinned host memory and its outputs out, inside the timed region.  Two device sets
    # of inputs / outputs / workspaces let step i+1's host-to-device copy and step i-1's
    # device-to-host copy run on their own streams while step i computes.  Each set's inputs
    # sit back to back in one arena and its outputs in another, so a step's inputs cross the
    # link as one copy and its outputs as one copy (many small copies spread over several
    # streams reached the link rate in some processes and two thirds of it in others).
    second, _, _, arenas2 = build_calls()
    sets = [calls, second]
    set_arenas = [arenas, arenas2]
    for c1, c2 in zip(sets[0], sets[1]):
        c2["args"] = c1["args"]  # the tuned knobs
    in_used, out_used = arenas[0].used, arenas[1].used
    host_in = torch.empty(in_used, dtype=torch.uint8, pin_memory=True)
    host_in.copy_(arenas[0].buf[:in_used])
    host_out = [torch.empty(out_used, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    s_main = torch.cuda.current_stream(dev)
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def merged(spans):
        spans = sorted(spans)
        out_ = [list(spans[0])]
        for lo, hi in spans[1:]:
            if lo <= -(-out_[-1][1] // Arena.ALIGN) * Arena.ALIGN:
                out_[-1][1] = max(out_[-1][1], hi)
            else:
                out_.append([lo, hi])
        return [tuple(x) for x in out_]

    ranges_all = [(0, in_used)]
    # the same with the weights resident in HBM: only the activations cross the link each step
    ranges_act = merged([arenas[0].span(t) for cl in calls for t in cl["acts"]])
    act_bytes = sum(t.numel() * t.element_size() for cl in calls for t in cl["acts"])

    timing = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    e2e_parts = []  # per run: median copy-in, compute and copy-out time of a step, and the lag
                    # from step i's compute start to step i+1's copy-in start

    def e2e_steps(n, ranges=ranges_all):
        e0, e1 = timing(), timing()
        marks = [[timing() for _ in range(6)] for _ in range(n)]  # h2d, compute, d2h: start, end
        torch.cuda.synchronize(dev)
        gc.disable()  # the host enqueues only a few steps ahead: a collector pause idles the GPU
        e0.record(s_main)
        s_h2d.wait_event(e0)
        for i in range(n):
            k = i % 2
            mk = marks[i]
            dst_in, dst_out = set_arenas[k][0].buf, set_arenas[k][1].buf
            if i >= 2:
                s_h2d.wait_event(ev_done[k])  # step i-2 has finished reading set k's inputs
            with torch.cuda.stream(s_h2d):
                mk[0].record(s_h2d)
                for lo, hi in ranges:
                    dst_in[lo:hi].copy_(host_in[lo:hi], non_blocking=True)
                mk[1].record(s_h2d)
                ev_in[k].record(s_h2d)
            s_main.wait_event(ev_in[k])
            if i >= 2:
                s_main.wait_event(ev_out[k])  # step i-2's outputs have been copied out
            mk[2].record(s_main)
            for cl in sets[k]:
                run_call(cl)
            mk[3].record(s_main)
            ev_done[k].record(s_main)
            s_d2h.wait_event(ev_done[k])
            with torch.cuda.stream(s_d2h):
                mk[4].record(s_d2h)
                host_out[k].copy_(dst_out[:out_used], non_blocking=True)
                mk[5].record(s_d2h)
                ev_out[k].record(s_d2h)
        for k in range(min(n, 2)):
            s_main.wait_event(ev_out[k])
        e1.record(s_main)
        torch.cuda.synchronize(dev)
        gc.enable()
        if n >= 4:
            mid = marks[1:n - 1]
            parts = {"h2d": [m[0].elapsed_time(m[1]) for m in mid],
                     "compute": [m[2].elapsed_time(m[3]) for m in mid],
                     "d2h": [m[4].elapsed_time(m[5]) for m in mid],
                     # step i's compute start to step i+1's copy-in start (the overlap), and
                     # step i's compute end to step i+1's compute start (the gap between steps)
                     "next_h2d_after_compute_start": [
                         marks[i][2].elapsed_time(marks[i + 1][0]) for i in range(1, n - 2)],
                     "compute_gap": [
                         marks[i][3].elapsed_time(marks[i + 1][2]) for i in range(1, n - 2)]}
            e2e_parts.append(dict(
                {f"{k_}_ms": statistics.median(v_) for k_, v_ in parts.items()},
                **{f"{k_}_max_ms": max(v_) for k_, v_ in parts.items()}))
        return e0.elapsed_time(e1)

    e2e_steps(2)  # warm-up (second set's tile orders, pinned pages)
    # steady state: the first step's copy-in and the last step's copy-out overlap nothing.  The
    # host link now and then holds a copy for 15-40 ms, which one short run cannot absorb: each
    # figure is the median of e2e_reps runs of n_e steps (every run moves every step's bytes)
    n_e = max(4, min(args.steps, 50))
    e2e_reps = 5

    def e2e_median(ranges=ranges_all):
        del e2e_parts[:]
        runs = [e2e_steps(n_e, ranges) / n_e for _ in range(e2e_reps)]
        parts = [dict({k_: round(v_, 4) for k_, v_ in p_.items()}, ms_per_step=round(r_, 4))
                 for p_, r_ in zip(e2e_parts, runs)]
        return statistics.median(runs), parts

    ms_e, runs_e = e2e_median()
    ms_act, runs_act = e2e_median(ranges_act)
    # The host-to-device copies of step i+1 run on the copy engines while step i computes, so an
    # AllGather whose chunks also move on the copy engines queues behind them.  Time the same
    # steps with the AllGather's chunks moved by the in-kernel TMA transfer and keep the faster.
    ag_be = {}
    ce_calls = [cl for cl in calls if cl["op"] == "ag" and
                cl["args"].backend in (dt.BACKENDS["copy_engine"], dt.BACKENDS["auto"])]
    be_before = [cl["args"].backend for cl in ce_calls]
    if ce_calls:
        for cl in ce_calls:
            cl["args"].backend = dt.BACKENDS["tma"]
        e2e_steps(2)
        ms_e_tma, runs_e_tma = e2e_median()
        ms_act_tma, runs_act_tma = e2e_median(ranges_act)
        ag_be = {"as_tuned": {"ms_per_step": ms_e, "weights_resident_ms_per_step": ms_act},
                 "tma": {"ms_per_step": ms_e_tma, "weights_resident_ms_per_step": ms_act_tma}}
        if ms_e_tma < ms_e:
            ms_e, runs_e = ms_e_tma, runs_e_tma
            ag_be["used"] = "tma"
        else:
            ag_be["used"] = "as_tuned"
        if ms_act_tma < ms_act:
            ms_act, runs_act = ms_act_tma, runs_act_tma
            ag_be["weights_resident_used"] = "tma"
        else:
            ag_be["weights_resident_used"] = "as_tuned"
        for cl, be in zip(ce_calls, be_before):
            cl["args"].backend = be
    for st in sets:
        for cl in st:
            code, info = dt.check(cl["ws"])
            if code != 0:
                raise RuntimeError(f"device error in the end-to-end run {info}")
    # the outputs that came back are the GEMM's: check the last step's against the device
    last = (n_e - 1) % 2
    if not torch.equal(set_arenas[last][1].buf[:out_used].cpu(), host_out[last]):
        raise RuntimeError("end-to-end outputs differ from the device's")
    # the host link's own rate, measured here: one 512 MiB pinned copy each way, best of 3; the
    # step's inputs cannot arrive faster than in_bytes at the host-to-device rate
    link_bytes = 1 << 29
    h_buf = torch.empty(link_bytes, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(link_bytes, dtype=torch.uint8, device=dev)

    def link_ms(h2d):
        best = 1e9
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(s_main)
            if h2d:
                d_buf.copy_(h_buf, non_blocking=True)
            else:
                h_buf.copy_(d_buf, non_blocking=True)
            e1.record(s_main)
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        return best

    h2d_gbs = link_bytes / (link_ms(True) * 1e-3) / 1e9
    d2h_gbs = link_bytes / (link_ms(False) * 1e-3) / 1e9
    del h_buf, d_buf
    ms_dev = flops_step / (value / world * 1e12) * 1e3  # the device-resident step
    floor_ms = max(in_bytes / (h2d_gbs * 1e9) * 1e3, ms_dev)
    out["e2e"] = {"value": world * flops_step / (ms_e * 1e-3) / 1e12, "unit": "TFLOP/s",
                  "ms_per_step": ms_e, "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                  "pipelined": "step i+1's inputs in and step i-1's outputs out overlap step i, "
                               "each as one copy (inputs and outputs packed in one buffer each)",
                  "runs": runs_e,
                  "timing": f"median of {e2e_reps} runs of {n_e} pipelined steps; per run the "
                            "median and the largest step time of each part (events on the copy "
                            "and compute streams), how long after step i's compute starts step "
                            "i+1's copy-in starts, and the gap from one step's compute to the "
                            "next",
                  "link": {"h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                           "floor_ms_per_step": floor_ms, "frac_of_floor": floor_ms / ms_e,
                           "note": "floor = the larger of the step's input bytes at the measured "
                                   "pinned host-to-device rate and the device step time"},
                  "weights_resident": {
                      "value": world * flops_step / (ms_act * 1e-3) / 1e12, "ms_per_step": ms_act,
                      "runs": runs_act,
                      "h2d_bytes_per_step": act_bytes, "d2h_bytes_per_step": out_bytes,
                      "floor_ms_per_step": max(act_bytes / (h2d_gbs * 1e9) * 1e3, ms_dev),
                      "note": "the weights (B, B_q, W1, W2) stay in HBM; the activations are "
                              "copied in and the outputs out every step"}}
    if ag_be:
        out["e2e"]["ag_transfer"] = dict(ag_be, note="the AllGather's chunk transfer while the "
                                         "host link's copies hold the copy engines")

    # the CPU oracle on a bounded sample (rank 0, N=1 only)
    if world == 1:
        f, s, desc = oracle_sample(ops, 1 << 30, 4096, inputs)
        out["cpu_baseline"] = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                               "kind": "oracle", "sample": desc, "seconds": s}
    return out


if __name__ == "__main__":
    sys.exit(main())
