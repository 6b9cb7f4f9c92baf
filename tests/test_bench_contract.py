"""bench.py's reference arm on the CPU: one JSON line with the keys the benchmark contract
asks for, the oracle's float64 throughput as value, cpu_baseline and e2e describing the run.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_reference(*extra):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          *extra], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _run_reference("--workload", "ag_w2_m512_n512_k512", "--steps", "2", "--warmup", "1")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "ag_w2_m512_n512_k512"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_names_the_default_workload():
    d = _run_reference("--steps", "1", "--warmup", "0")
    assert d["config"]["workload"].startswith("llama70b_like_tp8_ffn_pair")
    assert set(d["config"]) >= {"ag", "rs"}


def test_traffic_table_covers_every_reduce_tuner_candidate():
    """The roofline's DRAM traffic of the benchmark's dominant launch (the FFN pair's
    ReduceScatter) is looked up by the tuned knobs: every candidate the reduce tuner can pick
    (chunk rows 64 .. M/W, the automatic column bands or one band, at the library's 256-row
    tiles and L2 policies) has an entry, and each workload names the profile its figures come
    from."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from synth_inputs import WORKLOADS
    wl = WORKLOADS[bench.FFN_PAIR[1]]
    ms = wl.m // wl.world_size
    chunks = [c for c in (64, 128, 256, 512, 1024, 2048, 4096) if c < ms] + [ms]
    points = bench.NCU_TRAFFIC[wl.name]["points"]
    for cr in chunks:
        for nb in (16, 32):
            key = f"{cr}/256/{nb}/3"
            assert key in points, key
            assert points[key] > 0
    for entry in bench.NCU_TRAFFIC.values():
        assert os.path.exists(os.path.join(ROOT, entry["profile"])), entry["profile"]


def test_arena_packs_inputs_back_to_back():
    """The end-to-end step's inputs (and outputs) sit in one buffer each, so that a step's bytes
    cross the host link as one copy: consecutive 256-byte-aligned tensors, their byte spans, and
    the capacity bound that the input arrays give."""
    import numpy as np
    import pytest
    torch = pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench
    from synth_inputs import make_rs_inputs
    inp = make_rs_inputs(2, 64, 40, 24, seed=3)
    arrays = bench._input_arrays(inp)
    assert len(arrays) == 4 and all(a.dtype == np.uint16 for a in arrays)
    arena = bench.Arena(bench.Arena.capacity(arrays), "cpu")
    ts = [arena.put(a) for a in inp.a + inp.b]
    spans = [arena.span(t) for t in ts]
    for (lo, hi), t, a in zip(spans, ts, inp.a + inp.b):
        assert lo % bench.Arena.ALIGN == 0 and hi - lo == a.nbytes
        assert t.shape == a.shape and t.dtype == torch.bfloat16
        assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), a)
    assert all(spans[i][1] <= spans[i + 1][0] for i in range(len(spans) - 1))  # back to back
    assert arena.used <= arena.buf.numel()
    with pytest.raises(RuntimeError, match="arena too small"):
        arena.take((1024, 1024))
    # outputs: the step's bytes, padded per tensor
    wl = bench.WORKLOADS["rs_w8_m8192_n8192_k3584"]
    assert bench._output_bytes(wl) >= wl.m * wl.n * 2
