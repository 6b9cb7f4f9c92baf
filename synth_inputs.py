"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU oracle.

This module only draws numbers and rounds them to bfloat16; it holds none of
the arithmetic of the fused AllGather-GEMM / GEMM-ReduceScatter.  Both the CUDA
path and the oracle read the same bf16 bit patterns produced here.

Recipe (one generator per workload):
  * numpy ``Generator(PCG64(seed))``, float64 draws;
  * "uniform": U[-1, 1]; "normal(s)": N(0, s^2);
  * each float64 draw is rounded to the nearest bfloat16, ties to even;
  * AllGather-GEMM draw order: the gathered A (M x K, row-major; shard s is
    rows s*M/W .. (s+1)*M/W - 1), then B (K x N);
  * GEMM-ReduceScatter draw order: A_0 .. A_{W-1} (each M x K_rank), then
    B_0 .. B_{W-1} (each K_rank x N).

The workloads below stand in for the "real-model shapes" that the DITRON and
AutoOverlap/Syncopate evaluations draw from Llama/Qwen/Mixtral/GPT/DeepSeek
(their shape appendix is not available), with the sizes, seeds and value
distributions of the five benchmark configurations.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np


def bf16_bits_from_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (round to nearest, ties to even).

    Returns the uint16 bit patterns.  Rounding is done exactly in float64: the
    significand m in [0.5, 1) is scaled by 2^8, rounded half-to-even by rint,
    and scaled back; the result then has 8 significant bits and converts to
    float32 exactly, whose top 16 bits are the bfloat16 pattern.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    tiny = (r != 0) & (np.abs(r) < np.ldexp(1.0, -126))
    if np.any(tiny):
        raise ValueError("draw below the bf16 normal range; pick another seed")
    if np.any(np.abs(r) >= np.ldexp(1.0, 128)):
        raise ValueError("draw above the bf16 range")
    r32 = r.astype(np.float32)
    return (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f64_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of bfloat16 bit patterns."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _draw(rng: np.random.Generator, dist: str, shape) -> np.ndarray:
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    if dist.startswith("normal(") and dist.endswith(")"):
        std = float(dist[len("normal("):-1])
        return rng.normal(0.0, std, size=shape)
    raise ValueError(f"unknown distribution {dist!r}")


def _draw_bf16(rng, dist, shape, row_block=1024):
    """Draw a row-major matrix in row blocks (the same stream as one big draw).

    Draws are sequential; the rounding of each block runs on a thread pool."""
    rows, cols = shape
    out = np.empty(shape, dtype=np.uint16)

    def _round(r0, x):
        out[r0:r0 + x.shape[0]] = bf16_bits_from_f64(x)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        futs = []
        for r0 in range(0, rows, row_block):
            r1 = min(rows, r0 + row_block)
            futs.append(ex.submit(_round, r0, _draw(rng, dist, (r1 - r0, cols))))
        for f in futs:
            f.result()
    return out


@dataclass
class AGInputs:
    world_size: int
    shards: list            # W arrays uint16 [M/W, K]
    b: np.ndarray           # uint16 [K, N]


@dataclass
class RSInputs:
    world_size: int
    a: list                 # W arrays uint16 [M, K_rank]
    b: list                 # W arrays uint16 [K_rank, N]


def make_ag_inputs(world_size: int, m: int, n: int, k: int, seed: int,
                   dist_a: str = "uniform", dist_b: str = "uniform") -> AGInputs:
    """Inputs of one AllGather-GEMM: W row shards of A (M x K) and B (K x N)."""
    if m % world_size:
        raise ValueError("M must be a multiple of the world size")
    rng = np.random.Generator(np.random.PCG64(seed))
    a = _draw_bf16(rng, dist_a, (m, k))
    b = _draw_bf16(rng, dist_b, (k, n))
    ms = m // world_size
    shards = [np.ascontiguousarray(a[s * ms:(s + 1) * ms]) for s in range(world_size)]
    return AGInputs(world_size, shards, b)


def make_rs_inputs(world_size: int, m: int, n: int, k_rank: int, seed: int,
                   dist_a: str = "uniform", dist_b: str = "uniform") -> RSInputs:
    """Inputs of one GEMM-ReduceScatter: per rank A_q (M x K_rank), B_q (K_rank x N)."""
    if m % world_size:
        raise ValueError("M must be a multiple of the world size")
    rng = np.random.Generator(np.random.PCG64(seed))
    a = [_draw_bf16(rng, dist_a, (m, k_rank)) for _ in range(world_size)]
    b = [_draw_bf16(rng, dist_b, (k_rank, n)) for _ in range(world_size)]
    return RSInputs(world_size, a, b)


@dataclass
class A2AInputs:
    world_size: int
    a: list                 # W arrays uint16 [M/W, K]: each rank's sequence rows
    b: list                 # W arrays uint16 [K, N] (the same array W times when shared)


def make_a2a_inputs(world_size: int, m: int, n: int, k: int, seed: int,
                    dist_a: str = "uniform", dist_b: str = "uniform",
                    shared_b: bool = True) -> A2AInputs:
    """Inputs of one GEMM-AllToAll: per rank A_q (M/W x K); one B (K x N) that every rank
    holds (a replicated projection weight), or one per rank.  Draw order: A_0 .. A_{W-1},
    then B (or B_0 .. B_{W-1})."""
    if m % world_size or n % world_size:
        raise ValueError("M and N must be multiples of the world size")
    rng = np.random.Generator(np.random.PCG64(seed))
    ms = m // world_size
    a = [_draw_bf16(rng, dist_a, (ms, k)) for _ in range(world_size)]
    if shared_b:
        b0 = _draw_bf16(rng, dist_b, (k, n))
        b = [b0] * world_size
    else:
        b = [_draw_bf16(rng, dist_b, (k, n)) for _ in range(world_size)]
    return A2AInputs(world_size, a, b)


@dataclass
class FFNInputs:
    world_size: int
    x_shards: list          # W arrays uint16 [M/W, K]
    w1: np.ndarray          # uint16 [K, W*F_r]  (rank q's block = columns q*F_r ..)
    w2: list                # W arrays uint16 [F_r, N]


def make_ffn_inputs(world_size: int, m: int, k: int, f_rank: int, n: int, seed: int,
                    dist_x: str = "normal(1.0)", dist_w: str = "normal(0.02)") -> FFNInputs:
    """Inputs of one tensor-parallel feed-forward block: X (M x K, row shards), W1
    (K x W*F_r), W2_0 .. W2_{W-1} (F_r x N each); drawn in that order."""
    if m % world_size:
        raise ValueError("M must be a multiple of the world size")
    rng = np.random.Generator(np.random.PCG64(seed))
    x = _draw_bf16(rng, dist_x, (m, k))
    w1 = _draw_bf16(rng, dist_w, (k, world_size * f_rank))
    w2 = [_draw_bf16(rng, dist_w, (f_rank, n)) for _ in range(world_size)]
    ms = m // world_size
    return FFNInputs(world_size, [np.ascontiguousarray(x[s * ms:(s + 1) * ms])
                                  for s in range(world_size)], w1, w2)


@dataclass(frozen=True)
class Workload:
    """One benchmark / parity workload: shapes, seed, distributions, chunking."""
    name: str
    op: str                 # "ag", "rs", "ar", "ffn" or "a2a"
    world_size: int
    m: int                  # total rows (gathered M for AG; M for RS; W x rows per rank for A2A)
    n: int
    k: int                  # AG: full K; RS: K per rank
    seed: int
    dist_a: str
    dist_b: str
    chunk_rows: int
    f_rank: int = 0         # feed-forward block: hidden columns per rank
    act: str = "none"       # feed-forward block: activation between the GEMMs

    @property
    def flops(self) -> float:
        if self.op in ("ag", "a2a"):
            return 2.0 * self.m * self.n * self.k
        if self.op == "ffn":
            return 2.0 * self.m * self.world_size * self.f_rank * (self.k + self.n)
        return 2.0 * self.m * self.n * self.k * self.world_size

    def make(self):
        # "rs" and "ar" (GEMM-AllReduce) take the same per-rank inputs
        if self.op == "ffn":
            return make_ffn_inputs(self.world_size, self.m, self.k, self.f_rank, self.n, self.seed,
                                   self.dist_a, self.dist_b)
        if self.op == "a2a":
            return make_a2a_inputs(self.world_size, self.m, self.n, self.k, self.seed,
                                   self.dist_a, self.dist_b)
        if self.op == "ag":
            return make_ag_inputs(self.world_size, self.m, self.n, self.k, self.seed,
                                  self.dist_a, self.dist_b)
        return make_rs_inputs(self.world_size, self.m, self.n, self.k, self.seed,
                              self.dist_a, self.dist_b)


WORKLOADS = {
    # small AllGather-GEMM, W=2: A shards 256x512, B 512x512, U[-1,1], seed 0, chunk 128
    "ag_w2_m512_n512_k512": Workload("ag_w2_m512_n512_k512", "ag", 2, 512, 512, 512, 0,
                                     "uniform", "uniform", 128),
    # GEMM-ReduceScatter, W=4: A_q 2048x2048, B_q 2048x4096, N(0,0.02), seed 1, chunk 256
    "rs_w4_m2048_n4096_k2048": Workload("rs_w4_m2048_n4096_k2048", "rs", 4, 2048, 4096, 2048, 1,
                                        "normal(0.02)", "normal(0.02)", 256),
    # Llama-70B-like TP=8 FFN pair, seed 2: activations N(0,1), weights N(0,0.02)
    # (chunk rows: one chunk per rank, the best of the backend x chunk sweep)
    "ag_w8_m8192_n3584_k8192": Workload("ag_w8_m8192_n3584_k8192", "ag", 8, 8192, 3584, 8192, 2,
                                        "normal(1.0)", "normal(0.02)", 1024),
    # (chunk rows for the ReduceScatter: one chunk per destination rank, the best of the
    # 256 / 512 / 1024 sweep)
    "rs_w8_m8192_n8192_k3584": Workload("rs_w8_m8192_n8192_k3584", "rs", 8, 8192, 8192, 3584, 2,
                                        "normal(1.0)", "normal(0.02)", 1024),
    # the same ReduceScatter with half the tokens (M=4096): a profiling case whose inputs,
    # running sums and outputs (1.9 GB) still exceed L2
    "rs_w8_m4096_n8192_k3584": Workload("rs_w8_m4096_n8192_k3584", "rs", 8, 4096, 8192, 3584, 2,
                                        "normal(1.0)", "normal(0.02)", 512),
    # non-perfect tiling, W=6, U[-1,1], seed 3, chunk 192: every edge ragged
    "ag_w6_m6000_n3000_k5120": Workload("ag_w6_m6000_n3000_k5120", "ag", 6, 6000, 3000, 5120, 3,
                                        "uniform", "uniform", 192),
    "rs_w6_m6000_n5120_k3000": Workload("rs_w6_m6000_n5120_k3000", "rs", 6, 6000, 5120, 3000, 3,
                                        "uniform", "uniform", 192),
    # GEMM-AllReduce on the FFN pair's second GEMM (same inputs as the ReduceScatter)
    "ar_w8_m8192_n8192_k3584": Workload("ar_w8_m8192_n8192_k3584", "ar", 8, 8192, 8192, 3584, 2,
                                        "normal(1.0)", "normal(0.02)", 1024),
    # the whole Llama-70B-like TP=8 feed-forward block, chained: X 8192 x 8192 gathered,
    # H = GELU(X W1) with W1 8192 x (8 x 3584), then out = ReduceScatter(H W2), W2_q 3584 x 8192
    "ffn_w8_m8192_k8192_f3584_n8192": Workload("ffn_w8_m8192_k8192_f3584_n8192", "ffn", 8, 8192,
                                               8192, 8192, 2, "normal(1.0)", "normal(0.02)", 1024,
                                               f_rank=3584, act="gelu_tanh"),
    # GEMM-AllToAll (sequence parallelism), W=4, every edge ragged: 300 rows per rank, 200
    # columns per destination, K=520, chunk 96; U[-1,1], seed 5
    "a2a_w4_m1200_n800_k520": Workload("a2a_w4_m1200_n800_k520", "a2a", 4, 1200, 800, 520, 5,
                                       "uniform", "uniform", 96),
    # Llama-70B-like QKV projection under 8-way sequence parallelism: 2048 tokens per rank,
    # hidden 8192, N = 64 query + 2 x 8 key/value heads of 128 = 10240 (1280 per rank after
    # the all-to-all); activations N(0,1), weight N(0,0.02), seed 6
    "a2a_w8_m16384_n10240_k8192": Workload("a2a_w8_m16384_n10240_k8192", "a2a", 8, 16384, 10240,
                                           8192, 6, "normal(1.0)", "normal(0.02)", 512),
    # largest AllGather-GEMM (chunk/backend sweep), W=8, U[-1,1], seed 4
    "ag_w8_m16384_n8192_k8192": Workload("ag_w8_m16384_n8192_k8192", "ag", 8, 16384, 8192, 8192, 4,
                                         "uniform", "uniform", 256),
}
