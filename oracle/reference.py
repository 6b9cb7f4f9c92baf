"""Float64 reference results of the fused AllGather-GEMM and GEMM-ReduceScatter.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definitions followed (DITRON page, sections "4. 支持的并行策略" and "3.2 中端":
tensor parallelism uses AllGather+GEMM and GEMM+ReduceScatter; Triton-distributed
talk, "GEMM ReduceScatter" paragraph: every rank computes a partial product and
the reduced rows are scattered to their owner ranks):

* AllGather over W ranks (the collective on its own): every rank receives
  concat_rows(A_0, ..., A_{W-1}), shard s at rows s*M/W .. (s+1)*M/W - 1.
* AllGather-GEMM over W ranks: A = concat_rows(A_0, ..., A_{W-1}); C = A @ B.
* GEMM-ReduceScatter over W ranks: P_q = A_q @ B_q (rank q holds a K slice);
  S = sum_q P_q; rank s receives rows s*M/W .. (s+1)*M/W - 1 of S.
* GEMM-AllReduce over W ranks: the same S; every rank receives all of it.
* GEMM-AllToAll over W ranks (sequence parallelism, DITRON page section 4: SP uses
  GEMM+AllToAll): rank q holds the sequence rows A_q and computes Y_q = A_q @ B_q; the
  AllToAll sends column block h of Y_q to rank h, which stacks what it receives by source
  rank.

Inputs are float64 arrays holding exact bf16 values; outputs are float64.
"""
from __future__ import annotations

import numpy as np


def allgather(shards):
    """The gathered matrix: shard s's rows at rows s*M/W .. of the result, any dtype kept
    (a copy is exact, so bf16 bit patterns pass through unchanged)."""
    if len(shards) < 1:
        raise ValueError("need at least one shard")
    rows = {np.asarray(x).shape[0] for x in shards}
    if len(rows) != 1:
        raise ValueError("every rank holds M/W rows")
    return np.concatenate([np.asarray(x) for x in shards], axis=0)


def ag_gemm(shards, b):
    """C = concat_rows(shards) @ b, in float64 (one library matmul)."""
    a = np.concatenate([np.asarray(x, dtype=np.float64) for x in shards], axis=0)
    return a @ np.asarray(b, dtype=np.float64)


def gemm_rs(a_list, b_list):
    """Per-rank partial products, summed over ranks, rows scattered.

    Returns a list of W float64 arrays; entry s is rows [s*M/W, (s+1)*M/W) of
    sum_q a_list[q] @ b_list[q].
    """
    w = len(a_list)
    if w != len(b_list) or w < 1:
        raise ValueError("need one A and one B per rank")
    s_full = None
    for q in range(w):
        p_q = np.asarray(a_list[q], dtype=np.float64) @ np.asarray(b_list[q], dtype=np.float64)
        s_full = p_q if s_full is None else s_full + p_q
    m = s_full.shape[0]
    if m % w:
        raise ValueError("M must be a multiple of W")
    ms = m // w
    return [s_full[s * ms:(s + 1) * ms] for s in range(w)]


def gemm_ar(a_list, b_list):
    """GEMM-AllReduce over W ranks: every rank receives S = sum_q A_q @ B_q (all M rows).

    DITRON page, section 4 / 5.1 (GEMM-AR: GEMM followed by an AllReduce of the partial
    products).  Returns a list of W float64 arrays, all equal to S.
    """
    w = len(a_list)
    if w != len(b_list) or w < 1:
        raise ValueError("need one A and one B per rank")
    s_full = None
    for q in range(w):
        p_q = np.asarray(a_list[q], dtype=np.float64) @ np.asarray(b_list[q], dtype=np.float64)
        s_full = p_q if s_full is None else s_full + p_q
    return [s_full.copy() for _ in range(w)]


ACTIVATIONS = ("none", "gelu_tanh", "silu")


def activation(x, act):
    """Elementwise activation in float64.

    gelu_tanh: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), the tanh form of GELU used by
    GPT / Megatron feed-forward blocks; silu: x / (1 + exp(-x)).
    """
    x = np.asarray(x, dtype=np.float64)
    if act == "none":
        return x.copy()
    if act == "gelu_tanh":
        return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))
    if act == "silu":
        return x / (1.0 + np.exp(-x))
    raise ValueError(act)


def round_bf16_via_f32(x):
    """float64 -> float32 (nearest) -> bfloat16 (nearest, ties to even), returned as float64:
    how the CUDA epilogue stores an fp32 value as bf16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def ffn_tp(x_shards, w1, w2_list, act):
    """Tensor-parallel feed-forward block over W ranks, AllGather + ReduceScatter form.

    Rank q holds the column block q of W1 (F/W columns) and W2_q (F/W x N).  Every rank
    gathers X, computes H_q = act(X W1_q), stored as bf16, and the partial H_q W2_q; the
    partials are reduce-scattered by rows.  (DITRON page, section 5.1 "FFN模块": AllGather +
    ReduceScatter around the two GEMMs.)  Returns (H as float64 [M, F], list of W out_s).
    """
    w = len(x_shards)
    x = np.concatenate([np.asarray(s, dtype=np.float64) for s in x_shards], axis=0)
    h = round_bf16_via_f32(activation(x @ np.asarray(w1, dtype=np.float64), act))
    fr = h.shape[1] // w
    outs = gemm_rs([h[:, q * fr:(q + 1) * fr] for q in range(w)], w2_list)
    return h, outs


def ag_gemm_entries(shards, b, rows, cols):
    """Selected entries C[rows[t], cols[t]] of the AllGather-GEMM, one dot each.

    Row g of the gathered A is row g - s*Ms of shard s = g // Ms.
    """
    ms = shards[0].shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.float64)
    bt = np.asarray(b)
    for t in range(rows.shape[0]):
        s = int(rows[t]) // ms
        a_row = np.asarray(shards[s][int(rows[t]) - s * ms], dtype=np.float64)
        out[t] = float(np.dot(a_row, np.asarray(bt[:, int(cols[t])], dtype=np.float64)))
    return out


def gemm_rs_entries(a_list, b_list, dest, rows, cols):
    """Selected entries out_dest[t][rows[t], cols[t]] of the GEMM-ReduceScatter.

    out_s[m, n] = sum over q of A_q[s*Ms + m, :] . B_q[:, n], summed in q order.
    """
    w = len(a_list)
    ms = a_list[0].shape[0] // w
    out = np.empty(len(rows), dtype=np.float64)
    for t in range(len(rows)):
        g = int(dest[t]) * ms + int(rows[t])
        acc = 0.0
        for q in range(w):
            acc += float(np.dot(np.asarray(a_list[q][g], dtype=np.float64),
                                np.asarray(b_list[q][:, int(cols[t])], dtype=np.float64)))
        out[t] = acc
    return out


def gemm_a2a(a_list, b_list):
    """GEMM-AllToAll over W ranks, the sequence-parallel kernel of the DITRON page (section 4,
    "序列并行SP: GEMMAllToAll"; section 4.2, weak scaling with a fixed sequence length per rank).

    Rank q holds A_q [Ms, K] (its Ms sequence rows) and B_q [K, N], N = W * Nw.  It computes
    Y_q = A_q @ B_q; the all-to-all moves column block h of Y_q (columns h*Nw .. (h+1)*Nw - 1,
    e.g. the heads that rank h owns) to rank h, where the blocks are stacked in source-rank
    order:  out_h[q*Ms + r, c] = Y_q[r, h*Nw + c].  Returns a list of W float64 arrays
    [W*Ms, Nw].
    """
    w = len(a_list)
    if w != len(b_list) or w < 1:
        raise ValueError("need one A and one B per rank")
    ys = [np.asarray(a_list[q], dtype=np.float64) @ np.asarray(b_list[q], dtype=np.float64)
          for q in range(w)]
    n = ys[0].shape[1]
    if n % w:
        raise ValueError("N must be a multiple of W")
    nw = n // w
    return [np.concatenate([ys[q][:, h * nw:(h + 1) * nw] for q in range(w)], axis=0)
            for h in range(w)]


def gemm_a2a_entries(a_list, b_list, dest, rows, cols):
    """Selected entries out_dest[t][rows[t], cols[t]] of the GEMM-AllToAll, one dot each.

    Row m of out_h is row m - q*Ms of source q = m // Ms; column c is column h*Nw + c of B_q.
    """
    w = len(a_list)
    ms = a_list[0].shape[0]
    nw = b_list[0].shape[1] // w
    out = np.empty(len(rows), dtype=np.float64)
    for t in range(len(rows)):
        h, m, c = int(dest[t]), int(rows[t]), int(cols[t])
        q = m // ms
        out[t] = float(np.dot(np.asarray(a_list[q][m - q * ms], dtype=np.float64),
                              np.asarray(b_list[q][:, h * nw + c], dtype=np.float64)))
    return out
