"""Pins of the GEMM-AllToAll oracle (sequence parallelism) on the CPU.

The result is pinned against brute-force loops with exactly rounded sums, a closed form on
structured inputs that gives every output entry a distinct value fixed by (source rank, row,
global column), the special case W = 1 (a plain GEMM), and the identity with the AllGather-GEMM
when every rank holds the same B (stacking the destinations' blocks side by side gives
concat(A_q) @ B).  The tile order is pinned against hand-written orders in
tests/golden/a2a_scatter_orders.txt and the properties of the scatter schedule; the chunk
completion counts against a brute-force count.  Planted mistakes must fail some pin.
"""
import math
import os

import numpy as np
import pytest

from oracle import plan, reference
from synth_inputs import f64_from_bf16_bits, make_a2a_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_a2a(a_list, b_list):
    w = len(a_list)
    ms, k = a_list[0].shape
    nw = b_list[0].shape[1] // w
    outs = []
    for h in range(w):
        o = np.zeros((w * ms, nw))
        for q in range(w):
            for r in range(ms):
                for c in range(nw):
                    o[q * ms + r, c] = math.fsum(float(a_list[q][r, t]) * float(b_list[q][t, h * nw + c])
                                                 for t in range(k))
        outs.append(o)
    return outs


def _f64(inp):
    return [f64_from_bf16_bits(x) for x in inp.a], [f64_from_bf16_bits(x) for x in inp.b]


def _close(x, y):
    x = np.asarray(x)
    y = np.asarray(y)
    scale = max(1.0, float(np.max(np.abs(y))) if y.size else 1.0)
    return x.shape == y.shape and np.allclose(x, y, rtol=0, atol=1e-12 * scale)


CASES = [(1, 3, 5, 7), (2, 2, 3, 3), (3, 3, 2, 1), (4, 2, 2, 6), (2, 7, 5, 4)]  # W, Ms, Nw, K


# ---------------------------------------------------------------- pins on the result
# Each takes the implementation under test and returns True when the pin holds.

def pin_brute_force(a2a):
    for seed, (w, ms, nw, k) in enumerate(CASES):
        for shared in (True, False):
            a_list, b_list = _f64(make_a2a_inputs(w, w * ms, w * nw, k, seed=500 + seed,
                                                  shared_b=shared))
            got = a2a(a_list, b_list)
            want = _brute_a2a(a_list, b_list)
            if len(got) != w or not all(_close(g, x) for g, x in zip(got, want)):
                return False
    return True


def pin_closed_form(a2a):
    """A_q[r, t] = (1000 q + r + 1) if t == 0 else 0 and B_q[t, n] = (n + 1) if t == 0 else 0,
    so Y_q[r, n] = (1000 q + r + 1)(n + 1) and out_h[q Ms + r, c] = (1000 q + r + 1)(h Nw + c + 1)."""
    w, ms, nw, k = 3, 4, 5, 3
    a_list = []
    for q in range(w):
        a = np.zeros((ms, k))
        a[:, 0] = 1000 * q + np.arange(ms) + 1
        a_list.append(a)
    b = np.zeros((k, w * nw))
    b[0] = np.arange(w * nw) + 1
    got = a2a(a_list, [b] * w)
    for h in range(w):
        want = np.array([[(1000 * (g // ms) + g % ms + 1) * (h * nw + c + 1) for c in range(nw)]
                         for g in range(w * ms)], dtype=np.float64)
        if not np.array_equal(np.asarray(got[h]), want):
            return False
    return True


def pin_w1_is_plain_gemm(a2a):
    a_list, b_list = _f64(make_a2a_inputs(1, 6, 7, 5, seed=520))
    got = a2a(a_list, b_list)
    want = np.array([[math.fsum(a_list[0][r, t] * b_list[0][t, c] for t in range(5))
                      for c in range(7)] for r in range(6)])
    return len(got) == 1 and _close(got[0], want)


def pin_shared_b_is_allgather_gemm(a2a):
    """Same B on every rank: [out_0 | out_1 | ... ] = concat_rows(A_q) @ B, which is the
    AllGather-GEMM of the same shards (pinned on its own)."""
    a_list, b_list = _f64(make_a2a_inputs(4, 12, 8, 5, seed=521))
    got = a2a(a_list, b_list)
    return _close(np.concatenate(got, axis=1), reference.ag_gemm(a_list, b_list[0]))


def pin_integer_exact(a2a):
    rng = np.random.Generator(np.random.PCG64(22))
    w, ms, n, k = 3, 2, 6, 4
    a_list = [rng.integers(-5, 6, (ms, k)).astype(np.float64) for _ in range(w)]
    b_list = [rng.integers(-5, 6, (k, n)).astype(np.float64) for _ in range(w)]
    got = a2a(a_list, b_list)
    nw = n // w
    for h in range(w):
        for q in range(w):
            for r in range(ms):
                for c in range(nw):
                    exact = sum(int(a_list[q][r, t]) * int(b_list[q][t, h * nw + c]) for t in range(k))
                    if got[h][q * ms + r, c] != exact:
                        return False
    return True


PINS = [pin_brute_force, pin_closed_form, pin_w1_is_plain_gemm, pin_shared_b_is_allgather_gemm,
        pin_integer_exact]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_a2a_oracle_pin(pin):
    assert pin(reference.gemm_a2a)


def _mut_swapped_dest(a_list, b_list):
    outs = reference.gemm_a2a(a_list, b_list)
    return outs[1:] + outs[:1]


def _mut_source_order(a_list, b_list):
    w = len(a_list)
    outs = reference.gemm_a2a(list(reversed(a_list)), list(reversed(b_list)))
    return outs if w > 1 else [o * 0 for o in outs]


def _mut_rows_by_dest(a_list, b_list):
    # rows of destination h taken from the column block of the source instead
    w = len(a_list)
    ys = [np.asarray(a) @ np.asarray(b) for a, b in zip(a_list, b_list)]
    nw = ys[0].shape[1] // w
    return [np.concatenate([ys[h][:, q * nw:(q + 1) * nw] for q in range(w)], axis=0)
            for h in range(w)]


def _mut_dropped_term(a_list, b_list):
    return reference.gemm_a2a([np.asarray(a)[:, 1:] for a in a_list],
                              [np.asarray(b)[1:] for b in b_list]) if a_list[0].shape[1] > 1 else \
        [o * 0 for o in reference.gemm_a2a(a_list, b_list)]


def _mut_transposed_block(a_list, b_list):
    outs = reference.gemm_a2a(a_list, b_list)
    return [o[::-1] for o in outs]


MUTANTS = [_mut_swapped_dest, _mut_source_order, _mut_rows_by_dest, _mut_dropped_term,
           _mut_transposed_block]


def _safe(pin, impl):
    try:
        return bool(pin(impl))
    except Exception:
        return False


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_a2a_pins_catch_planted_mistakes(mutant):
    assert [p.__name__ for p in PINS if not _safe(p, mutant)], mutant.__name__


def test_a2a_sampled_entries_match_brute_force():
    a_list, b_list = _f64(make_a2a_inputs(3, 9, 6, 5, seed=530, shared_b=False))
    want = _brute_a2a(a_list, b_list)
    dest, rows, cols = [0, 1, 2, 2, 1], [0, 4, 8, 3, 7], [1, 0, 1, 0, 1]
    got = reference.gemm_a2a_entries(a_list, b_list, dest, rows, cols)
    assert _close(got, [want[h][r, c] for h, r, c in zip(dest, rows, cols)])


# ---------------------------------------------------------------- the tile order

def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "a2a_scatter_orders.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, order = line.split(":")
            _, ms, bm, cr, tnw, g = head.split()
            rows.append(((int(ms), int(bm), int(cr), int(tnw), int(g)), [int(x) for x in order.split()]))
    return rows


def test_a2a_golden_orders():
    for (ms, bm, cr, tnw, g), order in _golden():
        assert plan.a2a_order(2, ms, 2 * tnw, cr, bm, 1, group=g) == order


GRID = [
    # (W, Ms, N, Cr, BM, BN)
    (1, 100, 300, 64, 128, 256),
    (2, 256, 1024, 128, 128, 256),
    (4, 300, 800, 96, 128, 256),
    (3, 7, 12, 2, 3, 2),
    (5, 11, 30, 4, 2, 4),
    (8, 2048, 10240, 512, 128, 256),
]


def _decode(t, w, tm, tnw):
    tn = w * tnw
    q, rem = divmod(t, tm * tn)
    i, n = divmod(rem, tn)
    h, c = divmod(n, tnw)
    return q, i, h, c


@pytest.mark.parametrize("case", GRID)
@pytest.mark.parametrize("swizzle", [True, False])
def test_a2a_order_is_a_bijection(case, swizzle):
    w, ms, n, cr, bm, bn = case
    _, _, tm, tnw = plan.a2a_geometry(w, ms, n, cr, bm, bn)
    order = plan.a2a_order(w, ms, n, cr, bm, bn, swizzle=swizzle)
    assert sorted(order) == list(range(w * tm * w * tnw))
    if not swizzle:
        assert order == list(range(len(order)))


@pytest.mark.parametrize("case", GRID)
def test_a2a_next_rank_first_own_last(case):
    """Per source rank the destinations come in ring order q+1, q+2, ..., q, each
    destination's tiles together; the source ranks run one after another."""
    w, ms, n, cr, bm, bn = case
    _, nc, tm, tnw = plan.a2a_geometry(w, ms, n, cr, bm, bn)
    order = plan.a2a_order(w, ms, n, cr, bm, bn)
    rank_step = []
    for t in order:
        q, i, h, c = _decode(t, w, tm, tnw)
        rank_step.append((q, (h - q - 1) % w))
    assert rank_step == sorted(rank_step)
    for q in range(w):
        dests = [_decode(t, w, tm, tnw)[2] for t in order if _decode(t, w, tm, tnw)[0] == q]
        firsts = [d for idx, d in enumerate(dests) if idx == 0 or dests[idx - 1] != d]
        assert firsts == [(q + 1 + d) % w for d in range(w)]


@pytest.mark.parametrize("case", GRID)
def test_a2a_chunks_complete_in_order(case):
    """Inside one destination a source's chunks complete in ascending chunk order: the last tile of
    chunk j comes no later than the last tile of chunk j+1 (AutoOverlap section 5.4)."""
    w, ms, n, cr, bm, bn = case
    _, nc, tm, tnw = plan.a2a_geometry(w, ms, n, cr, bm, bn)
    order = plan.a2a_order(w, ms, n, cr, bm, bn)
    last = {}
    for pos, t in enumerate(order):
        q, i, h, c = _decode(t, w, tm, tnw)
        for j in plan.a2a_mtile_chunks(i, ms, cr, bm):
            last[(h, q, j)] = pos
    for (h, q, j), pos in last.items():
        if j + 1 < nc:
            assert pos <= last[(h, q, j + 1)]


@pytest.mark.parametrize("case", GRID[:5])
def test_a2a_expected_counts_brute_force(case):
    w, ms, n, cr, bm, bn = case
    nw, nc, tm, tnw = plan.a2a_geometry(w, ms, n, cr, bm, bn)
    counts = plan.a2a_expected_counts(w, ms, n, cr, bm, bn)
    hits = {}
    for t in range(w * tm * w * tnw):
        q, i, h, c = _decode(t, w, tm, tnw)
        for r in range(i * bm, min(ms, (i + 1) * bm)):
            hits.setdefault((h, q, r // cr), set()).add(t)
    assert counts == {key: len(v) for key, v in hits.items()}
    assert len(counts) == w * w * nc


def test_a2a_plan_pins_catch_planted_mistakes(monkeypatch):
    """A reversed send order (own block first) breaks the golden orders and the ring test."""
    original = plan.rs_dpos
    monkeypatch.setattr(plan, "rs_dpos", lambda q, s, w: (q - s) % w)
    caught = False
    try:
        test_a2a_golden_orders()
    except AssertionError:
        caught = True
    monkeypatch.setattr(plan, "rs_dpos", original)
    assert caught
