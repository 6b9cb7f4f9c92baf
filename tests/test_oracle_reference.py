"""Pins of the float64 oracle (AllGather-GEMM and GEMM-ReduceScatter) on the CPU.

Each pin checks the oracle against something other than itself: brute-force
loops with exactly rounded sums (math.fsum), closed forms on structured
inputs, the special cases W=1 and the K-split identity, and integer inputs
whose results are exact.  ``test_pins_catch_planted_mistakes`` plants typical
mistakes in copies of the oracle and checks that some pin fails for each.
"""
import math

import numpy as np
import pytest

from oracle import reference
from synth_inputs import (bf16_bits_from_f64, f64_from_bf16_bits, make_ag_inputs,
                          make_rs_inputs)


def _brute_ag(shards, b):
    ms = shards[0].shape[0]
    m = ms * len(shards)
    k, n = b.shape
    out = np.zeros((m, n))
    for g in range(m):
        s = g // ms
        row = shards[s][g - s * ms]
        for c in range(n):
            out[g, c] = math.fsum(float(row[t]) * float(b[t, c]) for t in range(k))
    return out


def _brute_rs(a_list, b_list):
    w = len(a_list)
    m = a_list[0].shape[0]
    ms = m // w
    n = b_list[0].shape[1]
    outs = []
    for s in range(w):
        o = np.zeros((ms, n))
        for r in range(ms):
            g = s * ms + r
            for c in range(n):
                terms = []
                for q in range(w):
                    kq = a_list[q].shape[1]
                    terms.extend(float(a_list[q][g, t]) * float(b_list[q][t, c]) for t in range(kq))
                o[r, c] = math.fsum(terms)
        outs.append(o)
    return outs


def _ag_f64(inp):
    return [f64_from_bf16_bits(x) for x in inp.shards], f64_from_bf16_bits(inp.b)


def _rs_f64(inp):
    return [f64_from_bf16_bits(x) for x in inp.a], [f64_from_bf16_bits(x) for x in inp.b]


def _close(x, y, scale=None):
    x = np.asarray(x)
    y = np.asarray(y)
    if scale is None:
        scale = max(1.0, float(np.max(np.abs(y))) if y.size else 1.0)
    return np.allclose(x, y, rtol=0, atol=1e-12 * scale)


# ---------------------------------------------------------------- pin functions
# Each takes (ag_impl, rs_impl) and returns True when the pin holds.

AG_CASES = [(1, 3, 5, 7), (2, 4, 3, 17), (3, 9, 8, 1), (6, 6, 2, 33), (2, 14, 33, 7)]
RS_CASES = [(1, 3, 5, 7), (2, 4, 3, 17), (3, 9, 8, 1), (4, 8, 5, 6)]


def pin_ag_brute_force(ag, rs):
    for seed, (w, m, n, k) in enumerate(AG_CASES):
        inp = make_ag_inputs(w, m, n, k, seed=100 + seed)
        shards, b = _ag_f64(inp)
        if not _close(ag(shards, b), _brute_ag(shards, b)):
            return False
    return True


def pin_rs_brute_force(ag, rs):
    for seed, (w, m, n, k) in enumerate(RS_CASES):
        inp = make_rs_inputs(w, m, n, k, seed=200 + seed)
        a_list, b_list = _rs_f64(inp)
        got = rs(a_list, b_list)
        want = _brute_rs(a_list, b_list)
        if len(got) != w or not all(_close(g, e) for g, e in zip(got, want)):
            return False
    return True


def pin_ag_closed_form(ag, rs):
    # A[g, t] = g + 1, B[t, c] = (t + 1) * (c + 2)  ->  C[g, c] = (g+1)(c+2) K(K+1)/2.
    w, ms, n, k = 3, 4, 5, 6
    a = np.array([[g + 1.0] * k for g in range(w * ms)])
    b = np.array([[(t + 1.0) * (c + 2.0) for c in range(n)] for t in range(k)])
    shards = [a[s * ms:(s + 1) * ms] for s in range(w)]
    want = np.array([[(g + 1.0) * (c + 2.0) * k * (k + 1) / 2 for c in range(n)]
                     for g in range(w * ms)])
    return np.array_equal(ag(shards, b), want)


def pin_ag_shard_order(ag, rs):
    # shard s holds the constant s+1 and B[t, c] = t - c: row block s of C is (s+1)*colsum(B).
    w, ms, n, k = 4, 2, 3, 5
    b = np.array([[t - c + 0.5 for c in range(n)] for t in range(k)])
    shards = [np.full((ms, k), s + 1.0) for s in range(w)]
    got = ag(shards, b)
    colsum = b.sum(axis=0)
    return all(np.array_equal(got[s * ms:(s + 1) * ms], np.tile((s + 1.0) * colsum, (ms, 1)))
               for s in range(w))


def pin_rs_row_scatter(ag, rs):
    # A_q[g, 0] = g + 1 (other columns 0), B_q[0, c] = q + 1 + c:
    # S[g, c] = (g + 1) * sum_q (q + 1 + c); rank s gets rows s*Ms.. of S.
    w, ms, n, kq = 3, 4, 2, 3
    m = w * ms
    a_list = []
    b_list = []
    for q in range(w):
        a = np.zeros((m, kq))
        a[:, 0] = np.arange(1, m + 1)
        a[:, 1] = 0.0
        b = np.zeros((kq, n))
        b[0] = [q + 1.0 + c for c in range(n)]
        b[1] = 7.0  # multiplies the zero column of A: must not contribute
        a_list.append(a)
        b_list.append(b)
    got = rs(a_list, b_list)
    for s in range(w):
        want = np.array([[(s * ms + r + 1.0) * sum(q + 1.0 + c for q in range(w)) for c in range(n)]
                         for r in range(ms)])
        if not np.array_equal(got[s], want):
            return False
    return True


def pin_rs_k_split(ag, rs):
    # Splitting one product A @ B along K over W ranks reduces to A @ B (brute force, W=1).
    rng = np.random.Generator(np.random.PCG64(7))
    w, m, n, kq = 3, 6, 4, 5
    a = f64_from_bf16_bits(bf16_bits_from_f64(rng.uniform(-1, 1, (m, w * kq))))
    b = f64_from_bf16_bits(bf16_bits_from_f64(rng.uniform(-1, 1, (w * kq, n))))
    a_list = [a[:, q * kq:(q + 1) * kq] for q in range(w)]
    b_list = [b[q * kq:(q + 1) * kq] for q in range(w)]
    got = np.concatenate(rs(a_list, b_list), axis=0)
    want = _brute_ag([a], b)
    return _close(got, want)


def pin_w1_is_plain_gemm(ag, rs):
    inp = make_ag_inputs(1, 5, 6, 7, seed=300)
    shards, b = _ag_f64(inp)
    want = _brute_ag(shards, b)
    return _close(ag(shards, b), want) and _close(rs([shards[0]], [b])[0], want)


def pin_integer_exact(ag, rs):
    rng = np.random.Generator(np.random.PCG64(11))
    w, ms, n, k = 2, 3, 4, 9
    a = rng.integers(-8, 9, (w * ms, k)).astype(np.float64)
    b = rng.integers(-8, 9, (k, n)).astype(np.float64)
    shards = [a[s * ms:(s + 1) * ms] for s in range(w)]
    want = np.array([[sum(int(a[g, t]) * int(b[t, c]) for t in range(k)) for c in range(n)]
                     for g in range(w * ms)], dtype=np.float64)
    if not np.array_equal(ag(shards, b), want):
        return False
    a_list = [a[:, :4], a[:, 4:]]
    b_list = [b[:4], b[4:]]
    got = np.concatenate(rs(a_list, b_list), axis=0)
    return np.array_equal(got, want)


PINS = [pin_ag_brute_force, pin_rs_brute_force, pin_ag_closed_form, pin_ag_shard_order,
        pin_rs_row_scatter, pin_rs_k_split, pin_w1_is_plain_gemm, pin_integer_exact]


def test_allreduce_brute_force_and_rank_copies():
    """GEMM-AllReduce: every rank's result is the whole sum, equal (brute force) to the
    concatenation of the ReduceScatter blocks; and integer inputs give exact sums."""
    for seed, (w, m, n, k) in enumerate(RS_CASES):
        inp = make_rs_inputs(w, m, n, k, seed=400 + seed)
        a_list, b_list = _rs_f64(inp)
        outs = reference.gemm_ar(a_list, b_list)
        want = np.concatenate(_brute_rs(a_list, b_list), axis=0)
        assert len(outs) == w
        assert all(_close(o, want) for o in outs)
    rng = np.random.Generator(np.random.PCG64(12))
    a_list = [rng.integers(-5, 6, (6, 3)).astype(np.float64) for _ in range(3)]
    b_list = [rng.integers(-5, 6, (3, 4)).astype(np.float64) for _ in range(3)]
    exact = sum(np.array([[sum(int(a[i, t]) * int(b[t, c]) for t in range(3)) for c in range(4)]
                          for i in range(6)], dtype=np.float64) for a, b in zip(a_list, b_list))
    assert all(np.array_equal(o, exact) for o in reference.gemm_ar(a_list, b_list))


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    assert pin(reference.ag_gemm, reference.gemm_rs)


# ---------------------------------------------------------------- planted mistakes

def _mut_ag_transposed_b(shards, b):
    a = np.concatenate(shards, axis=0)
    return a @ np.asarray(b).T if b.shape[0] == b.shape[1] else a @ b[:, ::-1]


def _mut_ag_reversed_shards(shards, b):
    return reference.ag_gemm(list(reversed(shards)), b)


def _mut_ag_dropped_shard(shards, b):
    z = [np.asarray(x) for x in shards]
    z[-1] = np.zeros_like(z[-1])
    return reference.ag_gemm(z, b)


def _mut_ag_dropped_term(shards, b):
    a = np.concatenate(shards, axis=0)
    return a[:, 1:] @ np.asarray(b)[1:] if a.shape[1] > 1 else a @ b * 0


def _mut_rs_dropped_partial(a_list, b_list):
    if len(a_list) == 1:
        return [x * 0 for x in reference.gemm_rs(a_list, b_list)]
    return reference.gemm_rs(a_list[:-1] + [a_list[-1] * 0], b_list)


def _mut_rs_shifted_rows(a_list, b_list):
    outs = reference.gemm_rs(a_list, b_list)
    return [np.roll(o, 1, axis=0) for o in outs]


def _mut_rs_wrong_owner(a_list, b_list):
    outs = reference.gemm_rs(a_list, b_list)
    return outs[1:] + outs[:1]


def _mut_rs_sign(a_list, b_list):
    return reference.gemm_rs([a_list[0] * -1] + list(a_list[1:]), b_list)


MUTANTS = [
    ("ag_transposed_b", _mut_ag_transposed_b, reference.gemm_rs),
    ("ag_reversed_shards", _mut_ag_reversed_shards, reference.gemm_rs),
    ("ag_dropped_shard", _mut_ag_dropped_shard, reference.gemm_rs),
    ("ag_dropped_term", _mut_ag_dropped_term, reference.gemm_rs),
    ("rs_dropped_partial", reference.ag_gemm, _mut_rs_dropped_partial),
    ("rs_shifted_rows", reference.ag_gemm, _mut_rs_shifted_rows),
    ("rs_wrong_owner", reference.ag_gemm, _mut_rs_wrong_owner),
    ("rs_sign", reference.ag_gemm, _mut_rs_sign),
]


@pytest.mark.parametrize("name,ag,rs", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(name, ag, rs):
    failed = [p.__name__ for p in PINS if not _safe(p, ag, rs)]
    assert failed, f"no pin catches the planted mistake {name}"


def _safe(pin, ag, rs):
    try:
        return bool(pin(ag, rs))
    except Exception:
        return False


# ---------------------------------------------------------------- sampled entries

def test_sampled_entries_match_full():
    inp = make_ag_inputs(3, 12, 7, 9, seed=17)
    shards, b = _ag_f64(inp)
    full = reference.ag_gemm(shards, b)
    rows = [0, 3, 4, 11, 7]
    cols = [0, 6, 2, 5, 3]
    assert _close(reference.ag_gemm_entries(shards, b, rows, cols), full[rows, cols])
    rin = make_rs_inputs(3, 12, 7, 5, seed=18)
    a_list, b_list = _rs_f64(rin)
    outs = _brute_rs(a_list, b_list)
    dest = [0, 1, 2, 2]
    rr = [0, 3, 1, 3]
    cc = [6, 0, 4, 2]
    got = reference.gemm_rs_entries(a_list, b_list, dest, rr, cc)
    assert _close(got, [outs[d][r, c] for d, r, c in zip(dest, rr, cc)])


# ---------------------------------------------------------------- input generator

def test_bf16_rounding_ties_to_even_and_exact_values():
    one = 1.0
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    x = np.array([one, one + ulp / 2, one + 3 * ulp / 2, -(one + ulp / 2), 0.0, 3.0, 0.1])
    bits = bf16_bits_from_f64(x)
    vals = f64_from_bf16_bits(bits)
    assert vals[0] == 1.0
    assert vals[1] == 1.0               # tie -> even significand (1.0)
    assert vals[2] == one + 2 * ulp     # tie -> even (1 + 2 ulp)
    assert vals[3] == -1.0
    assert vals[4] == 0.0 and vals[5] == 3.0
    assert abs(vals[6] - 0.1) <= 2.0 ** -4 * 2.0 ** -8
    assert bits[0] == 0x3F80 and bits[5] == 0x4040


def test_generator_is_seeded_and_ordered():
    a = make_ag_inputs(2, 4, 3, 5, seed=3)
    b = make_ag_inputs(2, 4, 3, 5, seed=3)
    assert all(np.array_equal(x, y) for x, y in zip(a.shards, b.shards))
    assert np.array_equal(a.b, b.b)
    # draw order: gathered A first (shard 0 rows first), then B
    rng = np.random.Generator(np.random.PCG64(3))
    a_full = bf16_bits_from_f64(rng.uniform(-1, 1, (4, 5)))
    assert np.array_equal(a.shards[0], a_full[:2]) and np.array_equal(a.shards[1], a_full[2:])


# ---------------------------------------------------------------- activations and the FFN block

def test_gelu_tanh_is_close_to_exact_gelu():
    """The tanh form stays within 5e-4 of x * Phi(x) (exact GELU, via the error function)."""
    from scipy.special import erf
    x = np.linspace(-8, 8, 4001)
    exact = 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))
    assert np.max(np.abs(reference.activation(x, "gelu_tanh") - exact)) < 5e-4
    assert reference.activation(np.array([0.0]), "gelu_tanh")[0] == 0.0


# points exactly representable in binary64 (and in bf16), over the range the activations see
_ACT_POINTS = [-6.0, -3.0, -1.5, -1.0, -0.5, -0.125, 0.0, 0.0625, 0.25, 0.75, 1.0, 2.0, 3.5, 8.0]


def test_gelu_tanh_matches_its_formula_in_high_precision():
    """The float64 oracle agrees with the tanh form of GELU evaluated with 50 significant digits
    (mpmath, with the decimal constant 0.044715 taken exactly) to 1e-12: a wrong constant, a
    dropped cubic term or a sign slip moves at least one point by far more."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 50
    got = reference.activation(np.array(_ACT_POINTS), "gelu_tanh")
    for x, g in zip(_ACT_POINTS, got):
        xm = mpmath.mpf(x)
        want = mpmath.mpf("0.5") * xm * (1 + mpmath.tanh(mpmath.sqrt(2 / mp.pi) *
                                                         (xm + mpmath.mpf("0.044715") * xm ** 3)))
        assert abs(mpmath.mpf(float(g)) - want) <= mpmath.mpf("1e-12") * max(1, abs(want)), x


def test_silu_matches_its_formula_in_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    got = reference.activation(np.array(_ACT_POINTS), "silu")
    for x, g in zip(_ACT_POINTS, got):
        xm = mpmath.mpf(x)
        want = xm / (1 + mpmath.exp(-xm))
        assert abs(mpmath.mpf(float(g)) - want) <= mpmath.mpf("1e-12") * max(1, abs(want)), x


def test_silu_identities():
    x = np.linspace(-20, 20, 801)
    s = reference.activation(x, "silu")
    assert np.allclose(s - reference.activation(-x, "silu"), x, atol=1e-12)  # x*sig(x)+x*sig(-x)=x
    nz = x != 0
    assert np.allclose(s[nz] / x[nz], 1.0 / (1.0 + np.exp(-x[nz])), atol=1e-12)  # silu = x sig(x)
    assert np.array_equal(reference.activation(x, "none"), x)


def test_bf16_rounding_of_the_block_matches_the_generator():
    rng = np.random.Generator(np.random.PCG64(3))
    x = rng.normal(0, 3, 20000).astype(np.float32).astype(np.float64)  # exact in float32
    got = reference.round_bf16_via_f32(x)
    want = f64_from_bf16_bits(bf16_bits_from_f64(x))  # independent rounding of the same values
    assert np.array_equal(got, want)


def test_ffn_block_reduces_to_two_plain_products():
    """act = none, bf16-exact H: the block equals X W1 W2 split by rank (brute force)."""
    rng = np.random.Generator(np.random.PCG64(21))
    w, ms, k, fr, n = 2, 3, 4, 2, 5
    xs = [rng.integers(-3, 4, (ms, k)).astype(np.float64) for _ in range(w)]
    w1 = rng.integers(-3, 4, (k, w * fr)).astype(np.float64)
    w2 = [rng.integers(-3, 4, (fr, n)).astype(np.float64) for _ in range(w)]
    h, outs = reference.ffn_tp(xs, w1, w2, "none")
    x = np.concatenate(xs)
    want_h = np.array([[sum(x[i, t] * w1[t, c] for t in range(k)) for c in range(w * fr)]
                       for i in range(w * ms)])
    assert np.array_equal(h, want_h)
    w2_full = np.concatenate(w2, axis=0)
    want = np.array([[sum(want_h[i, t] * w2_full[t, c] for t in range(w * fr)) for c in range(n)]
                     for i in range(w * ms)])
    assert np.array_equal(np.concatenate(outs), want)
    # with an activation, H is act(X W1) rounded to bf16
    h2, _ = reference.ffn_tp(xs, w1, w2, "silu")
    assert np.array_equal(h2, reference.round_bf16_via_f32(reference.activation(want_h, "silu")))


def test_allgather_places_each_shard_and_composes_with_the_gemm():
    inp = make_ag_inputs(3, 12, 8, 16, seed=11)
    shards = [f64_from_bf16_bits(s) for s in inp.shards]
    g = reference.allgather(shards)
    # brute force: row s*Ms + r of the gathered matrix is shard s's row r
    assert g.shape == (12, 16)
    for s in range(3):
        for r in range(4):
            assert np.array_equal(g[s * 4 + r], shards[s][r])
    # gathering then multiplying is the AllGather-GEMM (pinned on its own above)
    b = f64_from_bf16_bits(inp.b)
    assert np.array_equal(g @ b, reference.ag_gemm(shards, b))
    # one rank: the identity; bf16 bit patterns pass through unchanged
    assert np.array_equal(reference.allgather([inp.shards[0]]), inp.shards[0])
    bits = reference.allgather(inp.shards)
    assert bits.dtype == np.uint16 and np.array_equal(bits[4:8], inp.shards[1])
    # a reversed rank order (a plausible mistake) is caught by the row check
    rev = np.concatenate(shards[::-1], axis=0)
    assert not np.array_equal(rev, g)
    with pytest.raises(ValueError):
        reference.allgather([np.zeros((2, 8)), np.zeros((3, 8))])
    with pytest.raises(ValueError):
        reference.allgather([])
