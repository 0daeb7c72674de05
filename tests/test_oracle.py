"""Pins for the CPU oracle.

Every check here compares the oracle with something other than itself:
a hand-worked example, closed forms, exact rational brute force, torch's own
BF16 rounding and RMSNorm, and invariants of the mathematics.  The pages
print no numeric example, so the hand-worked fixture in tests/golden/ stands
in for one.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import bf16_bits_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# exact-rational references (independent of the C oracle)
# ---------------------------------------------------------------------------

def _f32_neighbors(f):
    f = np.float32(f)
    return (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf)))


def round_to_f32(q: Fraction, zero_sign: float = 1.0) -> np.float32:
    """Nearest float32 to the rational q, ties to the even significand.
    Values here stay well inside the normal range, so no overflow handling."""
    if q == 0:
        return np.float32(math.copysign(0.0, zero_sign))
    approx = np.float32(float(q))
    best = None
    for c in _f32_neighbors(approx):
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - q)
        key = (d, int(np.array(c, dtype=np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    r = best[1]
    if r == 0:
        return np.float32(math.copysign(0.0, float(q)))
    return np.float32(r)


def fma_ref(a, b, c) -> np.float32:
    """IEEE fused multiply-add a*b+c on float32 operands, one rounding."""
    a, b, c = np.float32(a), np.float32(b), np.float32(c)
    exact = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    if exact == 0:
        prod_neg = (math.copysign(1, a) * math.copysign(1, b)) < 0
        prod_zero = (a == 0 or b == 0)
        c_neg = math.copysign(1, c) < 0
        # exact zero: -0 only when both addends are zeros of negative sign
        neg = prod_zero and c == 0 and prod_neg and c_neg
        return np.float32(-0.0 if neg else 0.0)
    return round_to_f32(exact)


def add_ref(a, b) -> np.float32:
    a, b = np.float32(a), np.float32(b)
    exact = Fraction(float(a)) + Fraction(float(b))
    if exact == 0:
        neg = a == 0 and b == 0 and math.copysign(1, a) < 0 and math.copysign(1, b) < 0
        return np.float32(-0.0 if neg else 0.0)
    return round_to_f32(exact)


def weighted_residual_ref(E_bits, idx, w, res):
    E = bf16_bits_to_f64(E_bits).astype(np.float32)
    T, k = idx.shape
    R, H = E.shape
    x = np.empty((T, H), dtype=np.float32)
    for t in range(T):
        for h in range(H):
            acc = np.float32(0.0)
            for j in range(k):
                r = int(idx[t, j])
                if 0 <= r < R:
                    acc = fma_ref(w[t, j], E[r, h], acc)
            x[t, h] = add_ref(res[t, h], acc)
    return x


def bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def bf16_bits_torch(x_f32):
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits_torch(rng.standard_normal(shape).astype(np.float32) * scale)


# ---------------------------------------------------------------------------
# BF16 rounding
# ---------------------------------------------------------------------------

def test_bf16_from_f64_matches_torch_rounding_on_fp32_values(oracle_lib):
    """Every float32 is a double; for those the one-step double->BF16
    rounding must equal torch's float32->BF16 nearest-even conversion."""
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    edges = np.array([0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF,
                      0x00800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000, 0xFF800000,
                      0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF, 0x7F7F8000,
                      0x7F7F7FFF, 0x00008000, 0x00018000, 0x00007FFF],
                     dtype=np.uint32)
    # every tie pattern in one binade, and its neighbours
    ties = (0x3F800000 | (np.arange(128, dtype=np.uint32) << 16) | 0x8000)
    pats = np.concatenate([pats, edges, ties, ties - 1, ties + 1])
    f = pats.view(np.float32)
    finite = ~np.isnan(f)
    got = oracle_lib.bf16_from_f64(f[finite].astype(np.float64))
    want = bf16_bits_torch(f[finite])
    assert np.array_equal(got, want)
    with np.errstate(invalid="ignore"):
        nan_in = f[np.isnan(f)].astype(np.float64)
    nan_out = oracle_lib.bf16_from_f64(nan_in)
    assert np.all((nan_out & 0x7F80) == 0x7F80) and np.all((nan_out & 0x007F) != 0)


def test_bf16_from_f64_rounds_once_from_double(oracle_lib):
    """Closed forms: ties go to even, and a double just above a tie rounds up
    even when its nearest float32 sits exactly on the tie."""
    cases = [
        (1.0 + 2.0**-8, 0x3F80),               # tie between 1 and 1+2^-7 -> even (1)
        (1.0 + 2.0**-8 + 2.0**-40, 0x3F81),    # above the tie -> up (float32 path gives 0x3F80)
        (1.0 + 3 * 2.0**-8, 0x3F82),           # tie between mantissas 1 and 2 -> 2
        (-(1.0 + 3 * 2.0**-8), 0xBF82),
        (1.0 + 2.0**-8 - 2.0**-40, 0x3F80),
        (2.0**-133, 0x0001),                   # smallest subnormal
        (2.0**-134, 0x0000),                   # tie between 0 and 2^-133 -> 0
        (3 * 2.0**-134, 0x0002),               # tie between 1 and 2 units -> 2
        (-2.0**-134, 0x8000),
        ((2 - 2.0**-8) * 2.0**127, 0x7F80),    # tie above max finite -> even -> inf
        ((2 - 2.0**-8 - 2.0**-30) * 2.0**127, 0x7F7F),
        (2.0**200, 0x7F80),
        (-2.0**200, 0xFF80),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (1e-300, 0x0000),
        (-1e-300, 0x8000),
        (math.inf, 0x7F80),
        (-math.inf, 0xFF80),
    ]
    xs = np.array([c[0] for c in cases], dtype=np.float64)
    got = oracle_lib.bf16_from_f64(xs)
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    assert np.array_equal(got, want), [(x, hex(g), hex(w)) for x, g, w in zip(xs, got, want) if g != w]
    # the float32-then-BF16 route double-rounds the second case
    assert bf16_bits_torch(np.array([1.0 + 2.0**-8 + 2.0**-40], dtype=np.float32))[0] == 0x3F80


def test_bf16_from_f64_is_nearest_on_random_doubles(oracle_lib):
    """Definition check: the result is no farther from x than either BF16
    neighbour, and on an exact tie it has an even significand."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(50_000) * np.exp2(rng.integers(-20, 20, size=50_000))
    b = oracle_lib.bf16_from_f64(x)
    v = bf16_bits_to_f64(b)
    up = bf16_bits_to_f64((b.astype(np.int64) + 1).astype(np.uint16))
    dn = bf16_bits_to_f64((b.astype(np.int64) - 1).astype(np.uint16))
    d = np.abs(v - x)
    assert np.all(d <= np.abs(up - x)) and np.all(d <= np.abs(dn - x))


# ---------------------------------------------------------------------------
# the hand-worked example
# ---------------------------------------------------------------------------

def _golden():
    with open(os.path.join(GOLDEN, "hand_worked_t2_h8_k2.json")) as f:
        g = json.load(f)
    E = bf16_bits_torch(np.array(g["expert_out"], dtype=np.float32))
    gamma = np.array([int(s, 16) for s in g["gamma_bits"]], dtype=np.uint16)
    assert np.array_equal(bf16_bits_to_f64(gamma), np.array(g["gamma"], dtype=np.float64))
    return g, E, gamma


def test_hand_worked_example(oracle_lib):
    g, E, gamma = _golden()
    idx = np.array(g["permuted_row_of"], dtype=np.int32)
    w = np.array(g["topk_weights"], dtype=np.float32)
    res = np.array(g["residual_in"], dtype=np.float32)
    res_out, out, bad = oracle_lib.finalize_residual_rmsnorm(E, idx, w, res, gamma, g["eps"])
    assert bad == 0
    assert np.array_equal(bits(res_out), bits(np.array(g["expected_residual_out"], dtype=np.float32)))
    want = np.array([[int(s, 16) for s in row] for row in g["expected_out_bits"]], dtype=np.uint16)
    assert np.array_equal(out, want), (out, want)
    fin, bad = oracle_lib.finalize_only(E, idx, w)
    want_fin = np.array([[int(s, 16) for s in row] for row in g["expected_weighted_sum_bf16_bits"]],
                        dtype=np.uint16)
    assert np.array_equal(fin, want_fin)


# ---------------------------------------------------------------------------
# gather + FP32 FMA + residual
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (2, 16, 2), (3, 24, 8), (3, 8, 3), (2, 24, 5)])
def test_weighted_residual_brute_force_exact(oracle_lib, T, H, k):
    """Exact rational arithmetic, one rounding per FMA and per add."""
    rng = np.random.default_rng(100 + T * 31 + H + k)
    R = T * k + 3
    E = rand_bf16(rng, (R, H), 3.0)
    idx = np.stack([rng.permutation(R)[:k] for _ in range(T)]).astype(np.int32)
    w = (rng.standard_normal((T, k)) * 0.7).astype(np.float32)
    w[0, 0] = 0.0
    res = rng.standard_normal((T, H)).astype(np.float32)
    got, bad = oracle_lib.weighted_residual(E, idx, w, res)
    assert bad == 0
    want = weighted_residual_ref(E, idx, w, res)
    assert np.array_equal(bits(got), bits(want))


def test_weighted_residual_all_slot_orders_k3(oracle_lib):
    """For every order of the three slots the oracle follows the stated slot
    order exactly, and the order does matter for these values."""
    H = 4
    E = bf16_bits_torch(np.array([[1, 3, 1, 0.5], [2.0**24, -7, 2.0**20, 1],
                                  [-2.0**24, 5, -2.0**20, -1]], dtype=np.float32))
    res = np.array([[0.25, 0, 0, 2]], dtype=np.float32)
    base_w = np.array([1.0, 1.0, 1.0], dtype=np.float32)
    results = set()
    for perm in itertools.permutations(range(3)):
        idx = np.array([perm], dtype=np.int32)
        w = base_w[list(perm)][None, :]
        got, _ = oracle_lib.weighted_residual(E, idx, w, res)
        want = weighted_residual_ref(E, idx, w, res)
        assert np.array_equal(bits(got), bits(want))
        results.add(tuple(bits(got)[0]))
    assert len(results) > 1  # order-sensitive, as FP32 accumulation must be


def test_k1_unit_weight_is_residual_plus_row(oracle_lib):
    """k = 1 with weight 1: fma(1, e, 0) = e, so x = residual + row (one FP32 add,
    done here by NumPy), and the output is RMSNorm of that row (torch, float64)."""
    rng = np.random.default_rng(3)
    T, H, R = 5, 64, 9
    E = rand_bf16(rng, (R, H))
    idx = rng.integers(0, R, size=(T, 1)).astype(np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    gamma = bf16_bits_torch((1 + 0.3 * rng.standard_normal(H)).astype(np.float32))
    eps = 1e-6
    res_out, out, _ = oracle_lib.finalize_residual_rmsnorm(E, idx, w, res, gamma, eps)
    Ef = bf16_bits_to_f64(E).astype(np.float32)
    want_x = res + Ef[idx[:, 0]]
    assert np.array_equal(bits(res_out), bits(want_x))
    y = oracle_lib.rmsnorm_f64(res_out, gamma, eps)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(want_x.astype(np.float64)), (H,),
                                       weight=torch.from_numpy(bf16_bits_to_f64(gamma)), eps=eps)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13, atol=0)


def test_one_hot_weights_select_one_row(oracle_lib):
    rng = np.random.default_rng(4)
    T, H, k = 4, 32, 8
    R = T * k
    E = rand_bf16(rng, (R, H))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    Ef = bf16_bits_to_f64(E).astype(np.float32)
    for j in range(k):
        w = np.zeros((T, k), dtype=np.float32)
        w[:, j] = 1.0
        got, _ = oracle_lib.weighted_residual(E, idx, w, res)
        assert np.array_equal(bits(got), bits(res + Ef[idx[:, j]]))


def test_exact_integer_closed_form(oracle_lib):
    """Small-integer rows and power-of-two weights keep every partial sum
    exact in FP32, so x equals the order-free float64 sum bit for bit."""
    rng = np.random.default_rng(5)
    T, H, k = 6, 40, 8
    R = T * k + 5
    Ev = rng.integers(-64, 65, size=(R, H)).astype(np.float32)
    E = bf16_bits_torch(Ev)
    assert np.array_equal(bf16_bits_to_f64(E), Ev.astype(np.float64))
    idx = np.stack([rng.permutation(R)[:k] for _ in range(T)]).astype(np.int32)
    w = (np.exp2(rng.integers(-3, 3, size=(T, k))) * rng.choice([-1, 1], size=(T, k))).astype(np.float32)
    res = rng.integers(-1000, 1000, size=(T, H)).astype(np.float32)
    got, _ = oracle_lib.weighted_residual(E, idx, w, res)
    want = res.astype(np.float64) + np.einsum("tk,tkh->th", w.astype(np.float64),
                                              Ev.astype(np.float64)[idx])
    assert np.array_equal(got.astype(np.float64), want)


def test_identity_permutation_matches_dense_sum_within_fp32_bound(oracle_lib):
    rng = np.random.default_rng(6)
    T, H, k = 7, 256, 8
    R = T * k
    E = rand_bf16(rng, (R, H))
    idx = np.arange(R, dtype=np.int32).reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    got, _ = oracle_lib.weighted_residual(E, idx, w, res)
    Ef = bf16_bits_to_f64(E).reshape(T, k, H)
    terms = w.astype(np.float64)[:, :, None] * Ef
    dense = res.astype(np.float64) + terms.sum(axis=1)
    u = 2.0**-24
    bound = (k + 1) * u * (np.abs(terms).sum(axis=1) + np.abs(res))
    assert np.all(np.abs(got - dense) <= bound)
    assert np.abs(got - dense).max() > 0  # really FP32, not exact


def test_regrouping_rows_is_invisible(oracle_lib):
    """Moving the rows of expert_out around, with the index map following,
    leaves every output bit unchanged."""
    rng = np.random.default_rng(7)
    T, H, k = 5, 48, 8
    R = T * k + 2
    E = rand_bf16(rng, (R, H))
    idx = np.stack([rng.permutation(R)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    gamma = rand_bf16(rng, (H,))
    a = oracle_lib.finalize_residual_rmsnorm(E, idx, w, res, gamma, 1e-6)
    perm = rng.permutation(R)             # new row p holds old row perm[p]
    inv = np.empty(R, dtype=np.int64)
    inv[perm] = np.arange(R)
    b = oracle_lib.finalize_residual_rmsnorm(E[perm], inv[idx].astype(np.int32), w, res, gamma, 1e-6)
    assert np.array_equal(bits(a[0]), bits(b[0])) and np.array_equal(a[1], b[1])


def test_out_of_range_slots_contribute_nothing_and_are_counted(oracle_lib):
    rng = np.random.default_rng(8)
    T, H, k = 3, 16, 4
    R = 10
    E = rand_bf16(rng, (R, H))
    idx = np.array([[1, -1, 3, 4], [R, 2, 5, R + 7], [0, 1, 2, 3]], dtype=np.int32)
    w = rng.random((T, k)).astype(np.float32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    got, bad = oracle_lib.weighted_residual(E, idx, w, res)
    assert bad == 3
    want = weighted_residual_ref(E, idx, w, res)
    assert np.array_equal(bits(got), bits(want))
    # same as dropping those slots
    t0, _ = oracle_lib.weighted_residual(E, idx[:1, [0, 2, 3]], w[:1, [0, 2, 3]], res[:1])
    assert np.array_equal(bits(got[:1]), bits(t0))
    t1, _ = oracle_lib.weighted_residual(E, idx[1:2, [1, 2]], w[1:2, [1, 2]], res[1:2])
    assert np.array_equal(bits(got[1:2]), bits(t1))


def test_duplicate_rows_are_read_twice(oracle_lib):
    rng = np.random.default_rng(9)
    H = 16
    E = rand_bf16(rng, (3, H))
    idx = np.array([[2, 2]], dtype=np.int32)
    w = np.array([[0.75, 0.5]], dtype=np.float32)
    res = rng.standard_normal((1, H)).astype(np.float32)
    got, _ = oracle_lib.weighted_residual(E, idx, w, res)
    assert np.array_equal(bits(got), bits(weighted_residual_ref(E, idx, w, res)))


def test_token_subset_equals_full_run(oracle_lib):
    rng = np.random.default_rng(10)
    T, H, k = 9, 24, 3
    R = T * k
    E = rand_bf16(rng, (R, H))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    gamma = rand_bf16(rng, (H,))
    full = oracle_lib.finalize_residual_rmsnorm(E, idx, w, res, gamma, 1e-5)
    sub = [7, 0, 3]
    part = oracle_lib.finalize_residual_rmsnorm(E, idx, w, res, gamma, 1e-5, tokens=sub)
    assert np.array_equal(bits(full[0][sub]), bits(part[0]))
    assert np.array_equal(full[1][sub], part[1])


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_matches_torch_float64(oracle_lib):
    rng = np.random.default_rng(11)
    for H, eps in [(8, 1e-6), (24, 0.5), (4096, 1e-5), (136, 0.0)]:
        x = (rng.standard_normal((4, H)) * rng.choice([1e-3, 1.0, 50.0])).astype(np.float32)
        gamma = rand_bf16(rng, (H,))
        y = oracle_lib.rmsnorm_f64(x, gamma, eps)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x.astype(np.float64)), (H,),
                                           weight=torch.from_numpy(bf16_bits_to_f64(gamma)),
                                           eps=float(np.float32(eps)))
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-300)


def test_rmsnorm_constant_row_closed_form(oracle_lib):
    """x = c everywhere: y = c / sqrt(c^2 + eps) * gamma.  eps = 3 and c = 1
    makes the scale exactly 1/2, which separates 'eps inside the root' from
    every other placement, mean from sum, and gamma from 1 + gamma."""
    H = 32
    gamma = bf16_bits_torch(np.linspace(-2, 2, H).astype(np.float32))
    g = bf16_bits_to_f64(gamma)
    y = oracle_lib.rmsnorm_f64(np.ones((1, H), dtype=np.float32), gamma, 3.0)
    assert np.array_equal(y[0], 0.5 * g)
    for c, eps in [(2.5, 1e-6), (-7.0, 0.25), (1e-3, 1e-6)]:
        y = oracle_lib.rmsnorm_f64(np.full((1, H), c, dtype=np.float32), gamma, eps)
        c32 = float(np.float32(c))
        want = c32 / math.sqrt(c32 * c32 + float(np.float32(eps))) * g
        np.testing.assert_allclose(y[0], want, rtol=1e-14)


def test_rmsnorm_unit_rms_as_eps_vanishes(oracle_lib):
    rng = np.random.default_rng(12)
    H = 4096
    x = rng.standard_normal((3, H)).astype(np.float32)
    gamma = bf16_bits_torch((1 + 0.3 * rng.standard_normal(H)).astype(np.float32))
    gamma[gamma == 0] = 0x3F80
    y = oracle_lib.rmsnorm_f64(x, gamma, 1e-12)
    rms = np.sqrt(np.mean((y / bf16_bits_to_f64(gamma)) ** 2, axis=1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-9)
    # and on the BF16 output, within the BF16 rounding
    E = bf16_bits_torch(x)
    idx = np.arange(3, dtype=np.int32)[:, None]
    w = np.ones((3, 1), dtype=np.float32)
    _, out, _ = oracle_lib.finalize_residual_rmsnorm(E, idx, w, np.zeros_like(x), gamma, 1e-12)
    rms_out = np.sqrt(np.mean((bf16_bits_to_f64(out) / bf16_bits_to_f64(gamma)) ** 2, axis=1))
    assert np.all(np.abs(rms_out - 1.0) < 2.0**-7)


def test_rmsnorm_power_of_two_scaling_invariant(oracle_lib):
    rng = np.random.default_rng(13)
    H = 100
    x = rng.standard_normal((2, H)).astype(np.float32)
    gamma = rand_bf16(rng, (H,))
    y = oracle_lib.rmsnorm_f64(x, gamma, 0.0)
    for m in (-20, -3, 5, 30):
        ys = oracle_lib.rmsnorm_f64((x * np.float32(2.0**m)).astype(np.float32), gamma, 0.0)
        assert np.array_equal(y, ys)


def test_output_is_nearest_bf16_of_norm(oracle_lib):
    rng = np.random.default_rng(14)
    T, H, k = 4, 64, 8
    R = T * k
    E = rand_bf16(rng, (R, H))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    res = rng.standard_normal((T, H)).astype(np.float32)
    gamma = rand_bf16(rng, (H,))
    res_out, out, _ = oracle_lib.finalize_residual_rmsnorm(E, idx, w, res, gamma, 1e-6)
    y = oracle_lib.rmsnorm_f64(res_out, gamma, 1e-6)
    v = bf16_bits_to_f64(out)
    up = bf16_bits_to_f64((out.astype(np.int64) + 1).astype(np.uint16))
    dn = bf16_bits_to_f64((out.astype(np.int64) - 1).astype(np.uint16))
    assert np.all(np.abs(v - y) <= np.abs(up - y)) and np.all(np.abs(v - y) <= np.abs(dn - y))


def test_finalize_only_is_rounded_weighted_sum(oracle_lib):
    rng = np.random.default_rng(15)
    T, H, k = 3, 24, 8
    R = T * k
    E = rand_bf16(rng, (R, H))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    got, _ = oracle_lib.finalize_only(E, idx, w)
    acc = weighted_residual_ref(E, idx, w, np.zeros((T, H), dtype=np.float32))
    assert np.array_equal(got, bf16_bits_torch(acc))
