"""Pins for the oracle's per-expert RMSNorm reading of the finalize:
out[t] = BF16(sum_j w[t,j] * RMSNorm(E[idx[t,j]]) * gamma), no residual.

They tie it to things other than its own formula: torch's RMSNorm in
float64 for each row, closed forms on constant rows (which separate a norm
per expert from a norm of the sum, eps inside the root, mean from sum and
gamma from 1 + gamma), exact invariance of each row's normalised value under
power-of-two scaling of that row alone, and the index-map rules shared with
the other paths."""
import numpy as np
import torch

from oracle import bf16_bits_to_f64
from test_oracle import bf16_bits_torch, rand_bf16


def torch_rms_rows(E_bits, gamma_bits, eps):
    e = torch.from_numpy(bf16_bits_to_f64(E_bits))
    g = torch.from_numpy(bf16_bits_to_f64(gamma_bits))
    return torch.nn.functional.rms_norm(e, (e.shape[-1],), weight=g, eps=float(np.float32(eps))).numpy()


def test_single_slot_is_torch_rms_norm_of_the_row(oracle_lib):
    rng = np.random.default_rng(41)
    for H, eps, wv in [(8, 1e-6, 1.0), (64, 0.5, 0.75), (4096, 1e-5, -2.0), (136, 0.0, 1.0)]:
        R, T = 7, 5
        E = rand_bf16(rng, (R, H), scale=float(rng.choice([1e-2, 1.0, 30.0])))
        gamma = rand_bf16(rng, (H,))
        idx = rng.integers(0, R, size=(T, 1)).astype(np.int32)
        w = np.full((T, 1), wv, dtype=np.float32)
        y, bad = oracle_lib.expert_rmsnorm_f64(E, idx, w, gamma, eps)
        assert bad == 0
        want = wv * torch_rms_rows(E, gamma, eps)[idx[:, 0]]
        np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-300)


def test_weighted_sum_of_torch_row_norms(oracle_lib):
    rng = np.random.default_rng(42)
    T, H, k = 4, 96, 8
    R = T * k + 3
    E = rand_bf16(rng, (R, H), scale=3.0)
    gamma = rand_bf16(rng, (H,))
    idx = rng.permutation(R)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y, _ = oracle_lib.expert_rmsnorm_f64(E, idx, w, gamma, 1e-6)
    n = torch_rms_rows(E, gamma, 1e-6)
    want = np.einsum("tj,tjh->th", w.astype(np.float64), n[idx])
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-14)


def test_constant_rows_closed_form(oracle_lib):
    """Rows of +1 and of -1 with eps = 3 normalise to exactly +gamma/2 and
    -gamma/2; weights (1, 0.25) give exactly 0.375 gamma.  A norm of the
    weighted sum would give 0.75 / sqrt(0.5625 + 3) gamma instead."""
    H = 32
    gamma = bf16_bits_torch(np.linspace(-2, 2, H).astype(np.float32))
    g = bf16_bits_to_f64(gamma)
    E = bf16_bits_torch(np.stack([np.ones(H), -np.ones(H)]).astype(np.float32))
    idx = np.array([[0, 1]], dtype=np.int32)
    w = np.array([[1.0, 0.25]], dtype=np.float32)
    y, _ = oracle_lib.expert_rmsnorm_f64(E, idx, w, gamma, 3.0)
    assert np.array_equal(y[0], 0.375 * g)
    for c, eps in [(2.5, 1e-6), (-7.0, 0.25), (1e-3, 1e-6)]:
        Ec = bf16_bits_torch(np.full((1, H), c, dtype=np.float32))
        cb = float(bf16_bits_to_f64(Ec)[0, 0])
        y, _ = oracle_lib.expert_rmsnorm_f64(Ec, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), gamma, eps)
        np.testing.assert_allclose(y[0], cb / np.sqrt(cb * cb + float(np.float32(eps))) * g, rtol=1e-14)


def test_scaling_one_row_by_a_power_of_two_changes_nothing(oracle_lib):
    """With eps = 0 each row's normalised value is invariant under scaling
    that row alone by 2^m, so the weighted sum is unchanged bit for bit."""
    rng = np.random.default_rng(43)
    T, H, k = 3, 48, 4
    R = T * k
    Ef = rng.standard_normal((R, H)).astype(np.float32)
    E = bf16_bits_torch(Ef)
    gamma = rand_bf16(rng, (H,))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y, _ = oracle_lib.expert_rmsnorm_f64(E, idx, w, gamma, 0.0)
    for row, m in [(int(idx[1, 2]), 7), (int(idx[0, 0]), -9)]:
        E2 = E.copy()
        E2[row] = bf16_bits_torch(bf16_bits_to_f64(E[row]).astype(np.float32) * np.float32(2.0 ** m))
        y2, _ = oracle_lib.expert_rmsnorm_f64(E2, idx, w, gamma, 0.0)
        assert np.array_equal(y, y2)


def test_out_of_range_slots_add_nothing_and_are_counted(oracle_lib):
    rng = np.random.default_rng(44)
    T, H, k = 3, 40, 4
    R = T * k
    E = rand_bf16(rng, (R, H))
    gamma = rand_bf16(rng, (H,))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    bad_idx = idx.copy()
    bad_idx[0, 1] = -1
    bad_idx[2, 3] = R
    bad_idx[2, 0] = 2 ** 31 - 1
    y, bad = oracle_lib.expert_rmsnorm_f64(E, bad_idx, w, gamma, 1e-6)
    assert bad == 3
    w0 = w.copy()
    w0[0, 1] = w0[2, 3] = w0[2, 0] = 0.0
    want, bad0 = oracle_lib.expert_rmsnorm_f64(E, idx, w0, gamma, 1e-6)
    assert bad0 == 0
    assert np.array_equal(y, want)


def test_duplicate_rows_count_twice(oracle_lib):
    rng = np.random.default_rng(45)
    H = 24
    E = rand_bf16(rng, (3, H))
    gamma = rand_bf16(rng, (H,))
    w = np.array([[0.5, 0.25]], dtype=np.float32)
    y, _ = oracle_lib.expert_rmsnorm_f64(E, np.array([[2, 2]], np.int32), w, gamma, 1e-6)
    y1, _ = oracle_lib.expert_rmsnorm_f64(E, np.array([[2]], np.int32), np.array([[0.75]], np.float32), gamma, 1e-6)
    np.testing.assert_allclose(y, y1, rtol=1e-15)


def test_output_is_the_nearest_bf16_and_tokens_select_rows(oracle_lib):
    rng = np.random.default_rng(46)
    T, H, k = 6, 64, 8
    R = T * k
    E = rand_bf16(rng, (R, H))
    gamma = rand_bf16(rng, (H,))
    idx = rng.permutation(R).reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    out, _ = oracle_lib.finalize_expert_rmsnorm(E, idx, w, gamma, 1e-6)
    y, _ = oracle_lib.expert_rmsnorm_f64(E, idx, w, gamma, 1e-6)
    v = bf16_bits_to_f64(out)
    up = bf16_bits_to_f64((out.astype(np.int64) + 1).astype(np.uint16))
    dn = bf16_bits_to_f64((out.astype(np.int64) - 1).astype(np.uint16))
    assert np.all(np.abs(v - y) <= np.abs(up - y)) and np.all(np.abs(v - y) <= np.abs(dn - y))
    sub = [5, 0, 3]
    part, _ = oracle_lib.finalize_expert_rmsnorm(E, idx, w, gamma, 1e-6, tokens=sub)
    assert np.array_equal(part, out[sub])


def test_hand_worked_example(oracle_lib):
    """tests/golden/expert_rmsnorm_hand_worked.json: two tokens worked by hand
    (powers of two throughout, so every value is exact and so are the BF16
    results)."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "expert_rmsnorm_hand_worked.json")
    g = json.load(open(path))
    E = np.array([[int(b, 16) for b in row] for row in g["expert_out_bits"]], dtype=np.uint16)
    gamma = np.array([int(b, 16) for b in g["gamma_bits"]], dtype=np.uint16)
    np.testing.assert_array_equal(bf16_bits_to_f64(E), np.array(g["expert_out"], dtype=np.float64))
    np.testing.assert_array_equal(bf16_bits_to_f64(gamma), np.array(g["gamma"], dtype=np.float64))
    idx = np.array(g["permuted_row_of"], dtype=np.int32)
    w = np.array(g["topk_weights"], dtype=np.float32)
    y, bad = oracle_lib.expert_rmsnorm_f64(E, idx, w, gamma, g["eps"])
    assert bad == 0
    np.testing.assert_array_equal(y, np.array(g["expected_out"], dtype=np.float64))
    out, bad = oracle_lib.finalize_expert_rmsnorm(E, idx, w, gamma, g["eps"])
    assert bad == 0
    want = np.array([[int(b, 16) for b in row] for row in g["expected_out_bits"]], dtype=np.uint16)
    np.testing.assert_array_equal(out, want)
