"""The seeded input generators: shapes, the grouped index map, determinism."""
import numpy as np
import torch

import workloads as W


def test_named_configs_have_the_stated_shapes():
    n = W.all_named()
    assert n["tiny_ref"].T == 16 and n["tiny_ref"].H == 4096 and n["tiny_ref"].E == 64
    assert n["prefill"].T == 16384 and n["prefill"].E == 128 and n["prefill"].zipf_s == 1.2
    assert n["stress"].T == 32768 and n["stress"].H == 8192 and n["stress"].E == 256
    assert [n[f"decode_T{t}"].T for t in W.DECODE_TOKENS] == [1, 2, 4, 8, 16, 32, 64, 128]
    assert all(n[f"wide_T{t}"].H == 8192 for t in W.WIDE_TOKENS)
    assert all(wl.k == 8 for wl in n.values())


def test_algorithmic_bytes_formula():
    assert W.algorithmic_bytes(1, 4096, 8) == 106_560
    assert W.algorithmic_bytes(16384, 4096, 8) == 1_745_879_040
    assert W.algorithmic_bytes(32768, 8192, 8) == 6_981_419_008


def test_index_map_is_the_stable_expert_grouping():
    d = W.make_inputs(W.TINY_REF)
    T, k = 16, 8
    idx = d["permuted_row_of"].numpy()
    eo = d["expert_of"]
    assert sorted(idx.reshape(-1).tolist()) == list(range(T * k))
    # walking rows in order visits experts in non-decreasing order, and within
    # one expert the (token, slot) pairs in increasing flat order
    pair_of_row = np.empty(T * k, dtype=np.int64)
    pair_of_row[idx.reshape(-1)] = np.arange(T * k)
    experts = eo.reshape(-1)[pair_of_row]
    assert np.all(np.diff(experts) >= 0)
    same = np.diff(experts) == 0
    assert np.all(np.diff(pair_of_row)[same] > 0)
    # k distinct experts per token, weights a descending softmax
    assert all(len(set(r)) == k for r in eo.tolist())
    w = d["topk_weights"].numpy()
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_generation_is_deterministic_and_seeded():
    a = W.make_inputs(W.decode(8))
    b = W.make_inputs(W.decode(8))
    c = W.make_inputs(W.decode(8).with_(seed=1))
    for key in ("expert_out", "permuted_row_of", "topk_weights", "residual", "gamma"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["expert_out"], c["expert_out"])


def test_zipf_routing_is_skewed_and_uniform_is_not():
    z = W.make_inputs(W.PREFILL, T=2048)["expert_of"]
    counts = np.bincount(z.reshape(-1), minlength=128)
    assert counts[0] > 5 * counts[64]
    u = W.make_inputs(W.decode(128), T=2048)["expert_of"]
    cu = np.bincount(u.reshape(-1), minlength=128)
    assert cu.max() < 2.0 * cu.mean()


def test_stress_outliers_and_unnormalised_weights():
    d = W.make_inputs(W.STRESS, T=64)
    n_out = round(0.01 * 64 * 8)
    assert len(d["outlier_rows"]) == n_out == len(set(d["outlier_rows"].tolist()))
    e = d["expert_out"].float()
    big = e[torch.as_tensor(d["outlier_rows"])].abs().mean()
    rest = np.setdiff1d(np.arange(64 * 8), d["outlier_rows"])
    assert big > 30 * e[torch.as_tensor(rest)].abs().mean()
    w = d["topk_weights"].numpy()
    assert np.all((w >= 0) & (w < 1)) and not np.allclose(w.sum(axis=1), 1.0)


def test_variances_follow_the_mean_variance_notation():
    d = W.make_inputs(W.wide(512))
    assert abs(d["residual"].std().item() - 2.0) < 0.02
    assert abs(d["expert_out"].float().std().item() - 0.5 ** 0.5) < 0.01
    assert abs(d["gamma"].float().mean().item() - 1.0) < 0.02
