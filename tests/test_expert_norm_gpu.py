"""The finalize with an RMSNorm per expert row (the reading of the PR 6544
page, section 2.1, built by moe_finalize_expert_rmsnorm_*) against the
oracle's finalize_expert_rmsnorm.

The oracle sums in double and the kernel in FP32 (per-row sums of squares in
a fixed tree, rsqrtf, FMAs in slot order), so the bar is: the bf16 output
within 1 ulp of the oracle's, or, where the weighted sum cancels, within the
FP32 error bound 2^-18 * S (S = the same sum over |w|, |E|, |gamma|; a
bound over k + 20 roundings of 2^-24 each) plus half an ulp of the result.
Repeated runs are bitwise identical."""
import ctypes

import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
import oracle
from helpers import bf16_bits, bf16_ulp_distance, host_inputs, oracle_expert_norm, over_all_tokens

pytestmark = pytest.mark.gpu
GUARD = 256
FP32_BOUND = 2.0 ** -18


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def run_expert_norm(inp, plan=None, **plan_kw):
    e, idx, w, g = inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["gamma"]
    T, k = idx.shape
    R, H = e.shape
    if plan is None:
        plan = mfr.ExpertNormPlan(T, H, k, R, **plan_kw)
    buf = torch.full((T * H + 2 * GUARD,), -5.0, dtype=torch.bfloat16, device="cuda")
    out = buf[GUARD:GUARD + T * H].view(T, H)
    plan.run(e, idx, w, g, inp["eps"], out)
    torch.cuda.synchronize()
    assert torch.all(buf[:GUARD] == -5.0) and torch.all(buf[-GUARD:] == -5.0), "a kernel wrote outside out"
    return bf16_bits(out), plan


def assert_expert_norm_close(got_bits, want_bits, y, s):
    d = bf16_ulp_distance(got_bits, want_bits)
    got = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    half_ulp = np.abs(got) * 2.0 ** -8      # at least half a bf16 ulp of got
    ok = (d <= 1) | (np.abs(got - y) <= FP32_BOUND * s + half_ulp)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"{(~ok).sum()} outputs out of tolerance; first at {i}: got {got[i]!r} "
                             f"oracle {y[i]!r} (bf16 0x{int(want_bits[i]):04x}), scale {s[i]!r}")


@pytest.mark.parametrize("T,H,k", [(1, 4096, 8), (5, 24, 3), (16, 4096, 8), (100, 8192, 8), (7, 4104, 16),
                                   (153, 1032, 1), (3, 16384, 8), (9, 8, 5), (160, 4104, 5), (305, 2048, 8),
                                   (40, 6144, 8), (20, 8000, 6)])
@pytest.mark.parametrize("variant", [mfr.VARIANT_AUTO, mfr.VARIANT_ROWS, mfr.VARIANT_STREAM, mfr.VARIANT_CLUSTER],
                         ids=["auto", "rows", "ring", "cluster"])
@pytest.mark.parametrize("pdl", [True, False])
def test_expert_norm_matches_oracle(T, H, k, variant, pdl):
    if variant == mfr.VARIANT_STREAM and (k > 8 or H > 8192):
        pytest.skip("the ring form holds at most 8 slots and 4 column tiles")
    if variant == mfr.VARIANT_CLUSTER and (k > 8 or (H // 8) % 2):
        pytest.skip("the cluster form holds at most 8 slots and splits H/8 evenly")
    wl = W.Workload(f"en_T{T}_H{H}", T=T, H=H, k=k, E=max(16, 2 * k), seed=T * 11 + H + k, extra_rows=3)
    inp = W.make_inputs(wl, "cuda")
    want, y, s, bad = oracle_expert_norm(inp)
    got, plan = run_expert_norm(inp, enable_pdl=pdl, variant=variant)
    assert bad == 0
    assert_expert_norm_close(got, want, y, s)
    assert np.mean(got != want) < 0.02
    assert plan.get_status() == 0
    info = plan.info()
    if variant == mfr.VARIANT_AUTO:
        small = k <= 8 and T * H <= 1 << 19
        assert info["variant"] in ((mfr.VARIANT_CLUSTER, mfr.VARIANT_ROWS) if small else (mfr.VARIANT_ROWS,))
    else:
        assert info["variant"] == variant
    assert (info["cluster"] > 1) == (info["variant"] == mfr.VARIANT_CLUSTER)
    again, _ = run_expert_norm(inp, plan=plan)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("T,H,k", [(2000, 4096, 2), (1200, 8192, 4), (1500, 4096, 7)])
def test_expert_norm_ring_wraps(T, H, k):
    """The ring form with fewer than 8 slots (deeper rings) and many tokens
    per CTA, so the ring wraps many times; at H = 8192 two of a token's four
    stages are held for the second pass.  Every token against the oracle;
    a repeated run is bitwise equal."""
    wl = W.Workload(f"en_ring_T{T}_H{H}_k{k}", T=T, H=H, k=k, E=16, seed=T + H + k, extra_rows=3)
    inp = W.make_inputs(wl, "cuda")
    want, y, s, bad = oracle_expert_norm(inp)
    got, plan = run_expert_norm(inp, variant=mfr.VARIANT_STREAM)
    assert bad == 0
    assert_expert_norm_close(got, want, y, s)
    assert plan.get_status() == 0
    assert plan.info()["variant"] == mfr.VARIANT_STREAM
    again, _ = run_expert_norm(inp, plan=plan)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("T,H", [(1, 4096), (3, 8192), (16, 4096), (64, 8192)])
@pytest.mark.parametrize("cluster", [2, 4, 8, 16])
def test_expert_norm_every_cluster_size(T, H, cluster):
    """The cluster form at every cluster size, against the oracle."""
    wl = W.Workload(f"en_c{cluster}_T{T}_H{H}", T=T, H=H, k=8, E=32, seed=T + H + cluster, extra_rows=1)
    inp = W.make_inputs(wl, "cuda")
    want, y, s, _ = oracle_expert_norm(inp)
    got, plan = run_expert_norm(inp, variant=mfr.VARIANT_CLUSTER, cluster_size=cluster)
    assert plan.info()["cluster"] == cluster
    assert_expert_norm_close(got, want, y, s)
    assert plan.get_status() == 0


def test_expert_norm_forms_reported():
    """One CTA per token takes the one-pass form (rows held in registers) for
    k <= 8 and at most two chunks per thread, unless its registers add a wave
    of CTAs; else the two-pass form.  plan_info reports it as slot_registers."""
    assert mfr.ExpertNormPlan(1, 4096, 8, variant=mfr.VARIANT_ROWS).info()["slot_registers"] == 1
    assert mfr.ExpertNormPlan(1, 4096, 16, variant=mfr.VARIANT_ROWS).info()["slot_registers"] == 0
    assert mfr.ExpertNormPlan(1, 16384, 8, variant=mfr.VARIANT_ROWS).info()["slot_registers"] == 0
    assert mfr.ExpertNormPlan(1, 4096, 8).info()["slot_registers"] == 1      # the cluster form


def test_expert_norm_stress_values_and_repeats():
    """Student-t rows with 1 % outlier rows x100 and unnormalised weights:
    each row is normalised on its own, so outliers do not swamp the others."""
    inp = W.make_inputs(W.STRESS.with_(T=64, H=4096), "cuda")
    want, y, s, _ = oracle_expert_norm(inp)
    got, plan = run_expert_norm(inp)
    assert_expert_norm_close(got, want, y, s)
    again, _ = run_expert_norm(inp, plan=plan)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("variant", [mfr.VARIANT_ROWS, mfr.VARIANT_STREAM, mfr.VARIANT_CLUSTER],
                         ids=["rows", "ring", "cluster"])
def test_expert_norm_bad_and_sentinel_slots(variant):
    inp = W.make_inputs(W.decode(8), "cuda")
    idx = inp["permuted_row_of"].clone()
    idx[2, 5] = -1
    idx[6, 0] = 10 ** 6
    inp["permuted_row_of"] = idx
    want, y, s, bad = oracle_expert_norm(inp)
    assert bad == 2
    got, plan = run_expert_norm(inp, variant=variant)
    assert_expert_norm_close(got, want, y, s)
    assert plan.get_status() & mfr.STATUS_BAD_INDEX
    # with sentinel_skip a negative index is a skipped non-local slot, not an error;
    # the out-of-range positive one was replaced by a valid row
    idx[6, 0] = idx[6, 1]
    got, plan = run_expert_norm(inp, sentinel_skip=True, variant=variant)
    want, y, s, _ = oracle_expert_norm(inp)
    assert_expert_norm_close(got, want, y, s)
    assert plan.get_status() == 0


@pytest.mark.parametrize("wl", [W.PREFILL, W.wide(4096)], ids=["prefill", "wide_T4096"])
def test_expert_norm_full_size_every_token(wl):
    """Full-size workloads in the launch configuration the benchmark times
    (the ring form); every token against the oracle, run over the host
    cores."""
    inp = W.make_inputs(wl, "cuda")
    got, plan = run_expert_norm(inp)
    assert plan.info()["variant"] == mfr.VARIANT_STREAM
    assert plan.get_status() == 0
    h = host_inputs(inp)
    del inp
    torch.cuda.empty_cache()
    E_abs, w_abs, g_abs = h["E"] & np.uint16(0x7FFF), np.abs(h["w"]), h["gamma"] & np.uint16(0x7FFF)

    def check(tk):
        want, bad = oracle.finalize_expert_rmsnorm(h["E"], h["idx"], h["w"], h["gamma"], h["eps"], tokens=tk)
        assert bad == 0
        y, _ = oracle.expert_rmsnorm_f64(h["E"], h["idx"], h["w"], h["gamma"], h["eps"], tokens=tk)
        sc, _ = oracle.expert_rmsnorm_f64(E_abs, h["idx"], w_abs, g_abs, h["eps"], tokens=tk)
        assert_expert_norm_close(got[tk[0]:tk[-1] + 1], want, y, sc)
    assert over_all_tokens(wl.T, check) == wl.T


def test_expert_norm_refuses_other_variants_and_other_plans():
    with pytest.raises(mfr.MFRError):
        mfr.ExpertNormPlan(64, 4096, 16, variant=mfr.VARIANT_STREAM)    # more than 8 slots
    with pytest.raises(mfr.MFRError):
        mfr.ExpertNormPlan(64, 16384, 8, variant=mfr.VARIANT_STREAM)    # more than 4 column tiles
    with pytest.raises(mfr.MFRError):
        mfr.ExpertNormPlan(64, 4096, 16, variant=mfr.VARIANT_CLUSTER)   # more than 8 slots
    assert mfr.ExpertNormPlan(64, 4096, 8, variant=mfr.VARIANT_CLUSTER).info()["cluster"] > 1
    assert mfr.ExpertNormPlan(1, 4096, 8).info()["variant"] == mfr.VARIANT_CLUSTER
    assert mfr.ExpertNormPlan(1, 4096, 16).info()["variant"] == mfr.VARIANT_ROWS
    assert mfr.ExpertNormPlan(16384, 4096, 8).info()["variant"] == mfr.VARIANT_STREAM
    assert mfr.ExpertNormPlan(16384, 4096, 16).info()["variant"] == mfr.VARIANT_ROWS
    inp = W.make_inputs(W.decode(4), "cuda")
    out = torch.empty((4, 4096), dtype=torch.bfloat16, device="cuda")
    plain = mfr.FinalizePlan(4, 4096, 8)
    with pytest.raises(mfr.MFRError):
        code = plain._lib.moe_finalize_expert_rmsnorm_run(plain.handle, inp["expert_out"].data_ptr(),
                                                          inp["permuted_row_of"].data_ptr(),
                                                          inp["topk_weights"].data_ptr(), inp["gamma"].data_ptr(),
                                                          ctypes.c_float(1e-6), out.data_ptr(), None)
        mfr._check(code, "run")
    en = mfr.ExpertNormPlan(4, 4096, 8)
    with pytest.raises(mfr.MFRError):
        mfr._check(en._lib.moe_finalize_run(en.handle, inp["expert_out"].data_ptr(), inp["permuted_row_of"].data_ptr(),
                                            inp["topk_weights"].data_ptr(), out.data_ptr(), None), "run")
    en.launch_floor()
    torch.cuda.synchronize()
    assert en.get_status() == 0
