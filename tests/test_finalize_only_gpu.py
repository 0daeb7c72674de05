"""The plain finalize (out = bf16 of the FP32 weighted sum; no residual, no
norm) against the oracle's finalize: bf16 output within 1 ulp (in practice
equal: both round the same FP32 value once)."""
import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from helpers import (assert_out_close, bf16_bits, check_every_token_finalize_only, host_inputs,
                     oracle_finalize_only)

pytestmark = pytest.mark.gpu
GUARD = 256


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def run_finalize(inp, **plan_kw):
    e, idx, w = inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"]
    T, k = idx.shape
    R, H = e.shape
    plan = mfr.FinalizePlan(T, H, k, R, **plan_kw)
    buf = torch.full((T * H + 2 * GUARD,), -5.0, dtype=torch.bfloat16, device="cuda")
    out = buf[GUARD:GUARD + T * H].view(T, H)
    plan.run(e, idx, w, out)
    torch.cuda.synchronize()
    assert torch.all(buf[:GUARD] == -5.0) and torch.all(buf[-GUARD:] == -5.0)
    return bf16_bits(out), plan


VARIANTS = [dict(), dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_STREAM),
            dict(variant=mfr.VARIANT_CLUSTER, cluster_size=4)]


@pytest.mark.parametrize("kw", VARIANTS, ids=["auto", "rows", "stream", "split4"])
@pytest.mark.parametrize("T,H,k", [(1, 4096, 8), (16, 4096, 8), (5, 24, 3), (300, 8192, 8), (7, 4104, 16),
                                   (153, 1032, 1)])
def test_finalize_only_matches_oracle(kw, T, H, k):
    if kw.get("cluster_size") and (H // 8) % kw["cluster_size"]:
        pytest.skip("column split must divide H/8")
    wl = W.Workload(f"fin_T{T}_H{H}", T=T, H=H, k=k, E=max(16, 2 * k), seed=T * 7 + H + k, extra_rows=2)
    inp = W.make_inputs(wl, "cuda")
    want, bad = oracle_finalize_only(inp)
    got, plan = run_finalize(inp, **kw)
    assert bad == 0
    assert_out_close(got, want)
    assert np.array_equal(got, want)       # same FP32 value rounded once on both sides
    assert plan.get_status() == 0


@pytest.mark.parametrize("T,H,k", [(2000, 4096, 2), (1500, 8192, 4), (1800, 4096, 16), (2000, 4096, 8),
                                   (512, 8192, 8), (2048, 8192, 8), (300, 24, 8), (400, 136, 8), (300, 2056, 8)])
def test_finalize_only_ring_wraps(T, H, k):
    """The ring form with ring depths from 3 stages (k = 16) to 8 (k = 2) and
    many tokens per CTA, with k = 8 in both the all-slots instantiation
    (H <= 4096, ragged widths included; H = 8192 up to 2^22 elements) and
    the general one: every token bitwise equal to the oracle."""
    wl = W.Workload(f"fin_ring_T{T}_H{H}_k{k}", T=T, H=H, k=k, E=max(16, 2 * k), seed=T + H + k, extra_rows=2)
    inp = W.make_inputs(wl, "cuda")
    want, bad = oracle_finalize_only(inp)
    got, plan = run_finalize(inp, variant=mfr.VARIANT_STREAM)
    assert bad == 0
    assert np.array_equal(got, want)
    assert plan.get_status() == 0
    assert plan.info()["variant"] == mfr.VARIANT_STREAM


@pytest.mark.parametrize("T,H", [(1500, 4096), (400, 8192)])
def test_finalize_only_ring_bad_slot_in_the_all_slots_form(T, H):
    """k = 8 in the ring's all-slots instantiation: a token with an
    out-of-range slot takes the general slot loop, adds nothing for that
    slot and raises the status bit; every token bitwise equal to the oracle."""
    wl = W.Workload(f"fin_bad_T{T}_H{H}", T=T, H=H, k=8, E=16, seed=T + H, extra_rows=2)
    inp = W.make_inputs(wl, "cuda")
    inp["permuted_row_of"][T // 3, 3] = wl.R          # == R: invalid
    want, bad = oracle_finalize_only(inp)
    assert bad == 1
    got, plan = run_finalize(inp, variant=mfr.VARIANT_STREAM)
    assert np.array_equal(got, want)
    assert plan.get_status() & mfr.STATUS_BAD_INDEX


@pytest.mark.parametrize("T,H", [(1, 4096), (4, 4096), (2, 8192), (33, 8192)])
@pytest.mark.parametrize("split", [2, 4, 8, 16])
def test_finalize_only_every_split(T, H, split):
    """Every number of CTAs per token, against the oracle, bitwise."""
    wl = W.Workload(f"fin_s{split}_T{T}_H{H}", T=T, H=H, k=8, E=32, seed=T + H + split, extra_rows=1)
    inp = W.make_inputs(wl, "cuda")
    want, _ = oracle_finalize_only(inp)
    got, plan = run_finalize(inp, variant=mfr.VARIANT_CLUSTER, cluster_size=split)
    assert plan.info()["cluster"] == split
    assert np.array_equal(got, want)
    assert plan.get_status() == 0


def test_finalize_only_bad_indices():
    inp = W.make_inputs(W.decode(8), "cuda")
    inp["permuted_row_of"][2, 5] = -1
    inp["permuted_row_of"][6, 0] = 10**6
    for kw in VARIANTS:
        want, bad = oracle_finalize_only(inp)
        got, plan = run_finalize(inp, **kw)
        assert bad == 2
        assert np.array_equal(got, want)
        assert plan.get_status() & mfr.STATUS_BAD_INDEX


def test_plan_kinds_do_not_mix():
    inp = W.make_inputs(W.decode(2), "cuda")
    fin = mfr.FinalizePlan(2, 4096, 8)
    fused = mfr.Plan(2, 4096, 8)
    out = torch.empty((2, 4096), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(inp["residual"])
    with pytest.raises(mfr.MFRError):          # residual + norm run on a finalize plan
        mfr.Plan.run(fin, inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout,
                     inp["gamma"], 1e-6, out)
    with pytest.raises(mfr.MFRError):
        mfr.FinalizePlan.run(fused, inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], out)


@pytest.mark.parametrize("wl", [W.PREFILL, W.STRESS], ids=lambda w: w.name)
def test_finalize_only_full_size_every_token(wl):
    inp = W.make_inputs(wl, "cuda")
    T = wl.T
    plan = mfr.FinalizePlan(T, wl.H, wl.k, wl.R)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    plan.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], out)
    torch.cuda.synchronize()
    assert plan.get_status() == 0
    h = host_inputs(inp)
    got = bf16_bits(out)
    del inp, out
    torch.cuda.empty_cache()
    assert check_every_token_finalize_only(h, got) == T
