"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every case compares every element, the full-size workloads too (in the
launch configuration the benchmark times, with the oracle spread over the
host cores).  Bars:
residual_out within max(1e-6 * |oracle|, 1e-6) per element (in practice
bit-equal: both sides do the same FP32 operations), out within 1 bf16 ulp,
and repeated runs bitwise identical.  Every output buffer sits between guard
regions that must come back untouched.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from helpers import (assert_out_close, assert_residual_close, bf16_bits, check_every_token, f32, host_inputs,
                     oracle_on)

pytestmark = pytest.mark.gpu

GUARD = 256  # elements of guard on each side of every output


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def guarded(shape, dtype, fill):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(*shape)


def check_guards(buf, fill):
    head, tail = buf[:GUARD], buf[-GUARD:]
    assert torch.equal(head, torch.full_like(head, fill)) and torch.equal(tail, torch.full_like(tail, fill)), \
        "a kernel wrote outside its output"


def run_gpu(inp, plan_kw=None, in_place=False, residual=None, plan=None):
    """Runs one call through the binding (C ABI) with guarded outputs.
    Returns host copies (residual_out f32, out bf16 bits) and the plan."""
    e, idx, w, g = inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["gamma"]
    res = inp["residual"] if residual is None else residual
    T, k = idx.shape
    R, H = e.shape
    if plan is None:
        plan = mfr.Plan(T, H, k, R, **(plan_kw or {}))
    ob, out = guarded((T, H), torch.bfloat16, -7.0)
    if in_place:
        rb, rout = guarded((T, H), torch.float32, -3.0)
        rout.copy_(res)
        rin = rout
    else:
        rb, rout = guarded((T, H), torch.float32, -3.0)
        rin = res
    plan.run(e, idx, w, rin, rout, g, inp["eps"], out)
    torch.cuda.synchronize()
    check_guards(ob, -7.0)
    check_guards(rb, -3.0)
    return f32(rout), bf16_bits(out), plan


def compare_full(inp, plan_kw=None, in_place=False, plan=None):
    want_res, want_out, bad = oracle_on(inp)
    got_res, got_out, plan = run_gpu(inp, plan_kw, in_place, plan=plan)
    assert_residual_close(got_res, want_res)
    assert_out_close(got_out, want_out)
    status = plan.get_status()
    assert bool(status & mfr.STATUS_BAD_INDEX) == (bad > 0)
    return got_res, want_res, got_out, want_out, plan


def inputs_for(T, H, k, R=None, seed=0, E=None, **kw):
    wl = W.Workload(f"case_T{T}_H{H}_k{k}", T=T, H=H, k=k, E=E or max(2 * k, 16), seed=seed,
                    extra_rows=0 if R is None else R - T * k, **kw)
    return W.make_inputs(wl, "cuda")


# --- small cases, every element -----------------------------------------------

def test_tiny_ref_auto_plan_is_bit_exact_on_the_residual():
    inp = W.make_inputs(W.TINY_REF, "cuda")
    got_res, want_res, got_out, want_out, plan = compare_full(inp)
    assert np.array_equal(got_res.view(np.uint32), want_res.view(np.uint32))
    # at most a small share of outputs sit one ulp away (rounding near ties)
    assert np.mean(got_out != want_out) < 0.02


@pytest.mark.parametrize("variant,cluster", [(mfr.VARIANT_ROWS, 0), (mfr.VARIANT_STREAM, 0),
                                             (mfr.VARIANT_CLUSTER, 2),
                                             (mfr.VARIANT_CLUSTER, 4), (mfr.VARIANT_CLUSTER, 8),
                                             (mfr.VARIANT_CLUSTER, 16)])
@pytest.mark.parametrize("pdl", [True, False])
def test_tiny_ref_every_variant(variant, cluster, pdl):
    inp = W.make_inputs(W.TINY_REF, "cuda")
    _, _, _, _, plan = compare_full(inp, dict(variant=variant, cluster_size=cluster, enable_pdl=pdl))
    info = plan.info()
    assert info["variant"] == variant
    if variant == mfr.VARIANT_CLUSTER:
        assert info["cluster"] == cluster


@pytest.mark.parametrize("T", W.DECODE_TOKENS + (3, 5, 7, 100))
def test_decode_sweep_auto_plan(T):
    compare_full(W.make_inputs(W.decode(T), "cuda", T=T))


@pytest.mark.parametrize("H", [8, 24, 136, 1024, 4104, 8192, 12288, 16384])
@pytest.mark.parametrize("k", [1, 5, 8, 16])
def test_shapes_with_ragged_tails(H, k):
    T = 5
    inp = inputs_for(T, H, k, R=T * k + 3, seed=H + k)
    compare_full(inp)
    compare_full(inp, dict(variant=mfr.VARIANT_ROWS))
    compare_full(inp, dict(variant=mfr.VARIANT_STREAM))
    if H % 64 == 0 and H >= 1024:
        compare_full(inp, dict(variant=mfr.VARIANT_CLUSTER, cluster_size=8))


def test_in_place_residual():
    inp = W.make_inputs(W.decode(16), "cuda")
    for kw in (dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_CLUSTER, cluster_size=4),
               dict(variant=mfr.VARIANT_STREAM)):
        compare_full(inp, kw, in_place=True)


def test_out_of_range_indices_add_nothing_and_raise_the_status_bit():
    inp = inputs_for(6, 1024, 8, seed=3)
    idx = inp["permuted_row_of"].clone()
    R = inp["expert_out"].shape[0]
    idx[0, 0] = -1
    idx[2, 7] = R
    idx[5, 3] = 2**31 - 1
    idx[4, 4] = -(2**31)
    inp["permuted_row_of"] = idx
    for kw in (dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_CLUSTER, cluster_size=2),
               dict(variant=mfr.VARIANT_STREAM)):
        compare_full(inp, kw)


@pytest.mark.parametrize("T", [129, 151, 152, 153, 304, 1000, 2049])
@pytest.mark.parametrize("H", [4096, 8192, 1032])
def test_stream_token_counts_around_the_sm_count(T, H):
    """The persistent kernel's static token schedule: fewer, equal and more
    tokens than CTAs, ragged last round, ragged last column tile."""
    inp = inputs_for(T, H, 8, seed=T + H)
    _, _, _, _, plan = compare_full(inp, dict(variant=mfr.VARIANT_STREAM))
    info = plan.info()
    assert info["variant"] == mfr.VARIANT_STREAM
    # the fewest rounds of one token per CTA, spread evenly: CTA loads differ by at most one
    sms = info["sm_count"]
    rounds = -(-T // sms)
    assert info["grid_x"] == (T if T <= sms else -(-T // rounds))
    assert -(-T // info["grid_x"]) == rounds


@pytest.mark.parametrize("k,H", [(1, 4096), (2, 4096), (4, 4096), (16, 4096), (4, 8192), (3, 1032),
                                 (8, 16384), (2, 12288), (8, 4096), (8, 8192)])
def test_stream_ring_wraps_at_every_depth(k, H):
    """Many tokens per CTA (T = 2000, or 700 at H > 8192, over at most 152
    CTAs) with every ring depth the plan gives, from 3 stages (k = 16) to 8
    (k <= 2): the ring wraps many times and the stage barriers' phases
    alternate (at H = 12288 and 16384 a token spans 6 and 8 tiles); every
    token against the oracle, an out-of-range row included (with k = 8 at
    H <= 8192 it sends that token's tiles through the general slot loop of
    the all-slots instantiation)."""
    T = 2000 if H <= 8192 else 700
    inp = inputs_for(T, H, k, R=T * k + 5, seed=31 + k + H)
    inp["permuted_row_of"][T // 2, k - 1] = T * k + 5          # == R: invalid
    _, _, _, _, plan = compare_full(inp, dict(variant=mfr.VARIANT_STREAM))
    info = plan.info()
    assert info["variant"] == mfr.VARIANT_STREAM
    stage = 128 + k * 2048 * 2 + 2048 * 4                       # header, k row segments, residual
    assert 2 * stage < info["smem_bytes"] <= 8 * stage + 128


@pytest.mark.parametrize("T", [100, 152, 153, 200, 400])
def test_rows_kernel_both_slot_forms(T):
    """The one-CTA-per-token kernel keeps the slot rows and weights in
    registers across the dependency wait unless that costs a wave of CTAs
    (512-thread CTAs at H=4096 fit twice per SM without them, once with
    them); both forms match the oracle, an invalid slot included."""
    inp = inputs_for(T, 4096, 8, seed=T)
    idx = inp["permuted_row_of"].clone()
    idx[T // 2, 3] = -1
    inp["permuted_row_of"] = idx
    _, _, _, _, plan = compare_full(inp, dict(variant=mfr.VARIANT_ROWS))
    info = plan.info()
    assert info["block"] == 512
    assert info["slot_registers"] == (1 if T <= info["sm_count"] else 0)
    assert mfr.Plan(8, 4096, 8, 64).info()["slot_registers"] == 1   # decode cluster


@pytest.mark.parametrize("T,H,variant,cluster", [
    (1, 4096, mfr.VARIANT_CLUSTER, 4), (4, 4096, mfr.VARIANT_CLUSTER, 4), (8, 4096, mfr.VARIANT_CLUSTER, 16),
    (32, 4096, mfr.VARIANT_CLUSTER, 16), (64, 4096, mfr.VARIANT_CLUSTER, 8), (128, 4096, mfr.VARIANT_CLUSTER, 2),
    (129, 4096, mfr.VARIANT_ROWS, 1), (304, 4096, mfr.VARIANT_ROWS, 1), (305, 4096, mfr.VARIANT_STREAM, 1),
    (1, 8192, mfr.VARIANT_CLUSTER, 8), (8, 8192, mfr.VARIANT_CLUSTER, 16), (64, 8192, mfr.VARIANT_CLUSTER, 4),
    (65, 8192, mfr.VARIANT_ROWS, 1), (152, 8192, mfr.VARIANT_ROWS, 1), (153, 8192, mfr.VARIANT_STREAM, 1),
    (2, 1024, mfr.VARIANT_ROWS, 1)])
def test_automatic_plan_choices(T, H, variant, cluster):
    """The variant and cluster size the plan picks by T*H (measured
    thresholds: clusters up to 2^19 elements, one CTA per token up to one
    wave (8192 elements per SM), the ring from there)."""
    info = mfr.Plan(T, H, 8).info()
    assert (info["variant"], info["cluster"]) == (variant, cluster)


def test_variants_agree_bitwise_on_the_residual():
    inp = W.make_inputs(W.PREFILL, "cuda", T=300)
    results = [run_gpu(inp, dict(variant=v, cluster_size=c))
               for v, c in ((mfr.VARIANT_ROWS, 0), (mfr.VARIANT_STREAM, 0), (mfr.VARIANT_CLUSTER, 4))]
    for r in results[1:]:
        assert np.array_equal(r[0].view(np.uint32), results[0][0].view(np.uint32))
        assert_out_close(r[1], results[0][1])


def test_plans_with_different_rings_coexist():
    """A k=16 plan (3 stages) keeps working after a k=8 plan (5 stages) of the
    same kernel was made: the shared-memory attribute is per kernel."""
    a_inp = inputs_for(300, 4096, 16, seed=11)
    b_inp = inputs_for(300, 4096, 8, seed=12)
    a_plan = mfr.Plan(300, 4096, 16, 300 * 16, variant=mfr.VARIANT_STREAM)
    b_plan = mfr.Plan(300, 4096, 8, 300 * 8, variant=mfr.VARIANT_STREAM)
    assert a_plan.info()["smem_bytes"] > b_plan.info()["smem_bytes"]
    compare_full(a_inp, plan=a_plan)
    compare_full(b_inp, plan=b_plan)
    compare_full(a_inp, plan=a_plan)


def test_launch_floor_runs_with_every_geometry():
    for kw in (dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_STREAM),
               dict(variant=mfr.VARIANT_CLUSTER, cluster_size=16)):
        plan = mfr.Plan(64, 4096, 8, 512, **kw)
        plan.launch_floor()
        torch.cuda.synchronize()
        assert plan.get_status() == 0


def test_debug_checks_turn_a_bad_index_into_an_error():
    inp = inputs_for(2, 512, 8, seed=4)
    inp["permuted_row_of"][1, 1] = -5
    with pytest.raises(mfr.MFRError) as ei:
        run_gpu(inp, dict(debug_checks=True))
    assert ei.value.code == 7


def test_duplicate_rows_and_special_weights():
    inp = inputs_for(4, 2048, 8, seed=5)
    idx = inp["permuted_row_of"].clone()
    idx[0, :] = idx[0, 0]                 # one row eight times
    idx[1, 1::2] = idx[1, 0::2]
    w = inp["topk_weights"].clone()
    w[2] = torch.tensor([0.0, -0.0, -1.5, 2.0**-30, 3.0e5, -1e-20, 0.25, 1.0])
    w[3] = -w[3]
    inp["permuted_row_of"], inp["topk_weights"] = idx, w
    compare_full(inp)


def test_nan_inf_and_zero_rows_propagate_like_ieee():
    inp = inputs_for(5, 1024, 4, seed=6)
    e = inp["expert_out"]
    idx = inp["permuted_row_of"]
    e[idx[0, 1]] = float("nan")
    e[idx[1, 2], 17] = float("inf")
    # token 2: every contribution cancels the residual exactly -> all-zero x
    inp["topk_weights"][2] = torch.tensor([1.0, 0.0, 0.0, 0.0])
    inp["residual"][2] = -e[idx[2, 0]].float()
    inp["eps"] = 0.0
    got_res, want_res, got_out, want_out, _ = compare_full(inp)
    assert np.isnan(got_res[0]).all()
    assert np.all(got_res[2] == 0)


def test_large_magnitudes_and_tiny_eps():
    inp = W.make_inputs(W.STRESS, "cuda", T=24)
    compare_full(inp)
    inp["eps"] = 1e-12
    compare_full(inp)


def test_zero_tokens_is_a_no_op():
    plan = mfr.Plan(0, 4096, 8, 0)
    z = torch.empty(0, device="cuda")
    code = plan.run_ptrs(0, 0, 0, 0, 0, 0, 1e-6, 0, 0)
    assert code == 0
    del z


@pytest.mark.parametrize("variant", [mfr.VARIANT_ROWS, mfr.VARIANT_STREAM])
def test_repeated_runs_are_bitwise_identical(variant):
    inp = W.make_inputs(W.PREFILL, "cuda", T=1000)
    a = run_gpu(inp, dict(variant=variant))
    b = run_gpu(inp, dict(variant=variant))
    assert np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))
    assert np.array_equal(a[1], b[1])


# --- argument checks on a real device --------------------------------------------

def test_run_rejects_bad_arguments_without_launching():
    inp = inputs_for(4, 1024, 8, seed=7)
    T, H, k, R = 4, 1024, 8, 32
    plan = mfr.Plan(T, H, k, R)
    e, idx, w, res, g = (inp[n] for n in ("expert_out", "permuted_row_of", "topk_weights", "residual", "gamma"))
    rout = torch.empty_like(res)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream
    ok = (p(e), p(idx), p(w), p(res), p(rout), p(g), 1e-6, p(out), s)
    assert plan.run_ptrs(*ok) == 0
    bad = list(ok); bad[0] = p(e) + 2                                  # misaligned expert_out
    assert plan.run_ptrs(*bad) == 3
    bad = list(ok); bad[7] = p(out) + 8                                # misaligned out
    assert plan.run_ptrs(*bad) == 3
    bad = list(ok); bad[1] = p(idx) + 2                                # misaligned index map
    assert plan.run_ptrs(*bad) == 3
    for eps in (-1.0, float("nan"), float("inf")):
        bad = list(ok); bad[6] = eps
        assert plan.run_ptrs(*bad) == 1
    bad = list(ok); bad[7] = p(res)                                    # out aliases residual_in
    assert plan.run_ptrs(*bad) == 1
    bad = list(ok); bad[4] = p(res) + 16                               # partial residual overlap
    assert plan.run_ptrs(*bad) == 1
    bad = list(ok); bad[2] = 0                                         # null weights
    assert plan.run_ptrs(*bad) == 1
    torch.cuda.synchronize()
    assert plan.get_status() == 0


# --- full sizes, in the benchmark's launch configuration -----------------------------

FULL = [W.PREFILL, W.wide(4096), W.wide(8192), W.STRESS]


@pytest.mark.parametrize("wl", FULL, ids=lambda w: w.name)
def test_full_size_every_token(wl):
    """Every token of the full-size call against the oracle (run on all host
    cores), in the plan the benchmark times; the stress call is run twice
    more and must repeat bit for bit."""
    inp = W.make_inputs(wl, "cuda")
    T = wl.T
    plan = mfr.Plan(T, wl.H, wl.k, wl.R)          # the benchmark's plan: auto variant, PDL on
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    rout = torch.empty_like(inp["residual"])
    plan.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout,
             inp["gamma"], inp["eps"], out)
    torch.cuda.synchronize()
    assert plan.get_status() == 0
    if wl is W.STRESS:
        # run twice more; every byte of both outputs must repeat
        out2, rout2 = torch.empty_like(out), torch.empty_like(rout)
        for _ in range(2):
            plan.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout2,
                     inp["gamma"], inp["eps"], out2)
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
            assert torch.equal(rout.view(torch.int32), rout2.view(torch.int32))
        del out2, rout2
    h = host_inputs(inp)
    got_res, got_out = f32(rout), bf16_bits(out)
    del inp, out, rout
    torch.cuda.empty_cache()
    assert check_every_token(h, got_res, got_out) == T


@pytest.mark.parametrize("kw", [dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_STREAM),
                                dict(variant=mfr.VARIANT_CLUSTER, cluster_size=8)],
                         ids=["rows", "stream", "cluster8"])
def test_sentinel_skip_for_non_local_experts(kw):
    """With sentinel_skip, a negative index is a non-local slot: it adds
    nothing (as every invalid slot does) and raises no status bit; an index
    >= R still does."""
    inp = inputs_for(6, 2048, 8, seed=21)
    idx = inp["permuted_row_of"].clone()
    R = inp["expert_out"].shape[0]
    idx[0, 3] = -1
    idx[4, 0] = -7
    inp["permuted_row_of"] = idx
    want_res, want_out, bad = oracle_on(inp)
    assert bad == 2
    got_res, got_out, plan = run_gpu(inp, dict(kw, sentinel_skip=True))
    assert_residual_close(got_res, want_res)
    assert_out_close(got_out, want_out)
    assert plan.get_status() == 0                        # negative entries are not errors
    _, _, plan = run_gpu(inp, dict(kw, sentinel_skip=False))
    assert plan.get_status() & mfr.STATUS_BAD_INDEX      # without the option they are
    idx[2, 2] = R                                         # out of range at the top: always an error
    got_res, got_out, plan = run_gpu(inp, dict(kw, sentinel_skip=True))
    assert plan.get_status() & mfr.STATUS_BAD_INDEX


def test_functional_wrapper_caches_plans():
    """The allocating wrapper reuses one plan per shape and options and keeps
    at most PLAN_CACHE_SIZE of them."""
    inp = W.make_inputs(W.decode(2), "cuda")
    want_res, want_out, _ = oracle_on(inp)
    args = (inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], inp["gamma"],
            inp["eps"])
    mfr._plan_cache.clear()
    for _ in range(3):
        res, out = mfr.moe_finalize_residual_rmsnorm(*args)
        torch.cuda.synchronize()
        assert_residual_close(f32(res), want_res)
        assert_out_close(bf16_bits(out), want_out)
    assert len(mfr._plan_cache) == 1
    mfr.moe_finalize_residual_rmsnorm(*args, variant=mfr.VARIANT_ROWS)
    assert len(mfr._plan_cache) == 2
    old = mfr.PLAN_CACHE_SIZE
    try:
        mfr.PLAN_CACHE_SIZE = 2
        for T in (1, 3, 5):
            x = W.make_inputs(W.decode(T), "cuda")
            mfr.moe_finalize_residual_rmsnorm(x["expert_out"], x["permuted_row_of"], x["topk_weights"],
                                              x["residual"], x["gamma"], x["eps"])
        torch.cuda.synchronize()
        assert len(mfr._plan_cache) == 2
    finally:
        mfr.PLAN_CACHE_SIZE = old
        mfr._plan_cache.clear()


@pytest.mark.parametrize("kw", [dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_STREAM),
                                dict(variant=mfr.VARIANT_CLUSTER, cluster_size=4)],
                         ids=["rows", "stream", "cluster4"])
def test_every_slot_non_local(kw):
    """A batch whose experts all live on other GPUs: R = 0 and every index -1
    with sentinel_skip.  No row is read, the residual passes through
    unchanged, out is the RMSNorm of the residual alone, the plain finalize
    and the per-expert form write zeros, and no status bit is raised."""
    T, H, k = 6, 4096, 8
    inp = W.make_inputs(W.decode(T), "cuda")
    inp["expert_out"] = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    inp["permuted_row_of"] = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    plan = mfr.Plan(T, H, k, 0, sentinel_skip=True, **kw)
    got_res, got_out, _ = run_gpu(inp, plan=plan)
    assert np.array_equal(got_res.view(np.uint32), f32(inp["residual"]).view(np.uint32))
    want_res, want_out, _ = oracle_on(inp)
    assert_out_close(got_out, want_out)
    assert plan.get_status() == 0
    for make in (mfr.FinalizePlan, mfr.ExpertNormPlan):
        p = make(T, H, k, 0, sentinel_skip=True, **kw)
        out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
        if make is mfr.FinalizePlan:
            p.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], out)
        else:
            p.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["gamma"], inp["eps"], out)
        torch.cuda.synchronize()
        assert torch.all(out.float() == 0)
        assert p.get_status() == 0


@pytest.mark.parametrize("kw", [dict(), dict(variant=mfr.VARIANT_ROWS), dict(variant=mfr.VARIANT_STREAM)],
                         ids=["auto_cluster", "rows", "stream"])
def test_one_plan_on_four_streams_at_once(kw):
    """A plan is immutable: one plan runs on four streams at the same time,
    each call on its own inputs, and every call matches the oracle."""
    T = 64 if not kw else 300
    calls = [W.make_inputs(W.PREFILL.with_(T=T, seed=40 + i), "cuda") for i in range(4)]
    plan = mfr.Plan(T, 4096, 8, T * 8, **kw)
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = []
    torch.cuda.synchronize()
    for inp, s in zip(calls, streams):
        rout = torch.empty_like(inp["residual"])
        out = torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):        # a few calls per stream, all in flight together
            plan.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout,
                     inp["gamma"], inp["eps"], out, s)
        outs.append((rout, out))
    torch.cuda.synchronize()
    for inp, (rout, out) in zip(calls, outs):
        want_res, want_out, _ = oracle_on(inp)
        assert_residual_close(f32(rout), want_res)
        assert_out_close(bf16_bits(out), want_out)
    assert plan.get_status() == 0
