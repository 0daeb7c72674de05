"""The allocation-free entry point (moe_finalize_rmsnorm_run_noalloc).

It serves callers that cannot allocate device memory (an engine that owns
all device memory through its own pool, a host that may not call cudaMalloc
on the request path): no plan, no allocation, the status word in the
library's static device scratch.  Its outputs must match the oracle within
the parity tolerances on two calls in a row, and equal those of the planned
entry point (moe_finalize_rmsnorm_plan + _run).

This file is collected last on purpose, and also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from helpers import assert_out_close, assert_residual_close, bf16_bits, f32, oracle_on

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    return mfr.load_library()


def _call_noalloc(lib, inp, rout, out, slot, status):
    e, idx, w, g, res = (inp[n] for n in ("expert_out", "permuted_row_of", "topk_weights", "gamma", "residual"))
    T, k = idx.shape
    R, H = e.shape
    return lib.moe_finalize_rmsnorm_run_noalloc(
        T, H, k, R, e.data_ptr(), idx.data_ptr(), w.data_ptr(), res.data_ptr(), rout.data_ptr(),
        g.data_ptr(), ctypes.c_float(inp["eps"]), out.data_ptr(), slot,
        ctypes.byref(status) if status is not None else None, torch.cuda.current_stream().cuda_stream)


def _planned(inp):
    T, k = inp["permuted_row_of"].shape
    R, H = inp["expert_out"].shape
    plan = mfr.Plan(T, H, k, R)
    rout = torch.empty_like(inp["residual"])
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    plan.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout,
             inp["gamma"], inp["eps"], out)
    torch.cuda.synchronize()
    return f32(rout), bf16_bits(out)


@pytest.mark.parametrize("wl", [W.TINY_REF, W.PREFILL.with_(T=1000), W.wide(64), W.STRESS.with_(T=300),
                                W.Workload("k2", T=2000, H=4096, k=2, E=16)],   # 8-stage ring, many wraps
                         ids=lambda w: f"{w.name}_T{w.T}")
def test_noalloc_matches_the_oracle_twice(lib, wl):
    inp = W.make_inputs(wl, "cuda")
    want_res, want_out, bad = oracle_on(inp)
    assert bad == 0
    plan_res, plan_out = _planned(inp)
    for call in range(2):
        rout = torch.full_like(inp["residual"], float("nan"))
        out = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = ctypes.c_int(-1)
        assert _call_noalloc(lib, inp, rout, out, slot=call, status=st) == 0
        assert st.value == 0
        torch.cuda.synchronize()
        assert_residual_close(f32(rout), want_res)
        assert_out_close(bf16_bits(out), want_out)
        # and the planned entry point's outputs, within the same tolerances
        assert_residual_close(f32(rout), plan_res)
        assert_out_close(bf16_bits(out), plan_out)


def test_noalloc_reports_bad_indices_and_clears_its_word(lib):
    inp = W.make_inputs(W.decode(8), "cuda")
    T, H = 8, 4096
    rout = torch.empty_like(inp["residual"])
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    bad = dict(inp)
    bad["permuted_row_of"] = inp["permuted_row_of"].clone()
    bad["permuted_row_of"][3, 2] = -1
    st = ctypes.c_int(0)
    assert _call_noalloc(lib, bad, rout, out, slot=5, status=st) == 0
    assert st.value & mfr.STATUS_BAD_INDEX
    # the read-back cleared the word: the next call on the same slot starts from zero
    assert _call_noalloc(lib, inp, rout, out, slot=5, status=st) == 0
    assert st.value == 0
    # a call without read-back leaves its bits for the next call that reads back
    assert _call_noalloc(lib, bad, rout, out, slot=6, status=None) == 0
    assert _call_noalloc(lib, inp, rout, out, slot=6, status=st) == 0
    assert st.value & mfr.STATUS_BAD_INDEX
    assert _call_noalloc(lib, inp, rout, out, slot=6, status=st) == 0
    assert st.value == 0


def test_noalloc_rejects_a_slot_beyond_the_scratch(lib):
    inp = W.make_inputs(W.decode(2), "cuda")
    rout = torch.empty_like(inp["residual"])
    out = torch.empty((2, 4096), dtype=torch.bfloat16, device="cuda")
    for slot in (-1, mfr.NOALLOC_SLOTS, 1 << 20):
        assert _call_noalloc(lib, inp, rout, out, slot=slot, status=None) == 1
        assert "beyond" in lib.moe_finalize_rmsnorm_last_error().decode()
    torch.cuda.synchronize()


def test_noalloc_allocates_nothing_through_torch(lib):
    """Asynchronous calls (no status read-back) leave torch's allocator
    untouched; the binding's helper works too."""
    inp = W.make_inputs(W.PREFILL.with_(T=500), "cuda")
    rout = torch.empty_like(inp["residual"])
    out = torch.empty((500, 4096), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats()["allocation.all.allocated"]
    for slot in (0, 1):
        mfr.run_noalloc(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout,
                        inp["gamma"], inp["eps"], out, slot=slot)
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == before
    want_res, want_out, _ = oracle_on(inp)
    assert_residual_close(f32(rout), want_res)
    assert_out_close(bf16_bits(out), want_out)


def test_noalloc_binding_rejects_wrong_tensors_before_the_call(lib):
    """The C call cannot check buffer sizes; the binding refuses a wrongly
    sized, typed or strided tensor before anything is launched."""
    inp = W.make_inputs(W.decode(4), "cuda")
    args = dict(expert_out=inp["expert_out"], permuted_row_of=inp["permuted_row_of"],
                topk_weights=inp["topk_weights"], residual_in=inp["residual"],
                residual_out=torch.empty_like(inp["residual"]), gamma=inp["gamma"], eps=inp["eps"],
                out=torch.empty((4, 4096), dtype=torch.bfloat16, device="cuda"))
    for name, bad in [("residual_out", torch.empty((3, 4096), dtype=torch.float32, device="cuda")),
                      ("out", torch.empty((4, 4096), dtype=torch.float32, device="cuda")),
                      ("residual_out", torch.empty((4096, 4), dtype=torch.float32, device="cuda").t()),
                      ("gamma", inp["gamma"].cpu())]:
        with pytest.raises(ValueError):
            mfr.run_noalloc(**{**args, name: bad})
    torch.cuda.synchronize()


def test_noalloc_ring_fits_after_a_plan_set_the_kernel_attribute(lib):
    """Plans and the allocation-free call set the same per-kernel shared-memory
    attribute; with k=5 the deepest ring the budget allows is 8 stages, which
    must still launch after a plan has set the attribute."""
    wl = W.PREFILL.with_(T=400, k=5)
    inp = W.make_inputs(wl, "cuda")
    _planned(inp)                            # makes a plan: sets the attribute
    want_res, want_out, _ = oracle_on(inp)
    rout = torch.empty_like(inp["residual"])
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    st = ctypes.c_int(-1)
    assert _call_noalloc(lib, inp, rout, out, slot=7, status=st) == 0, lib.moe_finalize_rmsnorm_last_error()
    assert st.value == 0
    torch.cuda.synchronize()
    assert_residual_close(f32(rout), want_res)
    assert_out_close(bf16_bits(out), want_out)
