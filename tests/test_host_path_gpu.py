"""The end-to-end entry point on host buffers (moe_finalize_rmsnorm_run_host)
gives exactly the device entry point's results, also when calls on two
streams overlap."""
import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from helpers import assert_out_close, assert_residual_close, bf16_bits, f32, oracle_on

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def _host(inp):
    h = {key: inp[key].cpu().pin_memory() for key in ("expert_out", "permuted_row_of", "topk_weights", "residual", "gamma")}
    h["eps"] = inp["eps"]
    return h


@pytest.mark.parametrize("wl", [W.decode(8), W.TINY_REF, W.PREFILL.with_(T=1500)], ids=lambda w: f"{w.name}_T{w.T}")
def test_run_host_matches_the_oracle(wl):
    inp = W.make_inputs(wl, "cuda")
    want_res, want_out, _ = oracle_on(inp)
    plan = mfr.Plan(wl.T, wl.H, wl.k, wl.R)
    ws = torch.empty(plan.host_workspace_bytes(), dtype=torch.uint8, device="cuda")
    h = _host(inp)
    ho = {"residual_out": torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory(),
          "out": torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()}
    s = torch.cuda.Stream()
    mfr.finalize_residual_rmsnorm_host(plan, h, ho, ws, s)
    s.synchronize()
    assert_residual_close(ho["residual_out"].numpy(), want_res)
    assert_out_close(ho["out"].view(torch.int16).numpy().view(np.uint16), want_out)


def test_overlapping_calls_on_two_streams():
    wl = W.PREFILL.with_(T=2000)
    inps = [W.make_inputs(wl.with_(seed=s), "cuda") for s in (0, 1)]
    wants = [oracle_on(i)[:2] for i in inps]
    plan = mfr.Plan(wl.T, wl.H, wl.k, wl.R)
    hs = [_host(i) for i in inps]
    hos = [{"residual_out": torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory(),
            "out": torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()} for _ in range(2)]
    wss = [torch.empty(plan.host_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    ss = [torch.cuda.Stream() for _ in range(2)]
    for rep in range(3):
        for i in range(2):
            mfr.finalize_residual_rmsnorm_host(plan, hs[i], hos[i], wss[i], ss[i])
    torch.cuda.synchronize()
    for i in range(2):
        assert_residual_close(hos[i]["residual_out"].numpy(), wants[i][0])
        assert_out_close(hos[i]["out"].view(torch.int16).numpy().view(np.uint16), wants[i][1])


def test_run_host_rejects_a_small_workspace():
    wl = W.decode(4)
    inp = W.make_inputs(wl, "cuda")
    plan = mfr.Plan(wl.T, wl.H, wl.k, wl.R)
    need = plan.host_workspace_bytes()
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    h = _host(inp)
    ho = {"residual_out": torch.empty((4, 4096), dtype=torch.float32), "out": torch.empty((4, 4096), dtype=torch.bfloat16)}
    with pytest.raises(mfr.MFRError) as ei:
        mfr.finalize_residual_rmsnorm_host(plan, h, ho, ws)
    assert ei.value.code == 1
    assert mfr.FinalizePlan(4, 4096, 8).host_workspace_bytes() == -1
