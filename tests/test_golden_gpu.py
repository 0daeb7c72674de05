"""The hand-worked examples of tests/golden/ through the CUDA path: the
kernels must reproduce values derived by hand (not only the oracle's), in
every variant that can run them.  The examples use powers of two, so the
residual is exact; the bf16 outputs are compared within 1 ulp (the kernels
round once from FP32, the derivations from the exact value)."""
import json
import os

import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
from helpers import bf16_ulp_distance

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def bf16_tensor(bits):
    a = np.array([[int(b, 16) for b in row] for row in bits] if isinstance(bits[0], list)
                 else [int(b, 16) for b in bits], dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def out_bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("variant", [mfr.VARIANT_ROWS, mfr.VARIANT_STREAM], ids=["rows", "ring"])
@pytest.mark.parametrize("pdl", [True, False])
def test_hand_worked_fused_path(variant, pdl):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_t2_h8_k2.json")))
    T, H, k, R = g["T"], g["H"], g["k"], g["R"]
    E = torch.tensor(g["expert_out"], dtype=torch.float32).to(torch.bfloat16).cuda()
    idx = torch.tensor(g["permuted_row_of"], dtype=torch.int32).cuda()
    w = torch.tensor(g["topk_weights"], dtype=torch.float32).cuda()
    res = torch.tensor(g["residual_in"], dtype=torch.float32).cuda()
    gamma = bf16_tensor(g["gamma_bits"])
    rout = torch.empty_like(res)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    plan = mfr.Plan(T, H, k, R, variant=variant, enable_pdl=pdl)
    plan.run(E, idx, w, res, rout, gamma, g["eps"], out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rout.cpu().numpy(), np.array(g["expected_residual_out"], dtype=np.float32))
    want = np.array([[int(b, 16) for b in row] for row in g["expected_out_bits"]], dtype=np.uint16)
    assert bf16_ulp_distance(out_bits(out), want).max() <= 1
    assert plan.get_status() == 0


@pytest.mark.parametrize("variant", [mfr.VARIANT_ROWS, mfr.VARIANT_STREAM], ids=["rows", "ring"])
def test_hand_worked_expert_norm(variant):
    g = json.load(open(os.path.join(GOLDEN, "expert_rmsnorm_hand_worked.json")))
    T, H, k, R = g["T"], g["H"], g["k"], g["R"]
    E = bf16_tensor(g["expert_out_bits"])
    idx = torch.tensor(g["permuted_row_of"], dtype=torch.int32).cuda()
    w = torch.tensor(g["topk_weights"], dtype=torch.float32).cuda()
    gamma = bf16_tensor(g["gamma_bits"])
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    plan = mfr.ExpertNormPlan(T, H, k, R, variant=variant)
    plan.run(E, idx, w, gamma, g["eps"], out)
    torch.cuda.synchronize()
    want = np.array([[int(b, 16) for b in row] for row in g["expected_out_bits"]], dtype=np.uint16)
    assert bf16_ulp_distance(out_bits(out), want).max() <= 1
    assert plan.get_status() == 0
