"""The launch-plus-one-pass floor kernel (moe_finalize_rmsnorm_launch_floor_work):
it runs with a plan's launch geometry, writes only inside its output
buffers, raises no status bit, and refuses plans and arguments it does not
cover."""
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W

pytestmark = pytest.mark.gpu
G = 512


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


@pytest.mark.parametrize("T,kw", [(1, {}), (8, {}), (64, {}), (300, {}),
                                  (4, dict(variant=mfr.VARIANT_ROWS)),
                                  (2, dict(variant=mfr.VARIANT_CLUSTER, cluster_size=16))],
                         ids=["T1", "T8", "T64", "T300", "T4_rows", "T2_c16"])
@pytest.mark.parametrize("work", range(8))
def test_floor_work_stays_in_bounds(T, kw, work):
    inp = W.make_inputs(W.decode(T) if T <= 128 else W.PREFILL.with_(T=T), "cuda")
    H = 4096
    plan = mfr.Plan(T, H, 8, T * 8, **kw)
    rb = torch.full((T * H + 2 * G,), -3.0, dtype=torch.float32, device="cuda")
    ob = torch.full((T * H + 2 * G,), -7.0, dtype=torch.bfloat16, device="cuda")
    rout, out = rb[G:G + T * H].view(T, H), ob[G:G + T * H].view(T, H)
    for _ in range(3):
        plan.launch_floor_work(work, inp["expert_out"], inp["permuted_row_of"], inp["residual"], rout, out)
    torch.cuda.synchronize()
    for buf, fill in ((rb, -3.0), (ob, -7.0)):
        assert torch.all(buf[:G] == fill) and torch.all(buf[-G:] == fill), "a write outside an output"
    if work & mfr.FLOOR_STORE and work & mfr.FLOOR_LOAD:
        assert torch.equal(rout, inp["residual"])        # the residual it loaded, stored back
    elif not work & mfr.FLOOR_STORE:
        assert torch.all(rout == -3.0)
    assert plan.get_status() == 0


def test_floor_work_refuses_what_it_does_not_cover():
    inp = W.make_inputs(W.decode(2), "cuda")
    plan = mfr.Plan(2, 4096, 8, 16)
    for work in (-1, 8):
        with pytest.raises(mfr.MFRError) as ei:
            plan.launch_floor_work(work, inp["expert_out"], inp["permuted_row_of"])
        assert ei.value.code == 1
    with pytest.raises(mfr.MFRError) as ei:                       # loads need their inputs
        plan.launch_floor_work(mfr.FLOOR_LOAD, None, inp["permuted_row_of"])
    assert ei.value.code == 1
    stream_plan = mfr.Plan(4096, 4096, 8, variant=mfr.VARIANT_STREAM)
    with pytest.raises(mfr.MFRError) as ei:
        stream_plan.launch_floor_work(0, None, inp["permuted_row_of"])
    assert ei.value.code == 2
    for other in (mfr.FinalizePlan(2, 4096, 8, 16), mfr.Nvfp4Plan(2, 4096, 8, 16)):
        with pytest.raises(mfr.MFRError) as ei:
            other.launch_floor_work(0, None, inp["permuted_row_of"])
        assert ei.value.code == 1
    torch.cuda.synchronize()
