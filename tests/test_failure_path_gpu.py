"""The failure path without a fault: every on-chip wait of the library is
bounded, and one that runs out sets MFR_STATUS_TIMEOUT and returns.  Here a
wait on a barrier that nothing arrives on runs out (about a millisecond),
the host reads the status, and the same plan then computes a correct call:
the context stays usable."""
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from test_parity_gpu import compare_full, run_gpu

pytestmark = pytest.mark.gpu
LIMIT = 2_000_000   # SM cycles: about 1 ms


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    inp = W.make_inputs(W.decode(8), "cuda")
    plan = mfr.Plan(8, 4096, 8, inp["expert_out"].shape[0])
    plan.wait_selftest(LIMIT, arrive=False)
    assert plan.get_status() == mfr.STATUS_TIMEOUT
    assert plan.get_status() == 0                      # reading clears the word
    plan.wait_selftest(LIMIT, arrive=True)             # the barrier completes: no timeout
    assert plan.get_status() == 0
    plan.wait_selftest(LIMIT, arrive=False)
    torch.cuda.synchronize()
    compare_full(inp, plan=plan)                       # a real call on the same plan and context
    with pytest.raises(mfr.MFRError):
        plan.wait_selftest(0, arrive=True)


def test_debug_checks_turn_a_timeout_into_an_error():
    inp = W.make_inputs(W.decode(4), "cuda")
    plan = mfr.Plan(4, 4096, 8, inp["expert_out"].shape[0], debug_checks=True)
    plan.wait_selftest(LIMIT, arrive=False)
    with pytest.raises(mfr.MFRError):
        run_gpu(inp, plan=plan)                        # the run reads the word and reports the timeout
    got_res, got_out, _ = run_gpu(inp, plan=plan)      # the word was cleared; the next call is clean
    assert plan.get_status() == 0
