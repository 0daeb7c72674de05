"""Random shapes and options against the oracle: every output kind (fused,
plain finalize, NVFP4 with row-major or tiled block scales, per-expert
RMSNorm) under every variant that takes the shape, with seeded draws of T, H, k, the variant and the cluster size.  The
bars are the ones of the per-kind parity tests; the point here is breadth of
shapes (ragged H, any k from 1 to 16, token counts around the thresholds)."""
import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import workloads as W
from helpers import assert_out_close, assert_residual_close, oracle_finalize_only, oracle_expert_norm
from test_expert_norm_gpu import assert_expert_norm_close, run_expert_norm
from test_finalize_only_gpu import run_finalize
from test_nvfp4_gpu import PAD, _oracle_y32, _s_enc, _tile_offsets, check_nvfp4, run_nvfp4, run_nvfp4_tiled
from test_parity_gpu import compare_full

pytestmark = pytest.mark.gpu
KINDS = ("fused", "finalize", "nvfp4", "expert_norm")


def draw_cases(n=48, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        kind = KINDS[len(cases) % len(KINDS)]
        H = int(rng.integers(1, 1025)) * (16 if kind == "nvfp4" else 8)
        T = int(rng.choice([1, 2, 3, 7, 16, 31, 64, 129, 200, 300]))
        k = int(rng.integers(1, 17))
        variant = int(rng.choice([mfr.VARIANT_AUTO, mfr.VARIANT_ROWS, mfr.VARIANT_CLUSTER, mfr.VARIANT_STREAM]))
        cluster = int(rng.choice([0, 2, 4, 8, 16])) if variant == mfr.VARIANT_CLUSTER else 0
        cases.append((kind, T, H, k, variant, cluster, int(rng.integers(0, 2**31))))
    return cases


def pdl_of(seed):
    return seed % 3 != 0          # a third of the cases launch without programmatic dependent launch


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


@pytest.mark.parametrize("kind,T,H,k,variant,cluster,seed", draw_cases(),
                         ids=lambda v: str(v))
def test_random_shape_matches_oracle(kind, T, H, k, variant, cluster, seed):
    wl = W.Workload(f"fuzz_{kind}_T{T}_H{H}_k{k}", T=T, H=H, k=k, E=max(16, 2 * k), seed=seed % 100000,
                    extra_rows=int(seed % 5))
    inp = W.make_inputs(wl, "cuda")
    kw = dict(variant=variant, enable_pdl=pdl_of(seed))
    if cluster:
        kw["cluster_size"] = cluster
    try:
        if kind == "fused":
            compare_full(inp, kw)
        elif kind == "finalize":
            want, _ = oracle_finalize_only(inp)
            got, plan = run_finalize(inp, **kw)
            assert np.array_equal(got, want)
            assert plan.get_status() == 0
        elif kind == "nvfp4":
            x_o, y32 = _oracle_y32(inp)
            s_enc = _s_enc(y32)
            if seed % 2:             # half of the NVFP4 cases write their scales in the tiled layout
                res, q, sf_tiled, plan = run_nvfp4_tiled(inp, s_enc, **kw)
                offsets, written = _tile_offsets(T, H // 16)
                assert np.all(sf_tiled[~written] == PAD)
                sf = sf_tiled[offsets]
            else:
                res, q, sf, plan = run_nvfp4(inp, s_enc, **kw)
            assert_residual_close(res, x_o)
            check_nvfp4(y32, s_enc, q, sf, max_ambiguous=0.05)
            assert plan.get_status() == 0
        else:
            want, y, s, _ = oracle_expert_norm(inp)
            got, plan = run_expert_norm(inp, **kw)
            assert_expert_norm_close(got, want, y, s)
            assert plan.get_status() == 0
    except mfr.MFRError as e:
        # a forced variant the shape cannot take is refused by the plan, never run
        assert variant != mfr.VARIANT_AUTO, f"the automatic plan refused a supported shape: {e}"
        assert e.code in (1, 2), e
