"""The NVFP4 epilogue (residual + RMSNorm, output quantised to NVFP4)
against the oracle.

The GPU computes the normalised value y in FP32 (rsqrtf, an FP32 sum of
squares); the oracle computes it in double and rounds once to FP32, so the
two y differ by a few units in the last place.  Both then take every
quantisation decision (block scale, codes) with the same FP32 steps.  A
decision can therefore only differ where the oracle's own decision flips
when y moves by a few ulps: such blocks / elements are "ambiguous" (found by
quantising y * (1 -/+ 2^-16) with the oracle) and are checked for validity
instead of equality.  Everything else must be equal.
"""
import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import oracle
import workloads as W
from helpers import assert_residual_close, bf16_bits, f32

pytestmark = pytest.mark.gpu
REL = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    mfr.build()
    mfr.load_library()


def _oracle_y32(inp, tokens=None):
    """Oracle x (FP32) and y rounded once to FP32, for the given tokens."""
    E, idx, w = bf16_bits(inp["expert_out"]), inp["permuted_row_of"].cpu().numpy(), f32(inp["topk_weights"])
    x, _ = oracle.weighted_residual(E, idx, w, f32(inp["residual"]), tokens=tokens)
    y = oracle.rmsnorm_f64(x, bf16_bits(inp["gamma"]), inp["eps"])
    return x, y.astype(np.float32)


def _s_enc(y32):
    return float(np.float32(448.0 * 6.0 / max(float(np.abs(y32).max()), 1e-30)))


def run_nvfp4(inp, s_enc, **kw):
    e = inp["expert_out"]
    T, k = inp["permuted_row_of"].shape
    R, H = e.shape
    plan = mfr.Nvfp4Plan(T, H, k, R, **kw)
    G = 64
    qb = torch.full((T * H // 2 + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    sb = torch.full((T * H // 16 + 2 * G,), 0x5A, dtype=torch.uint8, device="cuda")
    out_q, out_sf = qb[G:G + T * H // 2].view(T, H // 2), sb[G:G + T * H // 16].view(T, H // 16)
    rout = torch.empty_like(inp["residual"])
    plan.run(e, inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout, inp["gamma"], inp["eps"],
             s_enc, out_q, out_sf)
    torch.cuda.synchronize()
    for buf, fill in ((qb, 0xA5), (sb, 0x5A)):
        assert torch.all(buf[:G] == fill) and torch.all(buf[-G:] == fill), "write outside an NVFP4 output"
    return f32(rout), out_q.cpu().numpy(), out_sf.cpu().numpy(), plan


def _mag(codes):
    return np.where((codes & 7) == 0, 0, codes)       # +0 and -0 are the same value


def check_nvfp4(y32, s_enc, q_gpu, sf_gpu, max_ambiguous=0.01):
    q_o, sf_o = oracle.nvfp4_quantize(y32, s_enc)
    lo = oracle.nvfp4_quantize((y32 * np.float32(1 - REL)).astype(np.float32), s_enc)
    hi = oracle.nvfp4_quantize((y32 * np.float32(1 + REL)).astype(np.float32), s_enc)
    n, H = y32.shape
    c_o, c_g = oracle.unpack_e2m1(q_o), oracle.unpack_e2m1(q_gpu)
    c_lo, c_hi = oracle.unpack_e2m1(lo[0]), oracle.unpack_e2m1(hi[0])
    amb_block = (lo[1] != sf_o) | (hi[1] != sf_o)
    amb_elem = (c_lo != c_o) | (c_hi != c_o) | np.repeat(amb_block, 16, axis=1)
    sure_block = ~amb_block
    assert np.array_equal(sf_gpu[sure_block], sf_o[sure_block]), "block scale differs away from a rounding boundary"
    same_sf = np.repeat(sf_gpu == sf_o, 16, axis=1)
    sure = ~amb_elem & same_sf
    assert np.array_equal(_mag(c_g[sure]), _mag(c_o[sure])), "E2M1 code differs away from a rounding boundary"
    assert amb_elem.mean() <= max_ambiguous
    # every element, ambiguous or not: the GPU's code is a nearest E2M1 value of
    # y * enc for the GPU's own block scale, within the y uncertainty
    dec = (oracle.default().e4m3_to_f64(sf_gpu).astype(np.float32) / np.float32(s_enc)).astype(np.float32)
    with np.errstate(divide="ignore"):
        enc = np.where(sf_gpu == 0, np.float32(0), (np.float32(1) / dec).astype(np.float32))
    z = y32.astype(np.float64) * np.repeat(enc, 16, axis=1)
    vals = oracle.default().e2m1_to_f64(c_g)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    best = np.min(np.abs(np.abs(z)[..., None] - mags), axis=-1)
    assert np.all(np.abs(vals - z) <= best + np.abs(z) * 2 * REL + 1e-30)


CASES = [
    ("tiny_ref", W.TINY_REF, {}),
    ("decode_T1_cluster", W.decode(1), {}),
    ("decode_T8_cluster", W.decode(8), {}),
    ("decode_T64_rows", W.decode(64), dict(variant=mfr.VARIANT_ROWS)),
    ("prefill_T300_rows", W.PREFILL.with_(T=300), {}),
    ("prefill_T2000_stream", W.PREFILL.with_(T=2000), {}),
    ("wide_T64", W.wide(64), {}),
    ("wide_T200_stream", W.wide(200), dict(variant=mfr.VARIANT_STREAM)),
    ("stress_T40", W.STRESS.with_(T=40), {}),
    ("H16384_T5", W.Workload("h16k", T=5, H=16384, k=8, E=32), {}),
    ("H1040_T7_cluster", W.Workload("h1040", T=7, H=1040, k=5, E=16), dict(variant=mfr.VARIANT_CLUSTER)),
    ("decode_T32_cluster8", W.decode(32), {}),                           # 64-thread CTAs at 2^17
    ("decode_T4_cluster16", W.decode(4), dict(variant=mfr.VARIANT_CLUSTER, cluster_size=16)),
    ("wide_T2_cluster16", W.wide(2), dict(variant=mfr.VARIANT_CLUSTER, cluster_size=16)),
]


@pytest.mark.parametrize("name,wl,kw", CASES, ids=[c[0] for c in CASES])
def test_nvfp4_matches_oracle(name, wl, kw):
    inp = W.make_inputs(wl, "cuda")
    x_o, y32 = _oracle_y32(inp)
    s_enc = _s_enc(y32)
    res, q, sf, plan = run_nvfp4(inp, s_enc, **kw)
    assert_residual_close(res, x_o)
    check_nvfp4(y32, s_enc, q, sf)
    assert plan.get_status() == 0


def test_nvfp4_repeats_bitwise_and_small_scales():
    inp = W.make_inputs(W.PREFILL.with_(T=700), "cuda")
    _, y32 = _oracle_y32(inp)
    for s_enc in (_s_enc(y32), 1.0, 1e-3):     # 1e-3 pushes most blocks to the E4M3 subnormal scales
        a = run_nvfp4(inp, s_enc)
        b = run_nvfp4(inp, s_enc)
        assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
        check_nvfp4(y32, s_enc, a[1], a[2], max_ambiguous=0.05)


def test_nvfp4_full_size_sampled_tokens():
    wl = W.PREFILL
    inp = W.make_inputs(wl, "cuda")
    rng = np.random.default_rng(9)
    tokens = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, size=30, replace=False)]))
    x_o, y32 = _oracle_y32(inp, tokens=tokens)
    s_enc = float(np.float32(448.0 * 6.0 / 16.0))        # |y| stays well below 16 for these inputs
    res, q, sf, plan = run_nvfp4(inp, s_enc)
    assert plan.info()["variant_name"] == "stream"
    assert_residual_close(res[tokens], x_o)
    check_nvfp4(y32, s_enc, q[tokens], sf[tokens])


def test_nvfp4_argument_checks():
    with pytest.raises(mfr.MFRError) as ei:
        mfr.Nvfp4Plan(4, 4104, 8)                        # H % 16 != 0
    assert ei.value.code == 2
    inp = W.make_inputs(W.decode(4), "cuda")
    plan = mfr.Nvfp4Plan(4, 4096, 8, 32)
    q = torch.empty((4, 2048), dtype=torch.uint8, device="cuda")
    sf = torch.empty((4, 256), dtype=torch.uint8, device="cuda")
    rout = torch.empty_like(inp["residual"])
    for s_enc in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(mfr.MFRError) as ei:
            plan.run(inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout,
                     inp["gamma"], 1e-6, s_enc, q, sf)
        assert ei.value.code == 1
    lib = mfr.load_library()
    code = lib.moe_finalize_rmsnorm_nvfp4_run(plan.handle, inp["expert_out"].data_ptr(),
                                              inp["permuted_row_of"].data_ptr(), inp["topk_weights"].data_ptr(),
                                              inp["residual"].data_ptr(), rout.data_ptr(), inp["gamma"].data_ptr(),
                                              1e-6, 10.0, q.data_ptr() + 2, sf.data_ptr(), None)
    assert code == 3                                     # out_q must be 4-byte aligned
    with pytest.raises(mfr.MFRError):                    # a bf16 run on an NVFP4 plan
        mfr.Plan.run(plan, inp["expert_out"], inp["permuted_row_of"], inp["topk_weights"], inp["residual"],
                     rout, inp["gamma"], 1e-6, torch.empty((4, 4096), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
