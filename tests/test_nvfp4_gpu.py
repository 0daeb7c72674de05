"""The NVFP4 epilogue (residual + RMSNorm, output quantised to NVFP4)
against the oracle.

The rules of the output check are those of nvfp4_check.check_nvfp4: scales
and codes equal to the oracle's, except where the oracle's own decision
flips when y moves by 2^-16 relative; there the kernel's scale must be one of
the oracle's neighbouring decisions and its codes the oracle's codes at that
scale.
"""
import numpy as np
import pytest
import torch

import moe_finalize_residual_rmsnorm_gb300 as mfr
import oracle
import workloads as W
from helpers import assert_residual_close, bf16_bits, f32, host_inputs, over_all_tokens
from nvfp4_check import check_nvfp4

pytestmark = pytest.mark.gpu


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
    # the ring with small k: deeper rings that wrap many times per CTA
    ("k2_T1500_stream", W.Workload("k2", T=1500, H=4096, k=2, E=16), dict(variant=mfr.VARIANT_STREAM)),
    ("k4_H8192_T700_stream", W.Workload("k4w", T=700, H=8192, k=4, E=16), dict(variant=mfr.VARIANT_STREAM)),
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


def test_nvfp4_full_size_every_token():
    """Every token of the prefill call, with the oracle spread over the host
    cores."""
    wl = W.PREFILL
    inp = W.make_inputs(wl, "cuda")
    s_enc = float(np.float32(448.0 * 6.0 / 16.0))        # |y| stays well below 16 for these inputs
    res, q, sf, plan = run_nvfp4(inp, s_enc)
    assert plan.info()["variant_name"] == "stream"
    assert plan.get_status() == 0
    h = host_inputs(inp)
    del inp
    torch.cuda.empty_cache()

    def check(tk):
        x_o, _ = oracle.weighted_residual(h["E"], h["idx"], h["w"], h["res"], tokens=tk)
        y32 = oracle.rmsnorm_f64(x_o, h["gamma"], h["eps"]).astype(np.float32)
        sl = slice(tk[0], tk[-1] + 1)
        assert_residual_close(res[sl], x_o, what=f"residual_out tokens {tk[0]}..")
        check_nvfp4(y32, s_enc, q[sl], sf[sl])
    assert over_all_tokens(wl.T, check) == wl.T


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


# ---- block scales in the tiled layout of block-scaled FP4 GEMMs ----------------------

PAD = 0xEE


def _tile_offsets(T, S):
    """offsets[r, c]: the byte of scale (r, c) in the tiled layout, from the
    oracle's layout map applied to the scales' own indices."""
    idx = np.arange(T * S, dtype=np.int64).reshape(T, S)
    lo = oracle.nvfp4_swizzle_scales((idx & 0xFF).astype(np.uint8))
    mid = oracle.nvfp4_swizzle_scales(((idx >> 8) & 0xFF).astype(np.uint8))
    hi = oracle.nvfp4_swizzle_scales(((idx >> 16) & 0xFF).astype(np.uint8))
    flat = lo.astype(np.int64) | (mid.astype(np.int64) << 8) | (hi.astype(np.int64) << 16)
    written = np.zeros(flat.size, dtype=bool)
    written[oracle.nvfp4_swizzle_scales(np.ones((T, S), dtype=np.uint8), fill=0) == 1] = True
    offsets = np.empty(T * S, dtype=np.int64)
    offsets[flat[written]] = np.flatnonzero(written)
    return offsets.reshape(T, S), written


def run_nvfp4_tiled(inp, s_enc, **kw):
    e = inp["expert_out"]
    T, k = inp["permuted_row_of"].shape
    R, H = e.shape
    plan = mfr.Nvfp4Plan(T, H, k, R, sf_layout=mfr.SF_TILED_128x4, **kw)
    n = plan.sf_bytes()
    assert n == -(-T // 128) * 128 * (-(-(H // 16) // 4) * 4)
    G = 64
    qb = torch.full((T * H // 2 + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    sb = torch.full((n + 2 * G,), PAD, dtype=torch.uint8, device="cuda")
    out_q, out_sf = qb[G:G + T * H // 2].view(T, H // 2), sb[G:G + n]
    rout = torch.empty_like(inp["residual"])
    plan.run(e, inp["permuted_row_of"], inp["topk_weights"], inp["residual"], rout, inp["gamma"], inp["eps"],
             s_enc, out_q, out_sf)
    torch.cuda.synchronize()
    assert torch.all(qb[:G] == 0xA5) and torch.all(qb[-G:] == 0xA5), "write outside out_q"
    assert torch.all(sb[:G] == PAD) and torch.all(sb[-G:] == PAD), "write outside out_sf"
    return f32(rout), out_q.cpu().numpy(), out_sf.cpu().numpy(), plan


TILED_CASES = [
    ("decode_T1_cluster", W.decode(1), {}),
    ("decode_T8_cluster", W.decode(8), {}),
    ("prefill_T300_rows", W.PREFILL.with_(T=300), {}),
    ("prefill_T2000_stream", W.PREFILL.with_(T=2000), {}),
    ("wide_T129_stream", W.wide(129), dict(variant=mfr.VARIANT_STREAM)),
    ("H1040_T7_cluster", W.Workload("h1040", T=7, H=1040, k=5, E=16), dict(variant=mfr.VARIANT_CLUSTER)),
    ("H16384_T5", W.Workload("h16k", T=5, H=16384, k=8, E=32), {}),
    ("H4112_T700_stream", W.Workload("h4112", T=700, H=4112, k=8, E=64), dict(variant=mfr.VARIANT_STREAM)),
    ("H4144_T300_stream", W.Workload("h4144", T=300, H=4144, k=6, E=48), dict(variant=mfr.VARIANT_STREAM)),
]


@pytest.mark.parametrize("name,wl,kw", TILED_CASES, ids=[c[0] for c in TILED_CASES])
def test_nvfp4_tiled_scales(name, wl, kw):
    """The tiled plan writes every scale where the oracle's layout map puts
    it, leaves the padding alone, and its codes and scales are the row-major
    plan's, byte for byte (and pass the oracle check)."""
    inp = W.make_inputs(wl, "cuda")
    x_o, y32 = _oracle_y32(inp)
    s_enc = _s_enc(y32)
    res, q, sf_tiled, plan = run_nvfp4_tiled(inp, s_enc, **kw)
    offsets, written = _tile_offsets(wl.T, wl.H // 16)
    assert np.all(sf_tiled[~written] == PAD), "a padding byte of the scale tiles was written"
    sf = sf_tiled[offsets]
    assert_residual_close(res, x_o)
    check_nvfp4(y32, s_enc, q, sf)
    _, q_rm, sf_rm, _ = run_nvfp4(inp, s_enc, **kw)
    assert np.array_equal(q, q_rm) and np.array_equal(sf, sf_rm)
    assert plan.get_status() == 0


def test_nvfp4_tiled_output_feeds_a_block_scaled_gemm():
    """out_q with its tiled scales, handed to a block-scaled FP4 GEMM
    (torch._scaled_mm through cuBLASLt) as the A operand, gives the product
    of the dequantised values: the layout is the one such GEMMs read."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no FP4 dtype")
    wl = W.PREFILL.with_(T=256)
    inp = W.make_inputs(wl, "cuda")
    _, y32 = _oracle_y32(inp)
    s_enc = _s_enc(y32)
    _, q, sf_tiled, _ = run_nvfp4_tiled(inp, s_enc)
    T, H, N = wl.T, wl.H, 128
    rng = np.random.default_rng(3)
    b_codes = rng.integers(0, 16, (N, H)).astype(np.uint8)
    b_sf = rng.integers(0x30, 0x40, (N, H // 16)).astype(np.uint8)
    b_packed = (b_codes[:, 0::2] | (b_codes[:, 1::2] << 4)).astype(np.uint8)
    e2m1 = oracle.default().e2m1_to_f64(np.arange(16, dtype=np.uint8))
    e4m3 = oracle.default().e4m3_to_f64(np.arange(256, dtype=np.uint8))
    offsets, _ = _tile_offsets(T, H // 16)
    a = e2m1[oracle.unpack_e2m1(q)] * np.repeat(e4m3[sf_tiled[offsets]], 16, axis=1)
    b = e2m1[b_codes] * np.repeat(e4m3[b_sf], 16, axis=1)
    want = a @ b.T
    ta = torch.from_numpy(q).cuda().view(torch.float4_e2m1fn_x2)
    tb = torch.from_numpy(b_packed).cuda().view(torch.float4_e2m1fn_x2)
    sa = torch.from_numpy(sf_tiled).cuda().view(torch.float8_e4m3fn)
    sb = torch.from_numpy(oracle.nvfp4_swizzle_scales(b_sf)).cuda().view(torch.float8_e4m3fn)
    try:
        got = torch._scaled_mm(ta, tb.t(), sa, sb, out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError) as e:
        pytest.skip(f"no block-scaled FP4 GEMM in this torch build: {e}")
    got = got.cpu().double().numpy()
    # FP32 accumulation of H products in any order: within H * 2^-24 of the
    # sum of their magnitudes (a wrong scale layout misses by O(1))
    bound = H * 2.0 ** -24 * (np.abs(a) @ np.abs(b).T)
    assert np.all(np.abs(got - want) <= bound + 1e-30)
