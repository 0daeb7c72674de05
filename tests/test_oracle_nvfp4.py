"""Pins for the oracle's NVFP4 quantiser: torch's E4M3 rounding, the E2M1
and E4M3 format definitions (closed forms), a hand-worked two-block row, and
properties of the block scale."""
import json
import os

import numpy as np
import torch

from oracle import unpack_e2m1

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_rounding_matches_torch_below_saturation(oracle_lib):
    rng = np.random.default_rng(31)
    x = np.concatenate([
        rng.uniform(-460, 460, 20000), rng.standard_normal(20000) * np.exp2(rng.integers(-14, 8, 20000)),
        # every midpoint between adjacent positive E4M3 values, and its neighbours
    ]).astype(np.float32)
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)), -mids])
    x = x[np.abs(x) < 464]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_lib.e4m3_from_f64(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_e4m3_saturation_and_decoding(oracle_lib):
    for x, b in [(464.0, 0x7E), (480.0, 0x7E), (1e30, 0x7E), (-1e9, 0xFE), (float("nan"), 0x7F),
                 (float("inf"), 0x7E), (float("-inf"), 0xFE),
                 (0.0, 0x00), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (448.0, 0x7E)]:
        assert int(oracle_lib.e4m3_from_f64([x])[0]) == b, x
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(oracle_lib.e4m3_to_f64(codes), want)
    assert np.isnan(oracle_lib.e4m3_to_f64([0x7F])[0])


def test_e2m1_closed_forms(oracle_lib):
    cases = [(0.0, 0x0), (0.24, 0x0), (0.25, 0x0), (0.26, 0x1), (0.5, 0x1), (0.75, 0x2), (1.0, 0x2),
             (1.25, 0x2), (1.26, 0x3), (1.75, 0x4), (2.5, 0x4), (2.51, 0x5), (3.0, 0x5), (3.5, 0x6),
             (4.99, 0x6), (5.0, 0x6), (5.01, 0x7), (6.0, 0x7), (1e9, 0x7), (-1.75, 0xC), (-6.5, 0xF),
             (-0.1, 0x8), (-0.3, 0x9)]
    got = oracle_lib.e2m1_from_f64([c[0] for c in cases])
    assert [int(g) for g in got] == [c[1] for c in cases]


def test_e2m1_decoding_follows_the_bit_fields(oracle_lib):
    for c in range(16):
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        mag = (m * 0.5) if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert oracle_lib.e2m1_to_f64([c])[0] == (-mag if s else mag)


def test_hand_worked_two_blocks(oracle_lib):
    with open(os.path.join(GOLDEN, "nvfp4_two_blocks_hand_worked.json")) as f:
        g = json.load(f)
    y = np.array([g["y"]], dtype=np.float32)
    q, sf = oracle_lib.nvfp4_quantize(y, g["s_enc"])
    assert [f"{b:02X}" for b in sf[0]] == g["expected_scale_bytes"]
    assert [f"{b:02X}" for b in q[0]] == g["expected_packed_bytes"]
    codes = unpack_e2m1(q)[0]
    want = [int(c, 16) for blk in g["expected_codes"] for c in blk]
    assert [int(c) for c in codes] == want


def test_block_scale_properties(oracle_lib):
    """sf is the E4M3 rounding of amax/6*s_enc; every element's code is the
    nearest E2M1 value to y * enc with enc = s_enc / value(sf); zero blocks
    give sf = 0 and zero codes; scaling y and 1/s_enc together by a power of
    two changes nothing."""
    rng = np.random.default_rng(32)
    y = (rng.standard_normal((6, 64)) * np.exp2(rng.integers(-6, 6, (6, 1)))).astype(np.float32)
    y[2, 16:32] = 0.0
    s_enc = 448.0 * 6.0 / float(np.abs(y).max())
    q, sf = oracle_lib.nvfp4_quantize(y, s_enc)
    codes = unpack_e2m1(q)
    amax = np.abs(y.reshape(6, 4, 16)).max(axis=2)
    assert np.array_equal(sf, oracle_lib.e4m3_from_f64((amax.astype(np.float32) / np.float32(6)).astype(np.float32)
                                                      * np.float32(s_enc)))
    assert sf[2, 1] == 0 and not codes[2, 16:32].any()
    dec = (oracle_lib.e4m3_to_f64(sf).astype(np.float32) / np.float32(s_enc)).astype(np.float32)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for i in range(6):
        for b in range(4):
            if sf[i, b] == 0:
                continue
            enc = np.float32(1.0) / dec[i, b]
            z = (y[i, b * 16:(b + 1) * 16] * enc).astype(np.float64)
            vals = oracle_lib.e2m1_to_f64(codes[i, b * 16:(b + 1) * 16])
            err = np.abs(vals - z)
            best = np.min(np.abs(np.abs(z)[:, None] - mags[None, :]), axis=1)
            assert np.all(err <= best + 1e-12)                # nearest representable
    q2, sf2 = oracle_lib.nvfp4_quantize((y * np.float32(4)).astype(np.float32), s_enc / 4)
    assert np.array_equal(q2, q) and np.array_equal(sf2, sf)


def test_hand_worked_encode_at_given_scales(oracle_lib):
    """The codes for block scales the caller chooses (the check of an
    implementation whose scale decision may differ at a rounding boundary)."""
    with open(os.path.join(GOLDEN, "nvfp4_encode_at_given_scales_hand_worked.json")) as f:
        g = json.load(f)
    y = np.array([g["y"]], dtype=np.float32)
    sf = np.array([[int(b, 16) for b in g["scale_bytes"]]], dtype=np.uint8)
    q = oracle_lib.nvfp4_encode(y, g["s_enc"], sf)
    assert [f"{b:02X}" for b in q[0]] == g["expected_packed_bytes"]
    want = [int(c, 16) for blk in g["expected_codes"] for c in blk]
    assert [int(c) for c in unpack_e2m1(q)[0]] == want


def test_encode_at_the_quantisers_own_scales_gives_its_codes(oracle_lib):
    """At the scales the quantiser chose, encoding reproduces its codes; at
    any scale every code is the nearest E2M1 value of y * s_enc / value(sf)."""
    rng = np.random.default_rng(33)
    y = (rng.standard_normal((5, 48)) * np.exp2(rng.integers(-4, 4, (5, 1)))).astype(np.float32)
    s_enc = 448.0 * 6.0 / float(np.abs(y).max())
    q, sf = oracle_lib.nvfp4_quantize(y, s_enc)
    assert np.array_equal(oracle_lib.nvfp4_encode(y, s_enc, sf), q)
    other = np.clip(sf.astype(np.int64) + rng.integers(-3, 4, sf.shape), 1, 0x7E).astype(np.uint8)
    codes = unpack_e2m1(oracle_lib.nvfp4_encode(y, s_enc, other))
    dec = (oracle_lib.e4m3_to_f64(other).astype(np.float32) / np.float32(s_enc)).astype(np.float32)
    enc = (np.float32(1.0) / dec).astype(np.float32)
    z = (y * np.repeat(enc, 16, axis=1)).astype(np.float64)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    best = np.min(np.abs(np.abs(z)[..., None] - mags), axis=-1)
    assert np.all(np.abs(oracle_lib.e2m1_to_f64(codes) - z) <= best + 1e-12)


def test_hand_worked_scale_tile_offsets(oracle_lib):
    """The tiled block-scale layout of block-scaled FP4 GEMMs, by hand."""
    with open(os.path.join(GOLDEN, "nvfp4_scale_tiles_hand_worked.json")) as f:
        g = json.load(f)
    n, S = g["n"], g["S"]
    # every scale carries its own (row, col) code, so its position can be found
    sf = np.zeros((n, S), dtype=np.uint8)
    for case in g["cases"]:
        sf[case["row"], case["col"]] = 1 + g["cases"].index(case)
    out = oracle_lib.nvfp4_swizzle_scales(sf, fill=0)
    assert out.size == g["total_bytes"]
    for i, case in enumerate(g["cases"]):
        assert np.flatnonzero(out == i + 1).tolist() == [case["offset"]], case


def test_scale_tiles_are_a_bijection_and_leave_padding(oracle_lib):
    """Full tiles: every byte receives exactly one scale.  Partial tiles: the
    padding keeps its fill byte, nothing else does."""
    n, S = 256, 8
    idx = np.arange(n * S, dtype=np.int64)
    lo = (idx & 0xFF).astype(np.uint8).reshape(n, S)
    hi = (idx >> 8).astype(np.uint8).reshape(n, S)
    back = oracle_lib.nvfp4_swizzle_scales(lo).astype(np.int64) | \
        (oracle_lib.nvfp4_swizzle_scales(hi).astype(np.int64) << 8)
    assert sorted(back.tolist()) == list(range(n * S))
    sf = np.full((5, 3), 7, dtype=np.uint8)
    out = oracle_lib.nvfp4_swizzle_scales(sf, fill=0xEE)
    assert out.size == 128 * 4 and (out == 7).sum() == 15 and (out == 0xEE).sum() == 128 * 4 - 15
    # rows 32 apart share a 16-byte group; consecutive rows are 16 bytes apart
    pos = {v: int(np.flatnonzero(oracle_lib.nvfp4_swizzle_scales(
        np.where(np.arange(128)[:, None] == v, 9, 0).astype(np.uint8)[:, :4]) == 9)[0]) for v in (0, 1, 32, 64, 96)}
    assert pos == {0: 0, 1: 16, 32: 4, 64: 8, 96: 12}
