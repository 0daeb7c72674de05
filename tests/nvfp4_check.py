"""The NVFP4 output check shared by the GPU tests, itself tested on the CPU
(tests/test_nvfp4_check.py).  No quantisation arithmetic lives here: every
scale and code it compares against comes from the oracle.

The kernels compute the normalised value y in FP32 (an FP32 sum of squares,
rsqrtf); the oracle computes it in double and rounds once to FP32, so the two
y differ by a few units in the last place.  Both take every quantisation
decision (block scale, codes) with the same FP32 steps, so a decision can only
differ where the oracle's own decision flips when y moves by a few ulps.  The
check therefore quantises y and y * (1 -/+ 2^-16) with the oracle:

* a block whose scale is the same for all three is "sure": the kernel's scale
  must equal it;
* on the other ("ambiguous") blocks the kernel's scale must be one of the
  oracle's scales for y * (1 - 2^-16), y and y * (1 + 2^-16);
* whatever the block, the kernel's codes must be the oracle's codes at the
  kernel's own scale (oracle.nvfp4_encode), for y, or, where those codes
  differ between y * (1 - 2^-16) and y * (1 + 2^-16), for one of them;
* at most `max_ambiguous` of the elements may lie in ambiguous blocks or at an
  ambiguous code.
"""
import numpy as np

import oracle

REL = 2.0 ** -16


def _same_code(a, b):
    """E2M1 codes equal as values (+0 and -0 are the same value)."""
    za, zb = (a & 7) == 0, (b & 7) == 0
    return (a == b) | (za & zb)


def check_nvfp4(y32, s_enc, q_gpu, sf_gpu, max_ambiguous=0.01):
    """y32 float32 [n, H] (the oracle's y rounded to FP32), q_gpu uint8
    [n, H/2] and sf_gpu uint8 [n, H/16] from the kernel.  Raises
    AssertionError on the first rule broken."""
    y32 = np.ascontiguousarray(y32, dtype=np.float32)
    q_gpu = np.ascontiguousarray(q_gpu, dtype=np.uint8)
    sf_gpu = np.ascontiguousarray(sf_gpu, dtype=np.uint8)
    y_lo = (y32 * np.float32(1 - REL)).astype(np.float32)
    y_hi = (y32 * np.float32(1 + REL)).astype(np.float32)
    _, sf_o = oracle.nvfp4_quantize(y32, s_enc)
    _, sf_lo = oracle.nvfp4_quantize(y_lo, s_enc)
    _, sf_hi = oracle.nvfp4_quantize(y_hi, s_enc)
    amb_block = (sf_lo != sf_o) | (sf_hi != sf_o)
    if not np.array_equal(sf_gpu[~amb_block], sf_o[~amb_block]):
        raise AssertionError("block scale differs away from a rounding boundary")
    if not np.all((sf_gpu == sf_o) | (sf_gpu == sf_lo) | (sf_gpu == sf_hi)):
        i = np.argwhere(~((sf_gpu == sf_o) | (sf_gpu == sf_lo) | (sf_gpu == sf_hi)))[0]
        raise AssertionError(f"block scale at {tuple(i)} is 0x{int(sf_gpu[tuple(i)]):02X}, none of the "
                             f"oracle's neighbouring decisions 0x{int(sf_lo[tuple(i)]):02X} / "
                             f"0x{int(sf_o[tuple(i)]):02X} / 0x{int(sf_hi[tuple(i)]):02X}")
    # the oracle's codes at the kernel's own scales
    c_g = oracle.unpack_e2m1(q_gpu)
    c_at = oracle.unpack_e2m1(oracle.nvfp4_encode(y32, s_enc, sf_gpu))
    c_at_lo = oracle.unpack_e2m1(oracle.nvfp4_encode(y_lo, s_enc, sf_gpu))
    c_at_hi = oracle.unpack_e2m1(oracle.nvfp4_encode(y_hi, s_enc, sf_gpu))
    amb_code = ~_same_code(c_at_lo, c_at) | ~_same_code(c_at_hi, c_at)
    ok = _same_code(c_g, c_at) | (amb_code & (_same_code(c_g, c_at_lo) | _same_code(c_g, c_at_hi)))
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"E2M1 code at {tuple(i)} is 0x{int(c_g[tuple(i)]):X}, not the oracle's code "
                             f"0x{int(c_at[tuple(i)]):X} at the kernel's block scale")
    amb = amb_code | np.repeat(amb_block, 16, axis=1)
    if amb.mean() > max_ambiguous:
        raise AssertionError(f"{amb.mean():.4f} of the elements are ambiguous (limit {max_ambiguous})")
    return int(amb_block.sum()), int(amb_code.sum())
