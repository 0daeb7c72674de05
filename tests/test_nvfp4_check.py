"""The NVFP4 output check of the GPU tests (nvfp4_check.check_nvfp4),
exercised on the CPU with doctored kernel outputs: the oracle's own output
passes, the other valid decision at a scale-rounding boundary passes, and a
wrong scale (on a boundary block or elsewhere), or codes that do not belong
to the reported scale, fail.  No GPU is involved."""
import numpy as np
import pytest

import oracle
from nvfp4_check import check_nvfp4

S_ENC = 1.0


def _row_with_a_boundary_block():
    """Two rows of 64 elements.  Block (0, 1) has amax 6.375, so its scale
    input (6.375 / 6) * 1 = 1.0625 is the midpoint of the E4M3 values 1
    (0x38) and 1.125 (0x39): the oracle picks 0x38 (even) for y, 0x39 for
    y * (1 + 2^-16).  The other blocks sit well inside one E4M3 step."""
    rng = np.random.default_rng(5)
    y = rng.uniform(-1.0, 1.0, (2, 64)).astype(np.float32)
    for b in range(4):
        y[:, b * 16] = np.float32(2.9)                 # amax 2.9: 0.4833 is no E4M3 midpoint
    y[0, 16:32] = np.array([6.375, -5.0, 4.4, 3.3, 2.2, 1.1, 0.3, -0.7,
                            5.5, -2.6, 1.9, 0.9, -4.1, 3.7, 2.05, -1.45], dtype=np.float32)
    return y


def test_the_oracles_own_output_passes():
    y = _row_with_a_boundary_block()
    q, sf = oracle.nvfp4_quantize(y, S_ENC)
    assert sf[0, 1] == 0x38
    n_blocks, _ = check_nvfp4(y, S_ENC, q, sf, max_ambiguous=0.5)
    assert n_blocks == 1


def test_the_other_decision_at_a_scale_boundary_passes():
    y = _row_with_a_boundary_block()
    _, sf = oracle.nvfp4_quantize(y, S_ENC)
    sf2 = sf.copy()
    sf2[0, 1] = 0x39                                   # the decision for y * (1 + 2^-16)
    q2 = oracle.nvfp4_encode(y, S_ENC, sf2)
    check_nvfp4(y, S_ENC, q2, sf2, max_ambiguous=0.5)


@pytest.mark.parametrize("wrong", [0x3A, 0x37, 0x40])
def test_a_wrong_scale_on_a_boundary_block_fails(wrong):
    """Its codes are the nearest ones for that scale, so only the scale
    itself gives it away."""
    y = _row_with_a_boundary_block()
    _, sf = oracle.nvfp4_quantize(y, S_ENC)
    bad = sf.copy()
    bad[0, 1] = wrong
    q_bad = oracle.nvfp4_encode(y, S_ENC, bad)
    with pytest.raises(AssertionError, match="none of the oracle's neighbouring decisions"):
        check_nvfp4(y, S_ENC, q_bad, bad, max_ambiguous=0.5)


def test_a_wrong_scale_on_a_sure_block_fails():
    y = _row_with_a_boundary_block()
    _, sf = oracle.nvfp4_quantize(y, S_ENC)
    bad = sf.copy()
    bad[1, 2] += 1
    with pytest.raises(AssertionError, match="away from a rounding boundary"):
        check_nvfp4(y, S_ENC, oracle.nvfp4_encode(y, S_ENC, bad), bad, max_ambiguous=0.5)


def test_codes_of_another_scale_than_the_reported_one_fail():
    """Scale 0x39 reported on the boundary block, codes encoded at 0x38."""
    y = _row_with_a_boundary_block()
    q, sf = oracle.nvfp4_quantize(y, S_ENC)
    sf2 = sf.copy()
    sf2[0, 1] = 0x39
    assert not np.array_equal(oracle.nvfp4_encode(y, S_ENC, sf2)[0, 8:16], q[0, 8:16])
    with pytest.raises(AssertionError, match="not the oracle's code"):
        check_nvfp4(y, S_ENC, q, sf2, max_ambiguous=0.5)


def test_one_flipped_code_fails():
    y = _row_with_a_boundary_block()
    q, sf = oracle.nvfp4_quantize(y, S_ENC)
    bad = q.copy()
    bad[1, 5] ^= 0x01                                  # element 10 of row 1: one code step
    with pytest.raises(AssertionError, match="not the oracle's code"):
        check_nvfp4(y, S_ENC, bad, sf, max_ambiguous=0.5)


def test_plus_and_minus_zero_codes_are_the_same_value():
    y = _row_with_a_boundary_block()
    y[1, 40:44] = np.float32(0.0)
    q, sf = oracle.nvfp4_quantize(y, S_ENC)
    q2 = q.copy()
    q2[1, 20] |= 0x08                                  # element 40: -0 instead of +0
    q2[1, 21] |= 0x80                                  # element 43: -0 instead of +0
    check_nvfp4(y, S_ENC, q2, sf, max_ambiguous=0.5)


def test_too_many_ambiguous_elements_fail():
    y = _row_with_a_boundary_block()
    q, sf = oracle.nvfp4_quantize(y, S_ENC)
    with pytest.raises(AssertionError, match="ambiguous"):
        check_nvfp4(y, S_ENC, q, sf, max_ambiguous=0.01)
