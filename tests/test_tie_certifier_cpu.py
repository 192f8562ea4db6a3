"""The tie certifier of the GPU output tests (tests/gpu_case.py, certify_l2_codes), checked on the
CPU with planted codes: it accepts a differing L2-input code only where the oracle's value lies
within tau of the rounding midpoint between the two codes, and rejects any other difference (a
wrong code one step away from a value that is not at a midpoint, a code two steps away, or a
wrong block scale away from a scale boundary)."""
import numpy as np
import pytest

import gpu_case as G
from oracle import formats as OF
from oracle import moe as OM


def _row_with(value_at, v, n=32, base=0.3):
    """One MXFP8 block of 32 values whose amax 3.9 fixes the block exponent at -6 (3.9 <= 448 * 2^-6):
    codes hold the values times 64, so near 1.0 they step by 0.125 (E4M3 spacing 8 between 64 and 128),
    with element `value_at` set to v."""
    h = np.full((1, n), base, dtype=np.float64)
    h[0, 0] = 3.9            # fixes the block amax, so the exponent does not move
    h[0, value_at] = v
    return h


def _codes(h):
    return OM.l2_input_codes(h.astype(np.float32), "mxfp8")


def test_accepts_the_other_neighbour_of_a_midpoint():
    # 1.0625 is the midpoint of the E4M3 values 1.0 and 1.125: a value just above it rounds up
    h = _row_with(5, 1.0625 + 1e-7)
    codes, sf = _codes(h)
    got = codes.copy()
    assert sf[0, 0] == 127 - 6
    got[0, 5] = OF.e4m3_encode(np.array([64.0]))[0]      # 1.0 * 64: the other neighbour
    deq, n = G.certify_l2_codes(h, got, sf, "mxfp8", None, tau=1e-5)
    assert n == 1 and deq[0, 5] == 1.0


def test_rejects_a_wrong_code_away_from_a_midpoint():
    h = _row_with(5, 1.03)                               # rounds to 1.0, far from the midpoint 1.0625
    codes, sf = _codes(h)
    got = codes.copy()
    got[0, 5] = OF.e4m3_encode(np.array([72.0]))[0]      # 1.125 * 64: one step up, but 1.03 is no tie
    with pytest.raises(AssertionError):
        G.certify_l2_codes(h, got, sf, "mxfp8", None, tau=1e-5)


def test_rejects_a_code_two_steps_away_even_at_a_midpoint():
    h = _row_with(5, 1.0625 + 1e-7)
    codes, sf = _codes(h)
    got = codes.copy()
    got[0, 5] = OF.e4m3_encode(np.array([80.0]))[0]      # 1.25 * 64: two steps from the oracle's 1.125
    with pytest.raises(AssertionError):
        G.certify_l2_codes(h, got, sf, "mxfp8", None, tau=1e-5)


def test_rejects_a_wrong_block_scale_away_from_a_boundary():
    h = _row_with(5, 1.0)
    codes, sf = _codes(h)
    got_sf = sf.copy()
    got_sf[0, 0] += 1                                    # amax 3.9 is far from 448 * 2^e
    with pytest.raises(AssertionError):
        G.certify_l2_codes(h, codes, got_sf, "mxfp8", None, tau=1e-5)


def test_equal_codes_pass_with_no_difference():
    h = _row_with(7, 1.7)
    codes, sf = _codes(h)
    deq, n = G.certify_l2_codes(h, codes.copy(), sf.copy(), "mxfp8", None, tau=1e-5)
    assert n == 0
    assert np.array_equal(deq, OF.mxfp8_dequantize(codes, sf))
