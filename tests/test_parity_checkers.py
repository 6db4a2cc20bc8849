"""The parity checkers themselves (tests/parity.py), on hand-made arrays:
each accepts what the tolerances allow and rejects a case just outside
them, so a GPU parity test cannot pass by a lenient checker.  CPU only."""
import numpy as np
import pytest

from parity import (E4M3, E5M2, check_codes, check_f16, check_f32_exact,
                    check_master)


def codes(n=4000, seed=0):
    c = np.random.default_rng(seed).integers(0, 0x7F, n).astype(np.uint8)
    return c[(c & 0x7F) < 0x78]          # finite in both formats


def test_codes_one_apart_allowed_below_the_exact_share():
    ref = codes()
    got = ref.copy()
    got[:3] += 1                         # 3 of ~3700: above 99.9% identical
    assert check_codes(got, ref) > 0.999
    got = ref.copy()
    got[:10] += 1                        # 10 of ~3700: below 99.9%
    with pytest.raises(AssertionError, match="identical"):
        check_codes(got, ref)


def test_codes_two_apart_rejected():
    ref = codes()
    got = ref.copy()
    got[7] = ref[7] + 2
    with pytest.raises(AssertionError, match="apart"):
        check_codes(got, ref)


def test_codes_across_zero():
    ref = np.array([0x01, 0x00, 0x80] * 2000, np.uint8)
    got = ref.copy()
    got[1] = 0x80                        # -0 for +0: the same value
    assert check_codes(got, ref) < 1.0
    got[0] = 0x81                        # -min for +min: two steps apart
    with pytest.raises(AssertionError, match="apart"):
        check_codes(got, ref)


@pytest.mark.parametrize("fmt,nan", [(E4M3, 0x7F), (E5M2, 0x7E)])
def test_nan_positions_must_agree(fmt, nan):
    ref = codes()
    ref[5] = nan
    got = ref.copy()
    check_codes(got, ref, fmt)
    got[5] = 0x70
    with pytest.raises(AssertionError, match="NaN"):
        check_codes(got, ref, fmt)


def test_e5m2_infinity_is_no_neighbour_of_the_maximum():
    ref = codes()
    ref[9], ref[10] = 0x7C, 0xFC         # +inf, -inf
    got = ref.copy()
    check_codes(got, ref, E5M2)
    got[9] = 0x7B                        # 57344 for +inf
    with pytest.raises(AssertionError, match="infinity"):
        check_codes(got, ref, E5M2)
    got = ref.copy()
    got[10] = 0x7C                       # +inf for -inf
    with pytest.raises(AssertionError, match="infinity"):
        check_codes(got, ref, E5M2)


def test_f16_one_ulp():
    ref = np.float16(np.linspace(-3, 3, 1001)).view(np.uint16)
    got = ref.copy()
    got[100] += 1
    check_f16(got, ref)
    got[200] += 2
    with pytest.raises(AssertionError, match="ulp"):
        check_f16(got, ref)
    got = ref.copy()
    got[300] = 0x7E00                    # NaN where the oracle has a value
    with pytest.raises(AssertionError, match="NaN"):
        check_f16(got, ref)


def test_master_relative():
    ref = np.float16([1.0, -2.0, 1000.0])
    got = ref.copy()
    got[2] = np.float16(1001.0)          # 1e-3 relative
    check_master(got.view(np.uint16), ref.view(np.uint16))
    got[2] = np.float16(1004.0)          # 4e-3 relative
    with pytest.raises(AssertionError, match="relative"):
        check_master(got.view(np.uint16), ref.view(np.uint16))


def test_f32_exact():
    ref = np.float32([1.0, np.nan, 3.5])
    check_f32_exact(ref.copy(), ref)
    got = ref.copy()
    got[2] = np.nextafter(np.float32(3.5), np.float32(4.0))
    with pytest.raises(AssertionError, match="bit-exact"):
        check_f32_exact(got, ref)
    got = ref.copy()
    got[1] = 0.0
    with pytest.raises(AssertionError, match="NaN"):
        check_f32_exact(got, ref)
