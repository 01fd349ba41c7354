"""The tolerance helpers of the GPU parity tests, checked on the CPU.

* ``bf16_bits_rne`` (binary64 -> bfloat16, one rounding to nearest even)
  against the exact-rational rounding of ``tests/exact.py``, at random values
  and next to every kind of boundary (ties both ways, the subnormal range and
  its edge, overflow);
* ``assert_bf16_close`` accepts exactly what the precision contract allows:
  1 BF16 ulp from the oracle, or the BF16 image of the FP32 band where a sum
  cancels; a value 2 ulps away is rejected where the band is narrow (an
  ordinary element whose FP32 value sits next to a BF16 midpoint).
"""
from fractions import Fraction

import numpy as np
import pytest

import exact as ex
import gpu_util as G


def _ref_bits(v: float) -> int:
    r = ex.round_rne(Fraction(v), ex.BFLOAT16)
    if isinstance(r, float):                      # overflow
        return 0x7F80 if r > 0 else 0xFF80
    if r == 0:
        return 0x8000 if np.signbit(v) else 0
    return ex.bf16_bits(r)


def _edge_values():
    vals = [0.0, -0.0, 1.0, -1.0, 3.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40,
            1.0 + 2.0 ** -8 - 2.0 ** -40, 2.0 ** -126, 2.0 ** -127, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135,
            2.0 ** -134 + 2.0 ** -160, 2.0 ** -135, (2 - 2.0 ** -8) * 2.0 ** -126, (2 - 2.0 ** -9) * 2.0 ** -127,
            (2 - 2.0 ** -7) * 2.0 ** 127, (2 - 2.0 ** -8) * 2.0 ** 127, (2 - 2.0 ** -8) * 2.0 ** 127 - 2.0 ** 100,
            2.0 ** 128, 1e300, -1e300, 1e-300]
    return vals + [-v for v in vals]


def test_bf16_rounding_of_binary64_matches_exact_rationals():
    rng = np.random.default_rng(0)
    vals = _edge_values()
    vals += list(rng.standard_normal(2000) * np.exp2(rng.integers(-140, 130, 2000)))
    # values whose low bits put them exactly on, or one binary64 step beside, a bfloat16 midpoint
    mids = (rng.integers(128, 256, 500) * 2 + 1).astype(np.float64) * np.exp2(rng.integers(-130, 110, 500) - 9)
    vals += list(mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, np.inf))
    got = G.bf16_bits_rne(np.array(vals))
    want = np.array([_ref_bits(float(v)) for v in vals], np.uint16)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{len(bad)} values rounded differently, e.g. {vals[bad[0]]!r}: " \
                          f"{got[bad[0]]:#06x} vs {want[bad[0]]:#06x}"


def _bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0] >> 16)


def test_two_ulps_rejected_where_the_band_is_narrow():
    # ordinary element: S = |f|, FP32 value just above the midpoint between 1 and 1 + 2^-7
    f = np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)
    ref = np.array([_bits(1.0 + 2.0 ** -7)], np.uint16)          # the oracle's BF16 value
    s = np.array([abs(float(f))])
    fa = np.array([f])
    for k in (-1, 0, 1):                                         # within 1 ulp: accepted
        G.assert_bf16_close("near", ref + np.uint16(k) if k >= 0 else ref - np.uint16(1), ref, fa, s)
    with pytest.raises(AssertionError):
        G.assert_bf16_close("two ulps", ref + np.uint16(2), ref, fa, s)
    with pytest.raises(AssertionError):
        G.assert_bf16_close("two ulps below", ref - np.uint16(2), ref, fa, s)


def test_band_admits_cancelled_sums_only_within_its_image():
    # a sum that cancels: |f| much smaller than S, so 1e-6 * S spans many BF16 ulps of f
    f = np.float32(3.0e-4)
    s = np.array([1.0e3])                                        # band half-width 1e-3 > f itself
    ref = np.array([_bits(float(f))], np.uint16)
    fa = np.array([f])
    lo = G.bf16_bits_rne(np.array([float(f) - 1e-3]))[0]
    hi = G.bf16_bits_rne(np.array([float(f) + 1e-3]))[0]
    assert G.assert_bf16_close("band lo", np.array([lo]), ref, fa, s) == 1
    assert G.assert_bf16_close("band hi", np.array([hi]), ref, fa, s) == 1
    outside = G.bf16_bits_rne(np.array([float(f) + 1.2e-3]))
    with pytest.raises(AssertionError):
        G.assert_bf16_close("outside", outside, ref, fa, s)
