"""Pins of the exact-mode oracle (``oracle.exact_mode``) against facts fixed by
the page "det-train" (sections "Method" and "Correctness": the exact sum of the
products, rounded once to FP32; partials compose by adding digit arrays) and by
mathematics.

* ``pin_exact_closed_forms``  sums whose correctly rounded value is known in closed
                              form: cancellation across 2^200, ties to even, sticky
                              bits, FP32 overflow and its boundary, the subnormal
                              range, IEEE-754 special values;
* ``pin_exact_vs_rationals``  random products over a wide exponent range against
                              Python ``Fraction`` sums rounded by ``exact.round_rne``;
* ``pin_exact_rounding``      the integer rounding routine against ``exact.round_rne``
                              on values next to every kind of rounding boundary;
* ``pin_exact_headroom``      small-integer inputs, where every summation order is
                              exact: the exact mode equals the BF16 backward's dA and dB
                              (pinned by ``pins.pin_headroom_integers``);
* ``pin_exact_digits``        the digit layout (radix 2^32, digit i weighing
                              2^(32 i - 266), normalised) on closed-form sums;
* ``pin_exact_partition``     digit arrays of row shards, added in any grouping, equal
                              those of the whole; row order does not matter.

Each pin takes an ``ExactOracle`` and the C oracle (for dV) and raises
``AssertionError`` on a mismatch. The test suite also runs them against the
exact oracle's planted mistakes and requires that some pin fails for each.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import exact as ex
from deterministic_arithmetic_gb300 import synthetic as S

INF = math.inf


def _b(v) -> np.ndarray:
    return S.to_bf16_bits(np.asarray(v, np.float64))


def _f32bits(v) -> int:
    return int(np.asarray(v, np.float32).reshape(()).view(np.uint32))


def _want_bits(v) -> int:
    if isinstance(v, float) and math.isnan(v):
        return 0x7FC00000
    return _f32bits(np.float32(v))


def _same(name, got, want):
    g, w = _f32bits(got), _want_bits(want)
    if (w & 0x7F800000) == 0x7F800000 and (w & 0x7FFFFF):   # any NaN
        assert math.isnan(float(got)), f"{name}: {float(got)} is not NaN"
        return
    assert g == w, f"{name}: got {float(got)!r} ({g:#010x}), want {float(np.float32(want))!r} ({w:#010x})"


# products (a, b) -> value of the sum, rounded once
CLOSED_FORMS = [
    ("cancellation", [(2.0 ** 100, 1), (1, 1), (-(2.0 ** 100), 1)], 1.0),
    ("tiny survivor", [(2.0 ** 100, 1), (2.0 ** -100, 1), (-(2.0 ** 100), 1)], 2.0 ** -100),
    ("tie to even (down)", [(1, 1), (2.0 ** -24, 1)], 1.0),
    ("tie to even (up)", [(1, 1), (2.0 ** -23, 1), (2.0 ** -24, 1)], 1 + 2.0 ** -22),
    ("sticky bit", [(1, 1), (2.0 ** -24, 1), (2.0 ** -65, 2.0 ** -65)], 1 + 2.0 ** -23),
    ("negative tie", [(-1, 1), (-(2.0 ** -24), 1)], -1.0),
    ("FP32 overflow in between", [(2.0 ** 127, 1), (2.0 ** 127, 1), (-(2.0 ** 127), 1)], 2.0 ** 127),
    ("overflow", [(2.0 ** 127, 1), (2.0 ** 127, 1)], INF),
    ("max finite boundary (tie)", [(2.0 ** 127, 1), (2.0 ** 127, 1), (-(2.0 ** 103), 1)], INF),
    ("max finite", [(2.0 ** 127, 1), (2.0 ** 127, 1), (-(2.0 ** 103), 1), (-(2.0 ** -100), 1)],
     float(np.finfo(np.float32).max)),
    ("beyond any FP32 sum", [(2.0 ** 127, 2.0 ** 127)] * 2 + [(-(2.0 ** 127), 2.0 ** 127)] * 2 + [(1, 1)], 1.0),
    ("half the least subnormal", [(2.0 ** -75, 2.0 ** -75)], 0.0),
    ("least subnormal", [(2.0 ** -75, 2.0 ** -75)] * 2, 2.0 ** -149),
    ("subnormal tie up", [(2.0 ** -75, 2.0 ** -75)] * 3, 2.0 ** -148),
    ("subnormal below tie", [(2.0 ** -75, 2.0 ** -75)] * 3 + [(-(2.0 ** -100), 2.0 ** -100)], 2.0 ** -149),
    ("subnormal above half", [(2.0 ** -75, 2.0 ** -75), (2.0 ** -80, 2.0 ** -80)], 2.0 ** -149),
    ("negative to -0", [(-(2.0 ** -75), 2.0 ** -75)], -0.0),
    ("subnormal rounds to min normal", [(2.0 ** -63, 2.0 ** -63), (-(2.0 ** -75), 2.0 ** -75)], 2.0 ** -126),
    ("bf16 subnormal factors", [(2.0 ** -133, 2.0 ** -10), (3 * 2.0 ** -133, 2.0 ** -10)], 2.0 ** -141),
    ("exact zero", [(1, 1), (-1, 1)], 0.0),
    ("empty", [], 0.0),
    ("inf * 0", [(INF, 0), (1, 1)], math.nan),
    ("inf - inf", [(INF, 1), (-INF, 1)], math.nan),
    ("-inf", [(INF, -2), (1, 1), (2.0 ** 127, 2.0 ** 127)], -INF),
    ("inf * subnormal", [(INF, 2.0 ** -133)], INF),
    ("inf * inf", [(INF, INF), (-(2.0 ** 127), 2.0 ** 127)], INF),
    ("-inf * inf", [(-INF, INF)], -INF),
    ("NaN", [(math.nan, 1), (1, 1)], math.nan),
    ("NaN * 0", [(math.nan, 0)], math.nan),
]


def _pairs(products):
    if not products:
        return np.zeros((0, 1), np.uint16), np.zeros((0, 1), np.uint16)
    a = _b([[p[0]] for p in products])
    b = _b([[p[1]] for p in products])
    return a, b


def pin_exact_closed_forms(eo, o=None):
    for name, products, want in CLOSED_FORMS:
        a, b = _pairs(products)
        for bits, vals in ((a, [p[0] for p in products]), (b, [p[1] for p in products])):
            back = S.bf16_bits_to_f64(bits).ravel()
            assert all(float(x) == float(y) for x, y in zip(back, vals) if not math.isnan(float(y))), \
                f"{name}: a factor is not a BF16 value"
        _same(name, eo.exact_matmul(a, b)[0, 0], want)
        # the digit route gives the same value
        _same(name + " (digits)", eo.finalize(eo.digits(a, b))[0, 0], want)


def _rn32(q: Fraction) -> float:
    """exact.rn32 as a float, with the sign of zero IEEE-754 gives a negative value that
    rounds to zero (a Fraction has no -0)."""
    r = ex.rn32(q)
    if isinstance(r, float):
        return r
    if r == 0:
        return -0.0 if q < 0 else 0.0
    return float(ex.to_f32(r))


def _rational(bits):
    return ex.bf_value(int(bits))


def pin_exact_vs_rationals(eo, o=None, seed=31):
    rng = np.random.default_rng(seed)
    M, P, Q = 9, 3, 5
    # magnitudes over 2^-70 .. 2^70, some subnormal factors and exact zeros
    left = rng.standard_normal((M, P)) * np.exp2(rng.integers(-70, 70, (M, P)))
    right = rng.standard_normal((M, Q)) * np.exp2(rng.integers(-70, 70, (M, Q)))
    left[0, 0] = 2.0 ** -130
    right[1, 2] = 0.0
    lb, rb = _b(left), _b(right)
    got = eo.exact_matmul(lb, rb)
    for p in range(P):
        for q in range(Q):
            s = sum(_rational(lb[m, p]) * _rational(rb[m, q]) for m in range(M))
            _same(f"rationals[{p},{q}]", got[p, q], _rn32(s))
    # the sum of products spread over the whole BF16 range, and a tiny remainder of a cancellation
    big = _b([[2.0 ** 120], [2.0 ** -120], [-(2.0 ** 120)], [3 * 2.0 ** -60]])
    one = _b([[2.0 ** 7], [2.0 ** -9], [2.0 ** 7], [2.0 ** -70]])
    s = sum(_rational(big[m, 0]) * _rational(one[m, 0]) for m in range(4))
    _same("wide cancellation", eo.exact_matmul(big, one)[0, 0], _rn32(s))


def pin_exact_rounding(eo, o=None, seed=37):
    rng = np.random.default_rng(seed)
    vals = []
    for e in (-149, -140, -127, -126, -125, -1, 0, 1, 60, 126, 127):
        for ulp_off, odd in ((u, d) for u in (-1, 0, 1) for d in (0, 1)):
            # the midpoint between two FP32 neighbours at binary exponent e (the lower one even,
            # then odd), and the values just below and above it
            quantum = max(e, -126) - 23
            base = ((1 << 23 | 0x5A5A4) if e >= -126 else 0x2A4) + odd
            mid = (2 * base + 1) << (quantum + 266 - 1)
            vals.append(mid + ulp_off)
            vals.append(2 * base << (quantum + 266 - 1))       # exactly representable
            vals.append((2 * base + 2) << (quantum + 266 - 1))
    vals += [int(v) for v in rng.integers(1, 2 ** 62, 40)]
    vals += [int(rng.integers(1, 2 ** 60)) << int(rng.integers(0, 290)) for _ in range(60)]
    vals += [(1 << (128 + 266)) - (1 << (103 + 266)), (1 << (128 + 266)) - (1 << (103 + 266)) - 1]
    for v in vals:
        for s in (1, -1):
            _same(f"round({s * v})", eo.round_int(s * v), _rn32(Fraction(s * v, 1 << 266)))


def pin_exact_headroom(eo, o, seed=41):
    # small-integer values: every partial sum stays an integer below 2^24, so the BF16 backward's
    # dA and dB (tree-summed in FP32) are exact, and so is the exact mode
    rng = np.random.default_rng(seed)
    M, K, N, R = 40, 24, 16, 8
    x = _b(rng.integers(-8, 9, (M, K)))
    du = _b(rng.integers(-8, 9, (M, R)))
    u = _b(rng.integers(-8, 9, (M, R)))
    dy = _b(rng.integers(-8, 9, (M, N)))
    dv = o.dv(dy, 2.0)
    da, db = eo.grads(dv, x, u, du)
    want_da = o.da(du, x)
    want_db = o.db(dv, u)
    assert np.array_equal(da.view(np.uint32), want_da.view(np.uint32)), "headroom: dA"
    assert np.array_equal(db.view(np.uint32), want_db.view(np.uint32)), "headroom: dB"


def pin_exact_digits(eo, o=None):
    one = _b([[1.0]])
    d = eo.digits(one, one)[0, 0]
    want = [0] * 21
    want[8] = 1 << 10                       # 1 = 2^266 units of 2^-266: digit 8 weighs 2^256
    assert list(d) == want, f"digits of 1: {list(d)}"
    d = eo.digits(_b([[-1.0]]), one)[0, 0]
    want = [0] * 8 + [(1 << 32) - (1 << 10)] + [0xFFFFFFFF] * 8 + [-1, 0, 0, 0]
    assert list(d) == want, f"digits of -1: {list(d)}"
    d = eo.digits(_b([[2.0 ** -133]]), _b([[2.0 ** -133]]))[0, 0]   # the least product
    assert list(d) == [1] + [0] * 20, f"digits of 2^-266: {list(d)}"
    d = eo.digits(_b([[INF], [-INF], [math.nan], [INF]]), _b([[1.0], [1.0], [1.0], [0.0]]))[0, 0]
    assert list(d[18:]) == [1, 1, 2], f"counts: {list(d[18:])}"


def pin_exact_partition(eo, o=None, seed=43):
    rng = np.random.default_rng(seed)
    M, P, Q = 23, 2, 3
    left = _b(rng.standard_normal((M, P)) * np.exp2(rng.integers(-40, 40, (M, P))))
    right = _b(rng.standard_normal((M, Q)) * np.exp2(rng.integers(-40, 40, (M, Q))))
    whole = eo.digits(left, right)
    cuts = [0, 5, 6, 17, M]
    shards = [eo.digits(left[a:b], right[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    left_fold = shards[0].reshape(-1, 21)
    for s in shards[1:]:
        left_fold = eo.combine(left_fold, s)
    right_fold = shards[-1].reshape(-1, 21)
    for s in reversed(shards[:-1]):
        right_fold = eo.combine(s, right_fold)
    assert np.array_equal(left_fold.reshape(whole.shape), whole), "shards (left fold)"
    assert np.array_equal(right_fold.reshape(whole.shape), whole), "shards (right fold)"
    perm = rng.permutation(M)
    assert np.array_equal(eo.digits(left[perm], right[perm]), whole), "row permutation"
    got = eo.finalize(whole)
    want = eo.exact_matmul(left, right)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), "finalize"


EXACT_PINS = [pin_exact_closed_forms, pin_exact_vs_rationals, pin_exact_rounding, pin_exact_headroom,
              pin_exact_digits, pin_exact_partition]
