"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an ``oracle.oracle.Oracle`` and raises ``AssertionError``
when the oracle disagrees with:

* ``pin_golden``            hand-worked examples (tests/golden/worked_small.json);
* ``pin_rounding``          the IEEE-754 round-to-nearest-even definition, on exact rationals;
* ``pin_rational``          the whole operator computed with exact rationals and
                            correctly rounded at the pages' rounding points;
* ``pin_headroom_integers`` integer inputs where no partial sum can round (numpy int64 matmul);
* ``pin_permutation``       R = K, A a permutation matrix: U is X with permuted columns;
* ``pin_library_matmul``    dY_lora from a given U against numpy's binary64 matmul;
* ``pin_invariants``        B = 0, A = 0, linearity in alpha;
* ``pin_finite_differences`` the gradients against central differences of the scalar loss;
* ``pin_bf16_output``       the BF16 dY_lora variant: exact rationals rounded at its extra
                            rounding point, and constructed ties of round-to-nearest-even;
* ``pin_f32_dy``            the FP32-dY input variant's dV: exact rationals, and a value that
                            only two roundings (binary32, then bfloat16) send to the even side.

The test suite also runs every pin against builds of the oracle with a planted
mistake and requires that some pin fails for each.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

import exact as ex
from deterministic_arithmetic_gb300 import synthetic as S

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_small.json")


def _bits(values) -> np.ndarray:
    return S.to_bf16_bits(np.asarray(values, np.float64))


def _eq_bits(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{name}: shape {got.shape} != {want.shape}"
    if got.dtype == np.float32:
        # +0 and -0 are the same value
        g = got.view(np.uint32).copy(); w = want.astype(np.float32).view(np.uint32).copy()
        g[(g & 0x7FFFFFFF) == 0] = 0; w[(w & 0x7FFFFFFF) == 0] = 0
    else:
        g = got.astype(np.uint16).copy(); w = want.astype(np.uint16).copy()
        g[(g & 0x7FFF) == 0] = 0; w[(w & 0x7FFF) == 0] = 0
    bad = np.argwhere(g != w)
    assert bad.size == 0, f"{name}: {len(bad)} elements differ, first at {tuple(bad[0])}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


def _chain(o, x, a, b, dy, alpha):
    f = o.fwd(x, a, b, alpha)
    g = o.bwd(dy, x, a, b, f["u"], alpha)
    return {**f, **g}


# ----------------------------------------------------------------- golden
def pin_golden(o):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        x, a, b, dy = (_bits(c[k]) for k in ("x", "a", "b", "dy"))
        out = _chain(o, x, a, b, dy, c["alpha"])
        for key in ("u", "dv", "du"):
            _eq_bits(f"{c['name']}:{key}", out[key], _bits(c[key]))
        for key in ("delta_y", "db", "dx", "da"):
            _eq_bits(f"{c['name']}:{key}", out[key], np.asarray(c[key], np.float64).astype(np.float32))


# --------------------------------------------------------------- rounding
def pin_rounding(o):
    specials = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -8 + 2.0 ** -20,
                3.3895313892515355e38, 3.4028234663852886e38, 2.0 ** -130, 2.0 ** -133 * 3, 0.0, -0.0,
                1.9921875 + 2.0 ** -9, 255.5, 256.5, 257.0]
    rng = np.random.default_rng(7)
    rand = (rng.standard_normal(400) * np.exp2(rng.integers(-40, 40, 400))).astype(np.float32)
    for f in list(np.float32(specials)) + list(rand):
        want = ex.rnbf_of_f32(Fraction(float(f)))
        got = o.rnbf(float(f))
        if isinstance(want, float):   # overflow to infinity
            assert got == (0x7F80 if want > 0 else 0xFF80), (f, hex(got))
        else:
            w = ex.bf16_bits(want)
            assert (got & 0x7FFF or w & 0x7FFF) == 0 or got == w, (float(f), hex(got), hex(w))
    nan_in = np.array([0x7FA00001], np.uint32).view(np.float32)[0]
    nb = o.rnbf(float(nan_in))
    assert (nb & 0x7F80) == 0x7F80 and (nb & 0x7F) != 0, hex(nb)
    d64 = rng.standard_normal(400) * np.exp2(rng.integers(-60, 60, 400))
    d64 = np.concatenate([d64, [1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, 1 + 2.0 ** -24 + 2.0 ** -50]])
    for v in d64:
        want = ex.to_f32(ex.rn32(Fraction(float(v))))
        got = o.rn32(float(v))
        assert ex.f32_bits(got) == ex.f32_bits(want), (v, got, want)


# ------------------------------------------------------- exact rationals
def pin_rational(o, M=5, K=7, N=6, R=3, alpha=0.3, seed=11):
    w = S.Workload("rational", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": 0.4, "b": 0.6, "dy": 1.0})
    d = w.generate(seed)
    a32 = np.float32(alpha)
    want = ex.exact_chain(d["x"], d["a"], d["b"], d["dy"], a32)
    got = _chain(o, d["x"], d["a"], d["b"], d["dy"], float(a32))
    for key in ("u", "delta_y", "dv", "du", "db", "dx", "da"):
        _eq_bits(f"rational:{key}", got[key], want[key])


# ---------------------------------------- precision headroom (integers)
def _round_ints(vals, fmt):
    out = np.empty(vals.shape, np.float64)
    for idx, v in np.ndenumerate(vals):
        out[idx] = float(ex.round_rne(Fraction(int(v)), fmt))
    return out


def pin_headroom_integers(o, M=24, K=40, N=20, R=8, alpha=2.0, seed=3):
    """Integer inputs: every product and partial sum is an integer below 2^24,
    so FP32 accumulation is exact in any order and the only roundings left are
    the BF16 rounding points (page "[DSv4][P5-3] ...", sections "Summary" and
    "Agreement with the oracle")."""
    d = S.integers(M, K, N, R, alpha).generate(seed)
    X, A, B, DY = (S.bf16_bits_to_f64(d[k]).astype(np.int64) for k in ("x", "a", "b", "dy"))
    al = int(alpha)
    U = _round_ints(X @ A.T, ex.BFLOAT16).astype(np.int64)
    Y = (U @ B.T) * al
    DV = DY * al
    DU = _round_ints(DV @ B, ex.BFLOAT16).astype(np.int64)
    DB = DV.T @ U
    DX = DU @ A
    DA = DU.T @ X
    for T in (Y, DB, DX, DA):
        assert np.abs(T).max() < 2 ** 24
    got = _chain(o, d["x"], d["a"], d["b"], d["dy"], alpha)
    _eq_bits("ints:u", got["u"], _bits(U))
    _eq_bits("ints:dv", got["dv"], _bits(DV))
    _eq_bits("ints:du", got["du"], _bits(DU))
    for key, T in (("delta_y", Y), ("db", DB), ("dx", DX), ("da", DA)):
        _eq_bits(f"ints:{key}", got[key], T.astype(np.float32))


# --------------------------------------------- special cases / library
def pin_permutation(o, M=9, K=16, seed=5):
    """R = K and A a permutation matrix: U[m][r] = X[m][perm[r]] exactly."""
    d = S.Workload("perm", S.Shape(M, K, 4, K, 1.0), {"x": 1.0}).generate(seed, only=("x",))
    perm = np.random.default_rng(seed).permutation(K)
    A = np.zeros((K, K))
    A[np.arange(K), perm] = 1.0
    u = o.u(d["x"], _bits(A))
    _eq_bits("perm:u", u, d["x"][:, perm])


def pin_library_matmul(o, M=12, N=10, R=8, alpha=0.75, seed=9):
    """dY_lora from a given U against numpy's binary64 matmul: with R = 8 terms
    of 16-bit products the binary64 sum is exact in any order, so the FP32
    rounding then the FP32 multiply by alpha must match bit for bit."""
    w = S.Workload("lib", S.Shape(M, 4, N, R, alpha), {"b": 0.5})
    b = w.generate(seed, only=("b",))["b"]
    u = S.to_bf16_bits(S.normal_f64(seed, "x", M * R).reshape(M, R))
    Uf = S.bf16_bits_to_f64(u); Bf = S.bf16_bits_to_f64(b)
    want = ((Uf @ Bf.T).astype(np.float32) * np.float32(alpha)).astype(np.float32)
    _eq_bits("lib:delta_y", o.delta_y(u, b, alpha), want)
    # dX and dA against numpy as well (same exactness argument; M terms for dA)
    a = S.to_bf16_bits(S.normal_f64(seed, "a", R * 6).reshape(R, 6) * 0.5)
    du = u
    Af = S.bf16_bits_to_f64(a)
    _eq_bits("lib:dx", o.dx(du, a), (Uf @ Af).astype(np.float32))
    xs = S.to_bf16_bits(S.normal_f64(seed, "dy", M * 6).reshape(M, 6))
    _eq_bits("lib:da", o.da(du, xs), (Uf.T @ S.bf16_bits_to_f64(xs)).astype(np.float32))


# --------------------------------------------------------------- invariants
def pin_invariants(o, M=16, K=24, N=12, R=8, seed=21):
    d = S.Workload("inv", S.Shape(M, K, N, R, 1.0), {"x": 1.0, "a": 0.3, "b": 0.5, "dy": 1.0}).generate(seed)
    x, a, b, dy = d["x"], d["a"], d["b"], d["dy"]
    zb = np.zeros_like(b); za = np.zeros_like(a)
    # B = 0: the forward delta and every gradient that passes through B vanish; dB does not
    out = _chain(o, x, a, zb, dy, 2.0)
    for key in ("delta_y", "du", "dx", "da"):
        assert not np.any(S.bf16_bits_to_f64(out[key]) if out[key].dtype == np.uint16 else out[key]), f"B=0 -> {key} != 0"
    assert np.any(out["db"]), "B=0 but dB == 0"
    # A = 0: U = 0, dY_lora = 0, dB = 0
    out = _chain(o, x, za, b, dy, 2.0)
    assert not np.any(S.bf16_bits_to_f64(out["u"])) and not np.any(out["delta_y"]) and not np.any(out["db"]), "A=0"
    # linearity in alpha (powers of two scale exactly through every rounding)
    base = _chain(o, x, a, b, dy, 1.0)
    for al in (0.5, 2.0):
        out = _chain(o, x, a, b, dy, al)
        _eq_bits(f"alpha{al}:u", out["u"], base["u"])
        for key in ("delta_y", "db", "dx", "da"):
            _eq_bits(f"alpha{al}:{key}", out[key], (base[key] * np.float32(al)).astype(np.float32))
        for key in ("dv", "du"):
            _eq_bits(f"alpha{al}:{key}", out[key], _bits(S.bf16_bits_to_f64(base[key]) * al))


# -------------------------------------------------------- finite differences
def pin_finite_differences(o, M=6, K=10, N=7, R=3, seed=4):
    """Gradients of L(X, A, B) = alpha * sum(dY * ((X A^T) B^T)) by central
    differences in binary64. With small-integer inputs and alpha = 1 every
    rounding point is exact, so the oracle's dX, dA, dB must equal the
    derivative of L; L is linear in each single entry, so the central
    difference with step 1 is exact."""
    d = S.integers(M, K, N, R, 1.0, bound=2).generate(seed)
    X, A, B, DY = (S.bf16_bits_to_f64(d[k]) for k in ("x", "a", "b", "dy"))
    alpha = 1.0

    def L(X_, A_, B_):
        return alpha * float(np.sum(DY * ((X_ @ A_.T) @ B_.T)))

    def fd(T, which):
        g = np.zeros_like(T)
        for idx in np.ndindex(T.shape):
            P = T.copy(); P[idx] += 1.0
            Q = T.copy(); Q[idx] -= 1.0
            args_p = {"X": X, "A": A, "B": B}; args_q = dict(args_p)
            args_p[which] = P; args_q[which] = Q
            g[idx] = (L(args_p["X"], args_p["A"], args_p["B"]) - L(args_q["X"], args_q["A"], args_q["B"])) / 2.0
        return g

    out = _chain(o, d["x"], d["a"], d["b"], d["dy"], alpha)
    # U must be exact for L's gradient to be the oracle's (|U| <= 256 here)
    assert np.array_equal(S.bf16_bits_to_f64(out["u"]), X @ A.T)
    assert np.array_equal(S.bf16_bits_to_f64(out["du"]), (DY * alpha) @ B)
    np.testing.assert_array_equal(out["da"].astype(np.float64), fd(A, "A"))
    np.testing.assert_array_equal(out["db"].astype(np.float64), fd(B, "B"))
    np.testing.assert_array_equal(out["dx"].astype(np.float64), fd(X, "X"))


# ------------------------------------------------------ BF16 output variant
def pin_bf16_output(o, seed=13):
    # (1) the whole forward with exact rationals, correctly rounded at U, at the FP32 result and
    # then once more to BF16
    w = S.Workload("rational_bf16", S.Shape(5, 7, 6, 3, 0.3), {"x": 1.0, "a": 0.4, "b": 0.6, "dy": 1.0})
    d = w.generate(seed)
    a32 = np.float32(0.3)
    want = ex.exact_chain(d["x"], d["a"], d["b"], d["dy"], a32)
    got = o.delta_y_bf16(o.u(d["x"], d["a"]), d["b"], float(a32))
    exp = np.empty(want["delta_y"].shape, np.uint16)
    for idx, v in np.ndenumerate(want["delta_y"]):
        q = ex.rnbf_of_f32(Fraction(float(v)))
        exp[idx] = (0x7F80 if q > 0 else 0xFF80) if isinstance(q, float) else ex.bf16_bits(q)
    _eq_bits("bf16_output:rational", got, exp)
    # (2) sums placed exactly on and next to BF16 midpoints (alpha = 1, every product exact):
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 and goes to the even 1; 1 + 3*2^-8 goes up to
    # 1 + 2^-6; just above a midpoint goes up; the signs mirror
    u = _bits([[1.0, 2.0 ** -8, 2.0 ** -20, 0, 0, 0, 0, 0]])
    b = _bits([[1, 1, 0, 0, 0, 0, 0, 0],          # 1 + 2^-8           -> 1
               [1, 3, 0, 0, 0, 0, 0, 0],          # 1 + 3 * 2^-8       -> 1 + 2^-6
               [1, 1, 1, 0, 0, 0, 0, 0],          # 1 + 2^-8 + 2^-20   -> 1 + 2^-7
               [-1, -1, 0, 0, 0, 0, 0, 0],        # -(1 + 2^-8)        -> -1
               [-1, -3, 0, 0, 0, 0, 0, 0],        # -(1 + 3 * 2^-8)    -> -(1 + 2^-6)
               [1, -1, 0, 0, 0, 0, 0, 0]])        # 1 - 2^-8 (exact)   -> 1 - 2^-8
    got = o.delta_y_bf16(u, b, 1.0)
    _eq_bits("bf16_output:midpoints", got, _bits([[1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -1.0,
                                                   -(1.0 + 2.0 ** -6), 1.0 - 2.0 ** -8]]))


# ------------------------------------------------------ FP32-dY input variant
def pin_f32_dy(o, seed=17):
    # (1) exact rationals: dV = rnbf(rn32(dy * alpha)) for binary32 dy of every magnitude
    rng = np.random.default_rng(seed)
    dy = (rng.standard_normal((6, 40)) * np.exp2(rng.integers(-30, 30, (6, 40)))).astype(np.float32)
    for alpha in (0.3, 2.0, -1.5):
        a32 = np.float32(alpha)
        got = o.dv_f32(dy, float(a32))
        exp = np.empty(dy.shape, np.uint16)
        for idx, v in np.ndenumerate(dy):
            q32 = ex.rn32(Fraction(float(v)) * Fraction(float(a32)))
            q = ex.rnbf_of_f32(Fraction(float(ex.to_f32(q32))) if not isinstance(q32, float) else q32)
            exp[idx] = (0x7F80 if q > 0 else 0xFF80) if isinstance(q, float) else ex.bf16_bits(q)
        _eq_bits(f"f32_dy:alpha={alpha}", got, exp)
    # (2) two roundings, not one: (1 + 2^-8 + 2^-23) * (1 - 2^-24) lies just above the BF16
    # midpoint 1 + 2^-8 but rounds to it in binary32, so the BF16 result is the even 1;
    # 1 + 3 * 2^-8 is a midpoint already and goes up; a value past the binary32 range is infinite
    dy2 = np.array([[1 + 2.0 ** -8 + 2.0 ** -23, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.0e38]], np.float32)
    got = o.dv_f32(dy2[:, :3], float(np.float32(1 - 2.0 ** -24)))
    _eq_bits("f32_dy:double rounding", got[:, :1], _bits([[1.0]]))
    got = o.dv_f32(dy2, 1.0)
    assert got[0, 1] == _bits([[1 + 2.0 ** -6]])[0, 0] and got[0, 2] == _bits([[-1.0]])[0, 0], got
    assert o.dv_f32(dy2[:, 3:], 2.0)[0, 0] == 0x7F80


ALL_PINS = [pin_golden, pin_rounding, pin_rational, pin_headroom_integers, pin_permutation,
            pin_library_matmul, pin_invariants, pin_finite_differences, pin_bf16_output, pin_f32_dy]
