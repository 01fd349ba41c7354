"""Exact rational arithmetic used to pin the oracle (tests only).

Independent of the oracle's C code: values are Python ``Fraction`` objects and
rounding to a binary format is written here from the IEEE-754 definition of
round-to-nearest, ties-to-even, on exact rationals.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

import numpy as np

# (significand bits incl. the implicit one, minimum normal exponent, maximum exponent)
BINARY32 = (24, -126, 127)
BFLOAT16 = (8, -126, 127)


def round_rne(q: Fraction, fmt) -> Fraction | float:
    """Round the exact rational ``q`` to the nearest value of format ``fmt``
    (ties to even). Returns a Fraction, or +/-inf on overflow."""
    p, emin, emax = fmt
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)                       # below the normal range the quantum stays fixed
    quantum = Fraction(2) ** (e - p + 1)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * quantum
    largest = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if r > largest:
        return sign * math.inf
    return sign * r


def f32_bits(v) -> int:
    return struct.unpack("<I", struct.pack("<f", float(v)))[0]


def to_f32(q) -> np.float32:
    """Exact conversion of a value already representable in binary32."""
    if isinstance(q, float) and math.isinf(q):
        return np.float32(q)
    f = np.float32(float(q))
    assert Fraction(float(f)) == q, "value not representable in binary32"
    return f


def bf16_bits(q) -> int:
    """Bit pattern of a value already representable in bfloat16."""
    f = to_f32(q)
    bits = f32_bits(f)
    assert bits & 0xFFFF == 0, "value not representable in bfloat16"
    return bits >> 16


def bf_value(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))


def rn32(q: Fraction):
    return round_rne(q, BINARY32)


def rnbf_of_f32(q):
    """bfloat16 rounding of a binary32 value (as a Fraction)."""
    return round_rne(q, BFLOAT16)


# ------------------------------------------------- the operator, exactly
def exact_chain(x, a, b, dy, alpha32: np.float32):
    """The operator of page "[DSv4][P5-3] shared_grouped_lora_delta ...",
    section "Summary", with exact sums and correctly rounded results at each
    rounding point. Inputs are bf16 bit-pattern arrays; returns bit patterns
    (bf16 outputs) and float32 arrays (FP32 outputs)."""
    M, K = x.shape
    R = a.shape[0]
    N = b.shape[0]
    X = [[bf_value(int(v)) for v in row] for row in x]
    A = [[bf_value(int(v)) for v in row] for row in a]
    B = [[bf_value(int(v)) for v in row] for row in b]
    DY = [[bf_value(int(v)) for v in row] for row in dy]
    al = Fraction(float(alpha32))

    U = [[rnbf_of_f32(rn32(sum(X[m][k] * A[r][k] for k in range(K)))) for r in range(R)] for m in range(M)]
    Y = [[rn32(rn32(sum(U[m][r] * B[n][r] for r in range(R))) * al) for n in range(N)] for m in range(M)]
    DV = [[rnbf_of_f32(rn32(DY[m][n] * al)) for n in range(N)] for m in range(M)]
    DU = [[rnbf_of_f32(rn32(sum(DV[m][n] * B[n][r] for n in range(N)))) for r in range(R)] for m in range(M)]
    DB = [[rn32(sum(DV[m][n] * U[m][r] for m in range(M))) for r in range(R)] for n in range(N)]
    DX = [[rn32(sum(DU[m][r] * A[r][k] for r in range(R))) for k in range(K)] for m in range(M)]
    DA = [[rn32(sum(DU[m][r] * X[m][k] for m in range(M))) for k in range(K)] for r in range(R)]

    def bits(T):
        return np.array([[bf16_bits(v) for v in row] for row in T], np.uint16)

    def f32(T):
        return np.array([[to_f32(v) for v in row] for row in T], np.float32)

    return dict(u=bits(U), delta_y=f32(Y), dv=bits(DV), du=bits(DU), db=f32(DB), dx=f32(DX), da=f32(DA))
