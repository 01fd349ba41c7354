"""CPU oracle of the exact mode of the weight gradients.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs are the only callers.
It shares nothing with the CUDA library.

What it computes (page "det-train", sections "Method" and "API": every GEMM
output is the exact sum of its products -- each BF16 product is exact -- kept as
a long accumulator of int64 digits in radix 2^32 and rounded once to FP32)::

    dA[r][k] = rn32( sum_m du[m][r] * x[m][k] )
    dB[n][r] = rn32( sum_m dv[m][n] * u[m][r] ),   dv = bf16(fp32(dy * alpha))

Here the sums are Python integers: a finite BF16 value is m * 2^s with an
integer m, so the sum of products is an integer multiple of 2^-266 (the
smallest product unit) and is formed exactly; rn32 is round to nearest, ties to
even, written out below on that integer. dV comes from the C oracle (the BF16
backward's dV). Products with an infinite or NaN factor follow IEEE-754:
inf * 0 and NaN factors give NaN, and the result is NaN when a NaN product or
infinite products of both signs occur, else the infinity. An exact zero sum
gives +0.

Digit arrays (the composable form): 21 int64 per output -- 18 digits in radix
2^32, digit i weighing 2^(32 i - 266), written normalised (digits 0..16 in
[0, 2^32), digit 17 the signed rest), then the counts of +inf, -inf and NaN
products. The page does not give the number of digits: 18 cover every sum of
fewer than 2^31 BF16 products.

``ExactOracle(mutant=n)`` plants mistake n (tests only) so the test suite can
show that the pins of this module catch it.
"""
from __future__ import annotations

import math

import numpy as np

DIGITS = 18
SLOTS = DIGITS + 3
BASE = 266                 # a sum is an integer number of units of 2^-266
F32_MAX = float(np.finfo(np.float32).max)
N_MUTANTS = 3              # 1: ties away from zero; 2: no subnormal quantum; 3: inf * 0 dropped


def decode(bits: np.ndarray):
    """BF16 bit patterns -> (m, s, kind): value m * 2^s for finite values
    (kind 0), kind +1 / -1 for +inf / -inf, 2 for NaN (IEEE-754 binary16-bf
    layout: 1 sign, 8 exponent, 7 fraction bits, bias 127)."""
    b = np.asarray(bits, np.int64)
    sign = np.where(b & 0x8000, -1, 1)
    e = (b >> 7) & 0xFF
    f = b & 0x7F
    m = sign * np.where(e > 0, f | 0x80, f)            # normal: 1.f; subnormal: 0.f
    s = np.where(e > 0, e, 1) - 127 - 7
    kind = np.where(e == 0xFF, np.where(f != 0, 2, sign), 0)
    m = np.where(kind != 0, 0, m)
    return m, s, kind


class ExactOracle:
    def __init__(self, mutant: int = 0):
        self.mutant = int(mutant)

    # ---------------------------------------------------------- the sums
    def sums(self, left: np.ndarray, right: np.ndarray):
        """sum_m left[m][p] * right[m][q], exactly: returns (V, pinf, ninf, nan) with
        V[p][q] a Python int (value V * 2^-266) and the special-product counts."""
        left = np.asarray(left, np.uint16)
        right = np.asarray(right, np.uint16)
        M, P = left.shape
        M2, Q = right.shape
        assert M == M2
        lm, ls, lk = decode(left)
        rm, rs, rk = decode(right)
        V = [[0] * Q for _ in range(P)]
        cnt = np.zeros((3, P, Q), np.int64)
        npos = 2 * 127 + 2 * 7 + BASE                      # largest position + 1 (507)
        for p in range(P):
            finite = (lk[:, p, None] == 0) & (rk == 0)
            mm = lm[:, p, None] * rm                       # |mm| < 2^16, exact
            pos = ls[:, p, None] + rs + BASE               # in [0, 506]
            # bucket the products by position; every bucket sum is an integer below 2^53
            # in magnitude, so the binary64 accumulation of bincount is exact
            qi = np.broadcast_to(np.arange(Q)[None, :], mm.shape)
            sel = finite & (mm != 0)
            buckets = np.bincount((qi[sel] * npos + pos[sel]), weights=mm[sel].astype(np.float64),
                                  minlength=Q * npos).reshape(Q, npos)
            for q in range(Q):
                nz = np.flatnonzero(buckets[q])
                V[p][q] = sum(int(buckets[q, i]) << int(i) for i in nz)
            # products with an infinite or NaN factor
            special = ~finite
            lz = (lk[:, p, None] == 0) & (lm[:, p, None] == 0)       # left factor is zero
            rz = (rk == 0) & (rm == 0)
            nanp = special & ((lk[:, p, None] == 2) | (rk == 2) | lz | rz)
            if self.mutant == 3:                                     # inf * 0 dropped
                nanp = special & ((lk[:, p, None] == 2) | (rk == 2))
                special = special & ~(lz | rz)
            sl = np.where(lk[:, p, None] == 0, np.sign(lm[:, p, None]), lk[:, p, None])
            sr = np.where(rk == 0, np.sign(rm), rk)
            infp = special & ~nanp
            sgn = sl * sr
            cnt[0, p] = (infp & (sgn > 0)).sum(axis=0)
            cnt[1, p] = (infp & (sgn < 0)).sum(axis=0)
            cnt[2, p] = nanp.sum(axis=0)
        return V, cnt[0], cnt[1], cnt[2]

    # -------------------------------------------------------- rounding
    def round_int(self, V: int) -> np.float32:
        """V * 2^-266 rounded to the nearest binary32, ties to even; +0 for 0; +-inf
        beyond the largest finite value (IEEE-754 round to nearest)."""
        if V == 0:
            return np.float32(0.0)
        neg = V < 0
        a = -V if neg else V
        e = a.bit_length() - 1 - BASE                     # 2^e <= |value| < 2^(e+1)
        qe = (max(e, -126) if self.mutant != 2 else e) - 23   # exponent of the last kept bit
        shift = qe + BASE                                 # the same, in units of 2^-266
        if shift <= 0:
            n = a << -shift
        else:
            n = a >> shift
            rem = a - (n << shift)
            half = 1 << (shift - 1)
            if rem > half or (rem == half and (n & 1 or self.mutant == 1)):
                n += 1
        v = math.ldexp(n, qe)                             # exact: n < 2^25
        if v > F32_MAX:
            v = math.inf
        return np.float32(-v if neg else v)

    def result(self, V: int, pinf: int, ninf: int, nan: int) -> np.float32:
        if nan or (pinf and ninf):
            return np.float32(np.nan)
        if pinf:
            return np.float32(np.inf)
        if ninf:
            return np.float32(-np.inf)
        return self.round_int(V)

    def exact_matmul(self, left, right, transpose=False):
        """rn32 of the exact sums as an FP32 array [P][Q] (or [Q][P])."""
        V, pinf, ninf, nan = self.sums(left, right)
        P, Q = pinf.shape
        out = np.empty((P, Q), np.float32)
        for p in range(P):
            for q in range(Q):
                out[p, q] = self.result(V[p][q], pinf[p, q], ninf[p, q], nan[p, q])
        return out.T.copy() if transpose else out

    # ---------------------------------------------------- digit arrays
    @staticmethod
    def to_digits(V: int, pinf: int, ninf: int, nan: int) -> list[int]:
        """Normalised digit array of V * 2^-266 and the counts."""
        d = [(V >> (32 * i)) & 0xFFFFFFFF for i in range(DIGITS - 1)]
        d.append(V >> (32 * (DIGITS - 1)))                # floor: the signed rest
        return d + [int(pinf), int(ninf), int(nan)]

    @staticmethod
    def from_digits(d) -> tuple[int, int, int, int]:
        """Value and counts of a digit array, normalised or not."""
        V = sum(int(d[i]) << (32 * i) for i in range(DIGITS))
        return V, int(d[DIGITS]), int(d[DIGITS + 1]), int(d[DIGITS + 2])

    def digits(self, left, right, transpose=False) -> np.ndarray:
        """int64 digit arrays [P][Q][21] (or [Q][P][21])."""
        V, pinf, ninf, nan = self.sums(left, right)
        P, Q = pinf.shape
        out = np.empty((P, Q, SLOTS), np.int64)
        for p in range(P):
            for q in range(Q):
                out[p, q] = self.to_digits(V[p][q], pinf[p, q], ninf[p, q], nan[p, q])
        return out.transpose(1, 0, 2).copy() if transpose else out

    def combine(self, a, b) -> np.ndarray:
        """Digit arrays of the sums of two digit arrays (element by element)."""
        a = np.asarray(a, np.int64).reshape(-1, SLOTS)
        b = np.asarray(b, np.int64).reshape(-1, SLOTS)
        out = np.empty_like(a)
        for i in range(a.shape[0]):
            va, pa, na, qa = self.from_digits(a[i])
            vb, pb, nb, qb = self.from_digits(b[i])
            out[i] = self.to_digits(va + vb, pa + pb, na + nb, qa + qb)
        return out

    def finalize(self, d) -> np.ndarray:
        d = np.asarray(d, np.int64)
        flat = d.reshape(-1, SLOTS)
        out = np.array([self.result(*self.from_digits(row)) for row in flat], np.float32)
        return out.reshape(d.shape[:-1])

    # ------------------------------------------------ the two gradients
    def grads(self, dv, x, u, du):
        """(dA [R][K], dB [N][R]) in FP32 from dV (bf16 bits, already formed), x, u, du."""
        da = self.exact_matmul(du, x)
        db = self.exact_matmul(u, dv, transpose=True)
        return da, db
