"""CPU oracle for the batch-invariant shared LoRA delta operator (Python side).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers. The product path never imports this module.

This is a thin ctypes wrapper around ``lora_oracle.c`` (built here by
``build()``); every step of the operator, and all of its arithmetic, lives in
that C file. Arrays cross the boundary as numpy ``uint16`` (bfloat16 bit
patterns), ``float32`` and ``float64``; nothing here imports the CUDA package.

Operator (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
batch-invariant", section "Summary")::

    U  = bf16(X @ A^T)            dY_lora = (U @ B^T) * alpha   (FP32)
    dV = bf16(dY * alpha)         dU = bf16(dV @ B)
    dB = dV^T @ U                 dX = dU @ A          dA = dU^T @ X
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lora_oracle.c")
LIB = os.path.join(HERE, "liblora_oracle.so")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(out: str = LIB, mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with the host C compiler. ``mutant`` > 0 plants the
    numbered mistake (tests only)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, *CFLAGS, f"-DORACLE_MUTANT={int(mutant)}", "-o", out + ".tmp", SRC, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _p(arr, ptype):
    if arr is None:
        return ctypes.cast(None, ptype)
    return arr.ctypes.data_as(ptype)


@dataclass
class Oracle:
    """Handle on one build of the oracle library (the real one, or a mutant)."""

    lib: ctypes.CDLL
    threads: int = 0

    @classmethod
    def load(cls, path: str | None = None, threads: int = 0) -> "Oracle":
        path = path or build()
        lib = ctypes.CDLL(path)
        sigs = {
            "ora_u": [_u16p, _u16p, _i64, _i64, _i64, _u16p, _f32p, _f64p, ctypes.c_int],
            "ora_delta_y": [_u16p, _u16p, ctypes.c_float, _i64, _i64, _i64, _f32p, _f64p, ctypes.c_int],
            "ora_delta_y_bf16": [_u16p, _u16p, ctypes.c_float, _i64, _i64, _i64, _u16p, ctypes.c_int],
            "ora_dv": [_u16p, ctypes.c_float, _i64, _i64, _u16p],
            "ora_dv_f32": [_f32p, ctypes.c_float, _i64, _i64, _u16p],
            "ora_du": [_u16p, _u16p, _i64, _i64, _i64, _u16p, _f32p, _f64p, ctypes.c_int],
            "ora_db": [_u16p, _u16p, _i64, _i64, _i64, _f32p, _f64p, ctypes.c_int],
            "ora_dx": [_u16p, _u16p, _i64, _i64, _i64, _f32p, _f64p, ctypes.c_int],
            "ora_da": [_u16p, _u16p, _i64, _i64, _i64, _f32p, _f64p, ctypes.c_int],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.ora_rn32.argtypes = [ctypes.c_double]
        lib.ora_rn32.restype = ctypes.c_float
        lib.ora_rnbf.argtypes = [ctypes.c_float]
        lib.ora_rnbf.restype = ctypes.c_uint16
        lib.ora_mutant.restype = ctypes.c_int
        lib.ora_threads.argtypes = [ctypes.c_int]
        lib.ora_threads.restype = ctypes.c_int
        return cls(lib, threads)

    @property
    def n_threads(self) -> int:
        return int(self.lib.ora_threads(self.threads))

    # ---------------------------------------------------------------- steps
    @staticmethod
    def _c(a, dtype):
        a = np.ascontiguousarray(a)
        assert a.dtype == dtype, (a.dtype, dtype)
        return a

    def u(self, x, a, want_s=False, want_f32=False):
        """U (bf16 bits); with want_s also S = sum|x a|; with want_f32 also the
        FP32 value before the BF16 rounding."""
        x = self._c(x, np.uint16); a = self._c(a, np.uint16)
        M, K = x.shape; R = a.shape[0]
        assert a.shape == (R, K)
        u = np.empty((M, R), np.uint16)
        s = np.empty((M, R), np.float64) if want_s else None
        f = np.empty((M, R), np.float32) if want_f32 else None
        rc = self.lib.ora_u(_p(x, _u16p), _p(a, _u16p), M, K, R, _p(u, _u16p), _p(f, _f32p), _p(s, _f64p), self.threads)
        assert rc == 0
        return (u,) + ((s,) if want_s else ()) + ((f,) if want_f32 else ()) if (want_s or want_f32) else u

    def delta_y(self, u, b, alpha, want_s=False):
        u = self._c(u, np.uint16); b = self._c(b, np.uint16)
        M, R = u.shape; N = b.shape[0]
        assert b.shape == (N, R)
        y = np.empty((M, N), np.float32)
        s = np.empty((M, N), np.float64) if want_s else None
        rc = self.lib.ora_delta_y(_p(u, _u16p), _p(b, _u16p), float(alpha), M, N, R, _p(y, _f32p), _p(s, _f64p), self.threads)
        assert rc == 0
        return (y, s) if want_s else y

    def delta_y_bf16(self, u, b, alpha):
        """The BF16 output variant: delta_y rounded to bfloat16 (bits)."""
        u = self._c(u, np.uint16); b = self._c(b, np.uint16)
        M, R = u.shape; N = b.shape[0]
        assert b.shape == (N, R)
        y = np.empty((M, N), np.uint16)
        rc = self.lib.ora_delta_y_bf16(_p(u, _u16p), _p(b, _u16p), float(alpha), M, N, R, _p(y, _u16p), self.threads)
        assert rc == 0
        return y

    def dv(self, dy, alpha):
        dy = self._c(dy, np.uint16)
        M, N = dy.shape
        dv = np.empty((M, N), np.uint16)
        assert self.lib.ora_dv(_p(dy, _u16p), float(alpha), M, N, _p(dv, _u16p)) == 0
        return dv

    def dv_f32(self, dy, alpha):
        """dV (bf16 bits) of the FP32-dY input variant: rnbf(rn32(dy * alpha))."""
        dy = self._c(dy, np.float32)
        M, N = dy.shape
        dv = np.empty((M, N), np.uint16)
        assert self.lib.ora_dv_f32(_p(dy, _f32p), float(alpha), M, N, _p(dv, _u16p)) == 0
        return dv

    def du(self, dv, b, want_s=False, want_f32=False):
        """dU (bf16 bits); optionally S and the FP32 value before rounding."""
        dv = self._c(dv, np.uint16); b = self._c(b, np.uint16)
        M, N = dv.shape; R = b.shape[1]
        assert b.shape == (N, R)
        du = np.empty((M, R), np.uint16)
        s = np.empty((M, R), np.float64) if want_s else None
        f = np.empty((M, R), np.float32) if want_f32 else None
        assert self.lib.ora_du(_p(dv, _u16p), _p(b, _u16p), M, N, R, _p(du, _u16p), _p(f, _f32p), _p(s, _f64p),
                               self.threads) == 0
        return (du,) + ((s,) if want_s else ()) + ((f,) if want_f32 else ()) if (want_s or want_f32) else du

    def db(self, dv, u, want_s=False):
        dv = self._c(dv, np.uint16); u = self._c(u, np.uint16)
        M, N = dv.shape; R = u.shape[1]
        assert u.shape == (M, R)
        db = np.empty((N, R), np.float32)
        s = np.empty((N, R), np.float64) if want_s else None
        assert self.lib.ora_db(_p(dv, _u16p), _p(u, _u16p), M, N, R, _p(db, _f32p), _p(s, _f64p), self.threads) == 0
        return (db, s) if want_s else db

    def dx(self, du, a, want_s=False):
        du = self._c(du, np.uint16); a = self._c(a, np.uint16)
        M, R = du.shape; K = a.shape[1]
        assert a.shape == (R, K)
        dx = np.empty((M, K), np.float32)
        s = np.empty((M, K), np.float64) if want_s else None
        assert self.lib.ora_dx(_p(du, _u16p), _p(a, _u16p), M, K, R, _p(dx, _f32p), _p(s, _f64p), self.threads) == 0
        return (dx, s) if want_s else dx

    def da(self, du, x, want_s=False):
        du = self._c(du, np.uint16); x = self._c(x, np.uint16)
        M, R = du.shape; K = x.shape[1]
        assert x.shape == (M, K)
        da = np.empty((R, K), np.float32)
        s = np.empty((R, K), np.float64) if want_s else None
        assert self.lib.ora_da(_p(du, _u16p), _p(x, _u16p), M, K, R, _p(da, _f32p), _p(s, _f64p), self.threads) == 0
        return (da, s) if want_s else da

    # ---------------------------------------------------------- the chains
    def fwd(self, x, a, b, alpha, want_s=False):
        """Forward chain: returns dict(u, delta_y[, s_u, s_y])."""
        if want_s:
            u, s_u = self.u(x, a, True)
            y, s_y = self.delta_y(u, b, alpha, True)
            return dict(u=u, delta_y=y, s_u=s_u, s_y=s_y)
        u = self.u(x, a)
        return dict(u=u, delta_y=self.delta_y(u, b, alpha))

    def bwd(self, dy, x, a, b, u, alpha, du_in=None, want_s=False):
        """Backward chain. ``u`` is the saved forward U. When ``du_in`` is given,
        dX and dA are fed that dU (per-GEMM mode) instead of the oracle's own."""
        dv = self.dv(dy, alpha)
        out = dict(dv=dv)
        if want_s:
            out["du"], out["s_du"] = self.du(dv, b, True)
            out["db"], out["s_db"] = self.db(dv, u, True)
            du_use = out["du"] if du_in is None else du_in
            out["dx"], out["s_dx"] = self.dx(du_use, a, True)
            out["da"], out["s_da"] = self.da(du_use, x, True)
        else:
            out["du"] = self.du(dv, b)
            out["db"] = self.db(dv, u)
            du_use = out["du"] if du_in is None else du_in
            out["dx"] = self.dx(du_use, a)
            out["da"] = self.da(du_use, x)
        return out

    def rn32(self, v: float) -> np.float32:
        return np.float32(self.lib.ora_rn32(float(v)))

    def rnbf(self, f: float) -> int:
        return int(self.lib.ora_rnbf(float(f)))

    @property
    def mutant(self) -> int:
        return int(self.lib.ora_mutant())


_default: Oracle | None = None


def get(threads: int = 0) -> Oracle:
    """The (lazily built) real oracle."""
    global _default
    if _default is None or _default.threads != threads:
        _default = Oracle.load(threads=threads)
    return _default
