"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle at the tolerances of the precision contract.

Tolerances (written here, used by every parity test):
* FP32 outputs (delta_y, dB, dX, dA), each GEMM fed the same BF16 operands as
  the oracle: |gpu - oracle| <= 1e-6 * S elementwise, S = sum of |products|
  (times |alpha| for delta_y); S = 0 requires equality.
* BF16 intermediates (U, dU, and the BF16 dY_lora output): at most 1 BF16 ulp
  from the oracle (+0 and -0 equal). A value further away passes only when it
  lies in the BF16 image of the band the FP32 contract allows for the GPU's
  FP32 value before its rounding: [e - 1e-6 * S, e + 1e-6 * S] around the exact
  sum e, which lies within half an FP32 ulp of the oracle's FP32 value f (plus
  the oracle's own binary64 summation error, below 2e-12 * S). The band ends
  are rounded once, from binary64 straight to BF16 (nearest even), and nothing
  is added to them: rounding is monotone, so every FP32 value inside the band
  rounds inside its image. Where the image holds at most two BF16 values it
  cannot admit anything beyond 1 ulp; it matters only where the sum cancels
  so far that the band spans several BF16 ulps. Every call records how many
  elements took the band (BAND_LOG, printed at the end of the session).
* Batch invariance and reruns: bitwise.
"""
from __future__ import annotations

import numpy as np
import torch

from deterministic_arithmetic_gb300 import lora_delta as ld

REL_TOL = 1e-6


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def run(d: dict, alpha: float, device="cuda", rows: slice | None = None, check_status=True):
    """Forward + backward on the GPU for inputs ``d`` (bf16 bit arrays); with
    ``rows`` the batch is restricted to that row range (a sub-batch)."""
    x, dy = d["x"], d["dy"]
    if rows is not None:
        x, dy = x[rows], dy[rows]
    X, A, B, DY = dev_bf16(x, device), dev_bf16(d["a"], device), dev_bf16(d["b"], device), dev_bf16(dy, device)
    M, K = X.shape
    N, R = B.shape
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), device)
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), device)
    y, u = ld.lora_delta_fwd(X, A, B, alpha, workspace=wf)
    dx, da, db, du = ld.lora_delta_bwd(DY, X, A, B, u, alpha, workspace=wb)
    torch.cuda.synchronize()
    if check_status:
        assert ld.lora_delta_device_status(wf) == 0 and ld.lora_delta_device_status(wb) == 0
    return dict(u=host_bits(u), delta_y=host_f32(y), du=host_bits(du), dx=host_f32(dx), da=host_f32(da),
                db=host_f32(db))


def _line(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (sign-magnitude) mapped to a monotone integer line; +0 == -0."""
    v = np.asarray(v).astype(np.int32)
    return np.where(v & 0x8000, -(v & 0x7FFF), v)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between bf16 bit patterns."""
    return np.abs(_line(a) - _line(b))


def bf16_bits_rne(v64) -> np.ndarray:
    """bfloat16 bit patterns of binary64 values, each rounded once to the
    nearest bfloat16 (ties to even; beyond the largest finite value: +/-inf)."""
    v = np.asarray(v64, np.float64)
    _, e = np.frexp(v)                          # |v| in [2^(e-1), 2^e)
    q = np.maximum(e - 8, -133)                 # quantum: 8 significant bits, fixed below 2^-126
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.ldexp(np.rint(np.ldexp(v, -q)), q)   # exact scaling by powers of two; rint is ties-to-even
        f = r.astype(np.float32)                # exact: r is a bfloat16 value, or overflows to inf
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# (test, name, elements compared, elements that needed the FP32 band) of every BF16 check in this
# session; CURRENT_TEST is set by an autouse fixture in conftest.py
BAND_LOG: list[tuple[str, str, int, int]] = []
CURRENT_TEST = [""]


def assert_bf16_close(name, got, ref, ref_f32=None, s=None, rel=REL_TOL):
    """``got`` within 1 BF16 ulp of ``ref``, or (given the oracle's FP32 value
    before rounding and S) inside the BF16 image of the FP32 band of the exact
    sum. Returns the number of elements that needed the band."""
    got = np.asarray(got)
    far = bf16_ulp_distance(got, ref) > 1
    n_band = 0
    if ref_f32 is not None and s is not None and far.any():
        f = np.asarray(ref_f32, np.float32)
        slack = rel * np.asarray(s, np.float64) + 0.5 * np.spacing(np.abs(f)).astype(np.float64) \
            + 2e-12 * np.asarray(s, np.float64)
        lo = _line(bf16_bits_rne(f.astype(np.float64) - slack))
        hi = _line(bf16_bits_rne(f.astype(np.float64) + slack))
        g = _line(got)
        in_band = far & (g >= lo) & (g <= hi)
        n_band = int(in_band.sum())
        far &= ~in_band
    BAND_LOG.append((CURRENT_TEST[0], name, int(got.size), n_band))
    bad = np.argwhere(far)
    assert bad.size == 0, f"{name}: {len(bad)} elements outside tolerance, e.g. at {tuple(bad[0])}: " \
                          f"{got[tuple(bad[0])]:#06x} vs {ref[tuple(bad[0])]:#06x}"
    return n_band


def assert_f32_within(name, got, ref, s, rel=REL_TOL):
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = rel * s
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, f"{name}: {len(bad)} elements outside {rel}*sum|ab|, e.g. at {tuple(bad[0])}: " \
                          f"{got[tuple(bad[0])]!r} vs {ref[tuple(bad[0])]!r} (S={s[tuple(bad[0])]!r})"
    return float(np.max(err / np.where(s > 0, s, 1.0))) if err.size else 0.0


def assert_bitwise(name, got, ref):
    g = np.ascontiguousarray(got).view(np.uint8)
    r = np.ascontiguousarray(ref).view(np.uint8)
    assert got.shape == ref.shape and np.array_equal(g, r), f"{name}: not bitwise identical"


def check_parity(o, d: dict, alpha: float, out: dict):
    """Every boundary of ``out`` (a GPU run on all rows of ``d``) against the
    oracle: U and dU in chain mode, FP32 outputs per GEMM (fed the GPU's U/dU)."""
    ref_u, s_u, f_u = o.u(d["x"], d["a"], want_s=True, want_f32=True)
    worst = {"band_u": assert_bf16_close("U", out["u"], ref_u, f_u, s_u)}
    y, sy = o.delta_y(out["u"], d["b"], alpha, want_s=True)
    worst["delta_y"] = assert_f32_within("delta_y", out["delta_y"], y, sy)
    dv = o.dv(d["dy"], alpha)
    ref_du, s_du, f_du = o.du(dv, d["b"], want_s=True, want_f32=True)
    worst["band_du"] = assert_bf16_close("dU", out["du"], ref_du, f_du, s_du)
    db, sdb = o.db(dv, out["u"], True)
    worst["db"] = assert_f32_within("dB", out["db"], db, sdb)
    dx, sdx = o.dx(out["du"], d["a"], True)
    worst["dx"] = assert_f32_within("dX", out["dx"], dx, sdx)
    da, sda = o.da(out["du"], d["x"], True)
    worst["da"] = assert_f32_within("dA", out["da"], da, sda)
    return worst
