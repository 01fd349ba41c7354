"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle at the tolerances of the precision contract.

Tolerances (written here, used by every parity test):
* FP32 outputs (delta_y, dB, dX, dA), each GEMM fed the same BF16 operands as
  the oracle: |gpu - oracle| <= 1e-6 * S elementwise, S = sum of |products|
  (times |alpha| for delta_y); S = 0 requires equality.
* BF16 intermediates (U, dU): at most 1 BF16 ulp apart (+0 and -0 equal);
  where the sum cancels so far that the FP32 band oracle +/- 1e-6 * S spans
  more than one BF16 ulp, the GPU value must lie in the BF16 rounding of that
  band (widened by 1 ulp): the FP32 contract carried through the rounding.
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


def _bf16_bits_of(v64: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v64, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def assert_bf16_close(name, got, ref, ref_f32=None, s=None, max_ulp=1, rel=REL_TOL):
    """``got`` within ``max_ulp`` BF16 ulp of ``ref``, or (given the oracle's FP32
    value before rounding and S) inside the BF16 image of ref_f32 +/- rel*S."""
    bad = bf16_ulp_distance(got, ref) > max_ulp
    if ref_f32 is not None and s is not None and bad.any():
        lo = _line(_bf16_bits_of(ref_f32.astype(np.float64) - rel * s))
        hi = _line(_bf16_bits_of(ref_f32.astype(np.float64) + rel * s))
        g = _line(got)
        bad &= ~((g >= lo - max_ulp) & (g <= hi + max_ulp))
    bad = np.argwhere(bad)
    assert bad.size == 0, f"{name}: {len(bad)} elements outside tolerance, e.g. at {tuple(bad[0])}: " \
                          f"{got[tuple(bad[0])]:#06x} vs {ref[tuple(bad[0])]:#06x}"


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
    assert_bf16_close("U", out["u"], ref_u, f_u, s_u)
    worst = {}
    y, sy = o.delta_y(out["u"], d["b"], alpha, want_s=True)
    worst["delta_y"] = assert_f32_within("delta_y", out["delta_y"], y, sy)
    dv = o.dv(d["dy"], alpha)
    ref_du, s_du, f_du = o.du(dv, d["b"], want_s=True, want_f32=True)
    assert_bf16_close("dU", out["du"], ref_du, f_du, s_du)
    db, sdb = o.db(dv, out["u"], True)
    worst["db"] = assert_f32_within("dB", out["db"], db, sdb)
    dx, sdx = o.dx(out["du"], d["a"], True)
    worst["dx"] = assert_f32_within("dX", out["dx"], dx, sdx)
    da, sda = o.da(out["du"], d["x"], True)
    worst["da"] = assert_f32_within("dA", out["da"], da, sda)
    return worst
