"""Python binding of the C ABI in ``include/lora_delta.h`` (ctypes).

Argument marshalling only: every step of the operator runs in the CUDA
kernels of ``liblora_delta.so``. PyTorch provides device memory and streams.
There is no fallback: if the library is missing or the device is not a
GB300, the calls raise.

Names follow the C ABI: ``lora_delta_fwd(x, a, b, alpha)`` returns
``(delta_y, u)``; ``lora_delta_bwd(dy, x, a, b, u, alpha)`` returns
``(dx, da, db, du)`` (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA +
Triton, both batch-invariant", section "Summary").
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblora_delta.so")

LORA_OK = 0
STATUS_NAMES = {0: "LORA_OK", 1: "LORA_ERR_NULL", 2: "LORA_ERR_SHAPE", 3: "LORA_ERR_ALIGN", 4: "LORA_ERR_RANK",
                5: "LORA_ERR_WORKSPACE", 6: "LORA_ERR_CUDA", 7: "LORA_ERR_DEVICE", 8: "LORA_ERR_TIMEOUT"}


class LoraDeltaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_lib().lora_status_str(code).decode()})")


_LIB = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
MAX_SITES = 4


class FwdSite(ctypes.Structure):
    """``lora_fwd_site`` of include/lora_delta.h."""
    _fields_ = [("x", _vp), ("a", _vp), ("b", _vp), ("alpha", ctypes.c_float), ("M", _i64), ("K", _i64),
                ("N", _i64), ("delta_y", _vp), ("u", _vp)]


class BwdSite(ctypes.Structure):
    """``lora_bwd_site`` of include/lora_delta.h."""
    _fields_ = [("dy", _vp), ("x", _vp), ("a", _vp), ("b", _vp), ("u", _vp), ("alpha", ctypes.c_float),
                ("M", _i64), ("K", _i64), ("N", _i64), ("dx", _vp), ("da", _vp), ("db", _vp), ("du", _vp)]


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        lib.lora_delta_fwd.argtypes = [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                                       ctypes.c_size_t, _vp]
        lib.lora_delta_fwd.restype = ctypes.c_int
        lib.lora_delta_fwd_bf16.argtypes = lib.lora_delta_fwd.argtypes
        lib.lora_delta_fwd_bf16.restype = ctypes.c_int
        lib.lora_delta_fwd_fused.argtypes = [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64, _i64, _vp, _vp,
                                             ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        lib.lora_delta_fwd_fused.restype = ctypes.c_int
        lib.lora_delta_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                                       _vp, _vp, ctypes.c_size_t, _vp]
        lib.lora_delta_bwd.restype = ctypes.c_int
        if hasattr(lib, "lora_delta_bwd_f32dy"):
            lib.lora_delta_bwd_f32dy.argtypes = lib.lora_delta_bwd.argtypes
            lib.lora_delta_bwd_f32dy.restype = ctypes.c_int
            lib.lora_delta_bwd_f32dy_workspace_size.argtypes = [_i64, _i64, _i64, _i64]
            lib.lora_delta_bwd_f32dy_workspace_size.restype = ctypes.c_size_t
        for fn in (lib.lora_delta_fwd_workspace_size, lib.lora_delta_bwd_workspace_size,
                   lib.lora_delta_fwd_workspace, lib.lora_delta_bwd_workspace):
            fn.argtypes = [_i64, _i64, _i64, _i64]
            fn.restype = ctypes.c_size_t
        lib.lora_delta_fwd_noalloc.argtypes = [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64, _i64, _vp, _vp, _vp]
        lib.lora_delta_fwd_noalloc.restype = ctypes.c_int
        lib.lora_delta_fwd_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.lora_delta_fwd_noalloc_status.restype = ctypes.c_int
        if hasattr(lib, "lora_delta_fwd_grouped"):
            lib.lora_delta_fwd_grouped_workspace_size.argtypes = [ctypes.POINTER(FwdSite), ctypes.c_int, _i64]
            lib.lora_delta_fwd_grouped_workspace_size.restype = ctypes.c_size_t
            lib.lora_delta_bwd_grouped_workspace_size.argtypes = [ctypes.POINTER(BwdSite), ctypes.c_int, _i64]
            lib.lora_delta_bwd_grouped_workspace_size.restype = ctypes.c_size_t
            lib.lora_delta_fwd_grouped.argtypes = [ctypes.POINTER(FwdSite), ctypes.c_int, _i64, ctypes.c_int, _vp,
                                                   ctypes.c_size_t, _vp]
            lib.lora_delta_fwd_grouped.restype = ctypes.c_int
            lib.lora_delta_bwd_grouped.argtypes = [ctypes.POINTER(BwdSite), ctypes.c_int, _i64, _vp, ctypes.c_size_t,
                                                   _vp]
            lib.lora_delta_bwd_grouped.restype = ctypes.c_int
        if hasattr(lib, "lora_delta_grads_exact"):
            lib.lora_delta_exact_slots.argtypes = []
            lib.lora_delta_exact_slots.restype = ctypes.c_int
            lib.lora_delta_grads_exact_workspace_size.argtypes = [_i64, _i64, _i64, _i64]
            lib.lora_delta_grads_exact_workspace_size.restype = ctypes.c_size_t
            lib.lora_delta_grads_exact.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64, _i64, _vp,
                                                   _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
            lib.lora_delta_grads_exact.restype = ctypes.c_int
            lib.lora_delta_grads_exact_f32dy.argtypes = lib.lora_delta_grads_exact.argtypes
            lib.lora_delta_grads_exact_f32dy.restype = ctypes.c_int
            lib.lora_delta_grads_exact_f32dy_workspace_size.argtypes = [_i64, _i64, _i64, _i64]
            lib.lora_delta_grads_exact_f32dy_workspace_size.restype = ctypes.c_size_t
            lib.lora_delta_exact_combine.argtypes = [_vp, _vp, _i64, _vp, _vp]
            lib.lora_delta_exact_combine.restype = ctypes.c_int
            lib.lora_delta_exact_finalize.argtypes = [_vp, _i64, _vp, _vp]
            lib.lora_delta_exact_finalize.restype = ctypes.c_int
            lib.lora_delta_exact_rate_probe.argtypes = [_i64, _vp, ctypes.c_size_t, ctypes.POINTER(_i64), _vp]
            lib.lora_delta_exact_rate_probe.restype = ctypes.c_int
            lib.lora_delta_exact_rate_probe_sink_bytes.argtypes = []
            lib.lora_delta_exact_rate_probe_sink_bytes.restype = ctypes.c_size_t
        lib.lora_status_str.argtypes = [ctypes.c_int]
        lib.lora_status_str.restype = ctypes.c_char_p
        lib.lora_delta_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
        lib.lora_delta_device_status.restype = ctypes.c_int
        lib.lora_delta_set_profile_events.argtypes = [ctypes.POINTER(_vp), ctypes.c_int]
        lib.lora_delta_set_profile_events.restype = ctypes.c_int
        lib.lora_delta_set_schedule.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.lora_delta_set_schedule.restype = ctypes.c_int
        lib.lora_delta_schedule.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.lora_delta_schedule.restype = ctypes.c_int
        lib.lora_delta_plan.argtypes = [ctypes.c_int, _i64, _i64, _i64, _i64, ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_int)]
        lib.lora_delta_plan.restype = ctypes.c_int
        lib.lora_delta_describe.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
        lib.lora_delta_describe.restype = ctypes.c_size_t
        _LIB = lib
    return _LIB


def library() -> ctypes.CDLL:
    """The loaded ``liblora_delta.so`` (raises when it is missing)."""
    return _lib()


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def lora_delta_fwd_workspace_size(M: int, K: int, N: int, R: int) -> int:
    return int(_lib().lora_delta_fwd_workspace_size(M, K, N, R))


def lora_delta_bwd_workspace_size(M: int, K: int, N: int, R: int) -> int:
    return int(_lib().lora_delta_bwd_workspace_size(M, K, N, R))


def lora_delta_fwd_workspace(M: int, K: int, N: int, R: int) -> int:
    return int(_lib().lora_delta_fwd_workspace(M, K, N, R))


def lora_delta_bwd_workspace(M: int, K: int, N: int, R: int) -> int:
    return int(_lib().lora_delta_bwd_workspace(M, K, N, R))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed workspace (its first 256 bytes are the device status block)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def lora_delta_fwd(x, a, b, alpha: float, *, delta_y=None, u=None, workspace=None, stream=None):
    """Forward: ``u = bf16(x @ a.T)``, ``delta_y = fp32(u @ b.T) * alpha``.

    A BF16 ``delta_y`` selects ``lora_delta_fwd_bf16`` (the same FP32 value,
    rounded to BF16 inside the kernel)."""
    M, K = x.shape
    R = a.shape[0]
    N = b.shape[0]
    _check(x, "x", torch.bfloat16, (M, K)); _check(a, "a", torch.bfloat16, (R, K)); _check(b, "b", torch.bfloat16, (N, R))
    if delta_y is None:
        delta_y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if u is None:
        u = torch.empty((M, R), dtype=torch.bfloat16, device=x.device)
    y_bf16 = delta_y.dtype == torch.bfloat16
    _check(delta_y, "delta_y", torch.bfloat16 if y_bf16 else torch.float32, (M, N)); _check(u, "u", torch.bfloat16, (M, R))
    need = lora_delta_fwd_workspace_size(M, K, N, R)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    name = "lora_delta_fwd_bf16" if y_bf16 else "lora_delta_fwd"
    rc = getattr(_lib(), name)(_ptr(x), _ptr(a), _ptr(b), float(alpha), M, K, N, R, _ptr(delta_y), _ptr(u),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, name)
    return delta_y, u


def lora_delta_fwd_fused(x, a, b, alpha: float, *, delta_y=None, u=None, workspace=None, stream=None):
    """The forward in a single launch (same bits as ``lora_delta_fwd``); a BF16 ``delta_y``
    selects the BF16 output."""
    M, K = x.shape
    R = a.shape[0]
    N = b.shape[0]
    _check(x, "x", torch.bfloat16, (M, K)); _check(a, "a", torch.bfloat16, (R, K)); _check(b, "b", torch.bfloat16, (N, R))
    if delta_y is None:
        delta_y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if u is None:
        u = torch.empty((M, R), dtype=torch.bfloat16, device=x.device)
    y_bf16 = delta_y.dtype == torch.bfloat16
    _check(delta_y, "delta_y", torch.bfloat16 if y_bf16 else torch.float32, (M, N)); _check(u, "u", torch.bfloat16, (M, R))
    if workspace is None:
        workspace = new_workspace(lora_delta_fwd_workspace_size(M, K, N, R), x.device)
    rc = _lib().lora_delta_fwd_fused(_ptr(x), _ptr(a), _ptr(b), float(alpha), M, K, N, R, _ptr(delta_y), _ptr(u),
                                     int(y_bf16), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_fwd_fused")
    return delta_y, u


def lora_delta_bwd_f32dy_workspace_size(M: int, K: int, N: int, R: int) -> int:
    return int(_lib().lora_delta_bwd_f32dy_workspace_size(M, K, N, R))


def lora_delta_bwd(dy, x, a, b, u, alpha: float, *, dx=None, da=None, db=None, du=None, workspace=None, stream=None):
    """Backward: returns ``(dx, da, db, du)``; no base-weight gradient.

    An FP32 ``dy`` selects ``lora_delta_bwd_f32dy`` (dV = bf16(fp32(dy * alpha)))."""
    M, K = x.shape
    R = a.shape[0]
    N = b.shape[0]
    dy_f32 = dy.dtype == torch.float32
    _check(dy, "dy", torch.float32 if dy_f32 else torch.bfloat16, (M, N)); _check(x, "x", torch.bfloat16, (M, K))
    _check(a, "a", torch.bfloat16, (R, K)); _check(b, "b", torch.bfloat16, (N, R)); _check(u, "u", torch.bfloat16, (M, R))
    dev = x.device
    dx = torch.empty((M, K), dtype=torch.float32, device=dev) if dx is None else dx
    da = torch.empty((R, K), dtype=torch.float32, device=dev) if da is None else da
    db = torch.empty((N, R), dtype=torch.float32, device=dev) if db is None else db
    du = torch.empty((M, R), dtype=torch.bfloat16, device=dev) if du is None else du
    _check(dx, "dx", torch.float32, (M, K)); _check(da, "da", torch.float32, (R, K))
    _check(db, "db", torch.float32, (N, R)); _check(du, "du", torch.bfloat16, (M, R))
    need = (lora_delta_bwd_f32dy_workspace_size if dy_f32 else lora_delta_bwd_workspace_size)(M, K, N, R)
    if workspace is None:
        workspace = new_workspace(need, dev)
    name = "lora_delta_bwd_f32dy" if dy_f32 else "lora_delta_bwd"
    rc = getattr(_lib(), name)(_ptr(dy), _ptr(x), _ptr(a), _ptr(b), _ptr(u), float(alpha), M, K, N, R, _ptr(dx),
                               _ptr(da), _ptr(db), _ptr(du), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, name)
    return dx, da, db, du


def lora_delta_exact_slots() -> int:
    """int64 slots of one exact-mode digit array (18 digits, then +inf, -inf and NaN counts)."""
    return int(_lib().lora_delta_exact_slots())


def lora_delta_grads_exact_workspace_size(M: int, K: int, N: int, R: int) -> int:
    return int(_lib().lora_delta_grads_exact_workspace_size(M, K, N, R))


def lora_delta_grads_exact(dy, x, u, du, alpha: float, *, da=None, db=None, da_digits=None,
                           db_digits=None, want=("da", "db"), workspace=None, stream=None):
    """Exact mode of the weight gradients (page "det-train", section "Method"):
    dA = rn32(exact sum du^T x), dB = rn32(exact sum dv^T u), dv = bf16(fp32(dy * alpha)).

    ``want`` names the outputs to allocate when not given: any of "da", "db",
    "da_digits" ([R][K][slots] int64), "db_digits" ([N][R][slots] int64). Returns
    the dict of outputs written. ``dy`` or ``x`` may be None when its gradient
    is not wanted. An FP32 ``dy`` selects ``lora_delta_grads_exact_f32dy``
    (dV = bf16(fp32(dy * alpha)))."""
    M, R = (u if u is not None else du).shape
    K = x.shape[1] if x is not None else 8
    N = dy.shape[1] if dy is not None else 8
    dev = (u if u is not None else du).device
    slots = lora_delta_exact_slots()
    shapes = {"da": ((R, K), torch.float32), "db": ((N, R), torch.float32),
              "da_digits": ((R, K, slots), torch.int64), "db_digits": ((N, R, slots), torch.int64)}
    outs = {"da": da, "db": db, "da_digits": da_digits, "db_digits": db_digits}
    for k in want:
        if outs[k] is None:
            outs[k] = torch.empty(shapes[k][0], dtype=shapes[k][1], device=dev)
    for k, v in outs.items():
        if v is not None:
            _check(v, k, shapes[k][1], shapes[k][0])
    if x is not None:
        _check(x, "x", torch.bfloat16, (M, K))
    dy_f32 = dy is not None and dy.dtype == torch.float32
    if dy is not None:
        _check(dy, "dy", torch.float32 if dy_f32 else torch.bfloat16, (M, N))
    if u is not None:
        _check(u, "u", torch.bfloat16, (M, R))
    if du is not None:
        _check(du, "du", torch.bfloat16, (M, R))
    name = "lora_delta_grads_exact_f32dy" if dy_f32 else "lora_delta_grads_exact"
    if workspace is None:
        workspace = new_workspace(int(getattr(_lib(), name + "_workspace_size")(M, K, N, R)), dev)
    rc = getattr(_lib(), name)(_ptr(dy), _ptr(x), _ptr(u), _ptr(du), float(alpha), M, K, N, R,
                               _ptr(outs["da"]), _ptr(outs["db"]), _ptr(outs["da_digits"]),
                               _ptr(outs["db_digits"]), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, name)
    return {k: v for k, v in outs.items() if v is not None}


def lora_delta_exact_combine(a, b=None, *, out=None, stream=None):
    """Digit arrays of the sums a + b (same shape [..., slots] int64), normalised; out may be a or
    b. b None: a normalised."""
    slots = lora_delta_exact_slots()
    for t, name in ((a, "a"), (b, "b")):
        if t is None and name == "b":
            continue
        if t.dtype != torch.int64 or t.shape != a.shape or t.shape[-1] != slots or not t.is_contiguous():
            raise ValueError(f"digit arrays: contiguous [..., {slots}] int64 tensors of one shape")
    out = torch.empty_like(a) if out is None else out
    _check(out, "out", torch.int64, tuple(a.shape))
    rc = _lib().lora_delta_exact_combine(_ptr(a), _ptr(b), a.numel() // slots, _ptr(out), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_exact_combine")
    return out


def lora_delta_exact_rate_probe(iters: int, *, sink=None, stream=None) -> int:
    """Enqueue the exact mode's multiply-add rate probe; returns the number of multiply-adds the
    launch performs (time it with CUDA events on ``stream``)."""
    need = int(_lib().lora_delta_exact_rate_probe_sink_bytes())
    if need == 0:
        raise LoraDeltaError(7, "lora_delta_exact_rate_probe_sink_bytes")
    if sink is None:
        sink = torch.empty(need, dtype=torch.uint8, device="cuda")
    products = _i64(0)
    rc = _lib().lora_delta_exact_rate_probe(int(iters), _ptr(sink), sink.numel() * sink.element_size(),
                                            ctypes.byref(products), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_exact_rate_probe")
    return int(products.value)


def lora_delta_exact_all_reduce(digits, *, group=None, stream=None):
    """The digit arrays of the sum over the ranks of ``group`` (torch.distributed), in place:
    one int64 sum all-reduce -- exact and order-free, so the result is the same at any world
    size and rank order -- then normalised by the library (page "det-train", "API":
    det_all_reduce). Run by every rank of the group on its own digits."""
    import torch.distributed as dist

    dist.all_reduce(digits, op=dist.ReduceOp.SUM, group=group)
    return lora_delta_exact_combine(digits, None, out=digits, stream=stream)


def lora_delta_exact_finalize(digits, *, out=None, stream=None):
    """FP32 values of digit arrays [..., slots] (rounded to nearest even, once)."""
    slots = lora_delta_exact_slots()
    if digits.dtype != torch.int64 or digits.shape[-1] != slots or not digits.is_contiguous():
        raise ValueError(f"digit arrays: contiguous [..., {slots}] int64")
    out = torch.empty(tuple(digits.shape[:-1]), dtype=torch.float32, device=digits.device) if out is None else out
    _check(out, "out", torch.float32, tuple(digits.shape[:-1]))
    rc = _lib().lora_delta_exact_finalize(_ptr(digits), digits.numel() // slots, _ptr(out), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_exact_finalize")
    return out


def lora_delta_device_status(workspace: torch.Tensor) -> int:
    """Device status code of a workspace (0 = no kernel reported a problem)."""
    code = ctypes.c_int(0)
    rc = _lib().lora_delta_device_status(_ptr(workspace), ctypes.byref(code))
    if rc not in (LORA_OK, 8):
        raise LoraDeltaError(rc, "lora_delta_device_status")
    return int(code.value)


def lora_delta_fwd_noalloc(x, a, b, alpha: float, *, delta_y=None, u=None, stream=None):
    """Forward without a workspace (scratch from the library's fixed device array): for callers
    that may not allocate device memory. Same outputs and bits as ``lora_delta_fwd``."""
    M, K = x.shape
    R = a.shape[0]
    N = b.shape[0]
    _check(x, "x", torch.bfloat16, (M, K)); _check(a, "a", torch.bfloat16, (R, K)); _check(b, "b", torch.bfloat16, (N, R))
    if delta_y is None:
        delta_y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if u is None:
        u = torch.empty((M, R), dtype=torch.bfloat16, device=x.device)
    _check(delta_y, "delta_y", torch.float32, (M, N)); _check(u, "u", torch.bfloat16, (M, R))
    rc = _lib().lora_delta_fwd_noalloc(_ptr(x), _ptr(a), _ptr(b), float(alpha), M, K, N, R, _ptr(delta_y), _ptr(u),
                                       _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_fwd_noalloc")
    return delta_y, u


def lora_delta_fwd_noalloc_status() -> int:
    """Device status code of the latest ``lora_delta_fwd_noalloc`` call on the current device."""
    code = ctypes.c_int(0)
    rc = _lib().lora_delta_fwd_noalloc_status(ctypes.byref(code))
    if rc not in (LORA_OK, 8):
        raise LoraDeltaError(rc, "lora_delta_fwd_noalloc_status")
    return int(code.value)


def lora_delta_set_profile_events(events) -> None:
    """Record ``torch.cuda.Event``s around each internal kernel (None = off)."""
    if not events:
        _lib().lora_delta_set_profile_events(None, 0)
        return
    for ev in events:
        if not ev.cuda_event:        # torch creates the CUDA event lazily, at its first record
            ev.record()
    arr = (_vp * len(events))(*[ev.cuda_event for ev in events])
    rc = _lib().lora_delta_set_profile_events(arr, len(events))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_set_profile_events")


SCHEDULE_SEPARATE, SCHEDULE_CLUSTER_REDUCE, SCHEDULE_CLUSTER_SINGLE, SCHEDULE_AUTO = 0, 1, 2, 3


def lora_delta_set_schedule(schedule: int, cluster_size: int = 0) -> None:
    """Launch schedule of the single-site passes (``SCHEDULE_*``) and the cluster size of the
    cluster schedules (0: the default). Changes no result bit."""
    rc = _lib().lora_delta_set_schedule(int(schedule), int(cluster_size))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_set_schedule")


def lora_delta_schedule() -> tuple[int, int]:
    """(schedule, cluster size setting)."""
    cl = ctypes.c_int(0)
    return int(_lib().lora_delta_schedule(ctypes.byref(cl))), int(cl.value)


def lora_delta_plan(backward: bool, M: int, K: int, N: int, R: int) -> tuple[int, int]:
    """(schedule, launches) a single-site call of this shape takes on the current device."""
    sc, nl = ctypes.c_int(0), ctypes.c_int(0)
    rc = _lib().lora_delta_plan(1 if backward else 0, M, K, N, R, ctypes.byref(sc), ctypes.byref(nl))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_plan")
    return int(sc.value), int(nl.value)


def lora_delta_describe() -> str:
    n = _lib().lora_delta_describe(None, 0)
    buf = ctypes.create_string_buffer(n)
    _lib().lora_delta_describe(buf, n)
    return buf.value.decode()


def lora_status_str(code: int) -> str:
    return _lib().lora_status_str(code).decode()


def lora_delta_fwd_grouped(sites, *, y_bf16: bool = False, workspace=None, stream=None):
    """Forward of several sites in one call. ``sites``: sequence of dicts with
    ``x, a, b, alpha`` and optional ``delta_y, u`` outputs (allocated when
    absent; BF16 ``delta_y`` when ``y_bf16``). All sites share the rank R.
    Returns ``[(delta_y, u), ...]``."""
    n = len(sites)
    if not 1 <= n <= MAX_SITES:
        raise ValueError(f"1 to {MAX_SITES} sites per call, got {n}")
    R = sites[0]["a"].shape[0]
    arr = (FwdSite * n)()
    outs = []
    for i, s in enumerate(sites):
        x, a, b = s["x"], s["a"], s["b"]
        M, K = x.shape
        N = b.shape[0]
        _check(x, "x", torch.bfloat16, (M, K)); _check(a, "a", torch.bfloat16, (R, K)); _check(b, "b", torch.bfloat16, (N, R))
        ydt = torch.bfloat16 if y_bf16 else torch.float32
        y = s.get("delta_y")
        y = torch.empty((M, N), dtype=ydt, device=x.device) if y is None else y
        u = s.get("u")
        u = torch.empty((M, R), dtype=torch.bfloat16, device=x.device) if u is None else u
        _check(y, "delta_y", ydt, (M, N)); _check(u, "u", torch.bfloat16, (M, R))
        arr[i] = FwdSite(_ptr(x), _ptr(a), _ptr(b), float(s["alpha"]), M, K, N, _ptr(y), _ptr(u))
        outs.append((y, u))
    need = int(_lib().lora_delta_fwd_grouped_workspace_size(arr, n, R))
    if need == 0:
        raise LoraDeltaError(2, "lora_delta_fwd_grouped_workspace_size")
    if workspace is None:
        workspace = new_workspace(need, sites[0]["x"].device)
    rc = _lib().lora_delta_fwd_grouped(arr, n, R, int(bool(y_bf16)), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_fwd_grouped")
    return outs


def lora_delta_bwd_grouped(sites, *, workspace=None, stream=None):
    """Backward of several sites in one call. ``sites``: sequence of dicts
    with ``dy, x, a, b, u, alpha`` and optional ``dx, da, db, du`` outputs.
    Returns ``[(dx, da, db, du), ...]``."""
    n = len(sites)
    if not 1 <= n <= MAX_SITES:
        raise ValueError(f"1 to {MAX_SITES} sites per call, got {n}")
    R = sites[0]["a"].shape[0]
    arr = (BwdSite * n)()
    outs = []
    for i, s in enumerate(sites):
        dy, x, a, b, u = s["dy"], s["x"], s["a"], s["b"], s["u"]
        M, K = x.shape
        N = b.shape[0]
        _check(dy, "dy", torch.bfloat16, (M, N)); _check(x, "x", torch.bfloat16, (M, K))
        _check(a, "a", torch.bfloat16, (R, K)); _check(b, "b", torch.bfloat16, (N, R)); _check(u, "u", torch.bfloat16, (M, R))
        dev = x.device
        dx = torch.empty((M, K), dtype=torch.float32, device=dev) if s.get("dx") is None else s["dx"]
        da = torch.empty((R, K), dtype=torch.float32, device=dev) if s.get("da") is None else s["da"]
        db = torch.empty((N, R), dtype=torch.float32, device=dev) if s.get("db") is None else s["db"]
        du = torch.empty((M, R), dtype=torch.bfloat16, device=dev) if s.get("du") is None else s["du"]
        _check(dx, "dx", torch.float32, (M, K)); _check(da, "da", torch.float32, (R, K))
        _check(db, "db", torch.float32, (N, R)); _check(du, "du", torch.bfloat16, (M, R))
        arr[i] = BwdSite(_ptr(dy), _ptr(x), _ptr(a), _ptr(b), _ptr(u), float(s["alpha"]), M, K, N, _ptr(dx), _ptr(da),
                         _ptr(db), _ptr(du))
        outs.append((dx, da, db, du))
    need = int(_lib().lora_delta_bwd_grouped_workspace_size(arr, n, R))
    if need == 0:
        raise LoraDeltaError(2, "lora_delta_bwd_grouped_workspace_size")
    if workspace is None:
        workspace = new_workspace(need, sites[0]["x"].device)
    rc = _lib().lora_delta_bwd_grouped(arr, n, R, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    if rc != LORA_OK:
        raise LoraDeltaError(rc, "lora_delta_bwd_grouped")
    return outs
