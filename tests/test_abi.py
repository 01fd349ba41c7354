"""The C ABI without a GPU: the library builds and loads, exports every entry
point that include/lora_delta.h declares, and rejects bad arguments on the
host before touching the device."""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_delta.h")


@pytest.fixture(scope="module")
def lib():
    from deterministic_arithmetic_gb300 import build_lib
    from deterministic_arithmetic_gb300 import lora_delta as ld

    build_lib.build()
    return ld.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(lora_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


# The boundary as first listed for the operator: the two passes, their workspace queries
# and the status strings (with the enum as its argument type).
BOUNDARY = ("lora_delta_fwd", "lora_delta_bwd", "lora_delta_fwd_workspace", "lora_delta_bwd_workspace",
            "lora_status_str")


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in BOUNDARY + ("lora_delta_fwd_bf16", "lora_delta_fwd_workspace_size", "lora_delta_bwd_workspace_size",
                         "lora_delta_device_status", "lora_delta_set_profile_events", "lora_delta_describe",
                         "lora_delta_fwd_noalloc", "lora_delta_fwd_noalloc_status"):
        assert n in names, n
    text = open(HEADER).read()
    assert re.search(r"const char \*lora_status_str\(lora_status status\);", text)


def test_boundary_workspace_queries_agree(lib):
    for q in ("lora_delta_fwd_workspace", "lora_delta_bwd_workspace", "lora_delta_fwd_workspace_size",
              "lora_delta_bwd_workspace_size"):
        getattr(lib, q).argtypes = [ctypes.c_int64] * 4
        getattr(lib, q).restype = ctypes.c_size_t
    for shape in ((8192, 4096, 4096, 16), (300, 1032, 520, 40), (0, 128, 96, 8), (8, 100, 96, 8)):
        assert lib.lora_delta_fwd_workspace(*shape) == lib.lora_delta_fwd_workspace_size(*shape)
        assert lib.lora_delta_bwd_workspace(*shape) == lib.lora_delta_bwd_workspace_size(*shape)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/lora_delta.h but not exported"


def test_status_strings(lib):
    lib.lora_status_str.restype = ctypes.c_char_p
    seen = set()
    for code in range(9):
        s = lib.lora_status_str(code).decode()
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 9
    assert lib.lora_status_str(99).decode() == "unknown status"


def test_workspace_sizes():
    from deterministic_arithmetic_gb300 import lora_delta as ld

    f = ld.lora_delta_fwd_workspace_size(8192, 4096, 4096, 16)
    b = ld.lora_delta_bwd_workspace_size(8192, 4096, 4096, 16)
    control = 256 + 65536     # status block and control words (LORA_DELTA_CONTROL_BYTES)
    # U partials: 4 slices of 1024 x 8192 rows x 16 x fp32
    assert f == control + 4 * 8192 * 16 * 4
    # dU partials (8 slices of 512 columns: the fused dY pass), dB partials (room for one per 128-row
    # tile: the cluster reductions' units may be single tiles), dA chunk partials (32 chunks of 256 rows)
    assert b == control + 8 * 8192 * 16 * 4 + 64 * 16 * 4096 * 4 + 32 * 16 * 4096 * 4
    assert ld.lora_delta_fwd_workspace_size(0, 128, 96, 8) == control
    text = open(HEADER).read()
    assert re.search(r"#define LORA_DELTA_CONTROL_BYTES \(256 \+ 65536\)", text)
    for bad in ((8, 100, 96, 8), (8, 128, 90, 8), (8, 128, 96, 12), (8, 128, 96, 72), (-1, 128, 96, 8), (8, 0, 96, 8)):
        assert ld.lora_delta_fwd_workspace_size(*bad) == 0
        assert ld.lora_delta_bwd_workspace_size(*bad) == 0
    assert ld.lora_delta_fwd_workspace_size(100, 128, 96, 8) <= ld.lora_delta_fwd_workspace_size(200, 128, 96, 8)


def _fwd(lib, ptrs, M=64, K=128, N=96, R=8, ws_bytes=1 << 20, name="lora_delta_fwd"):
    f = getattr(lib, name)
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float] + [ctypes.c_int64] * 4 + [ctypes.c_void_p] * 3 + \
                 [ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    x, a, b, y, u, ws = ptrs
    return f(x, a, b, 2.0, M, K, N, R, y, u, ws, ws_bytes, None)


def _bwd(lib, ptrs, M=64, K=128, N=96, R=8, ws_bytes=1 << 22):
    f = lib.lora_delta_bwd
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_float] + [ctypes.c_int64] * 4 + [ctypes.c_void_p] * 5 + \
                 [ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    dy, x, a, b, u, dx, da, db, du, ws = ptrs
    return f(dy, x, a, b, u, 2.0, M, K, N, R, dx, da, db, du, ws, ws_bytes, None)


FAKE = 0x10000   # never dereferenced: every case below fails its host-side checks first


def test_argument_errors_are_host_side(lib):
    ok6 = [FAKE] * 6
    assert _fwd(lib, ok6, M=0) == 0                                   # M = 0 is a no-op
    assert _fwd(lib, [None] + ok6[1:]) == 1                           # LORA_ERR_NULL
    assert _fwd(lib, ok6, K=100) == 2                                 # LORA_ERR_SHAPE
    assert _fwd(lib, ok6, N=0) == 2
    assert _fwd(lib, ok6, M=-5) == 2
    assert _fwd(lib, ok6, R=12) == 4                                  # LORA_ERR_RANK
    assert _fwd(lib, ok6, R=72) == 4
    assert _fwd(lib, [FAKE + 2] + ok6[1:]) == 3                       # LORA_ERR_ALIGN
    assert _fwd(lib, ok6, ws_bytes=16) == 5                           # LORA_ERR_WORKSPACE
    # the BF16-output forward shares the checks
    assert _fwd(lib, ok6, M=0, name="lora_delta_fwd_bf16") == 0
    assert _fwd(lib, ok6[:3] + [None] + ok6[4:], name="lora_delta_fwd_bf16") == 1
    assert _fwd(lib, ok6, R=12, name="lora_delta_fwd_bf16") == 4
    assert _fwd(lib, ok6[:3] + [FAKE + 4] + ok6[4:], name="lora_delta_fwd_bf16") == 3
    assert _fwd(lib, ok6, ws_bytes=16, name="lora_delta_fwd_bf16") == 5
    ok10 = [FAKE] * 10
    assert _bwd(lib, ok10, M=0) == 0
    assert _bwd(lib, ok10[:8] + [None, FAKE]) == 1
    assert _bwd(lib, ok10, R=0) == 4
    assert _bwd(lib, ok10[:5] + [FAKE + 8] + ok10[6:]) == 3
    assert _bwd(lib, ok10, ws_bytes=300) == 5


def test_valid_call_without_gpu_fails_loudly(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is for hosts without one")
    # all arguments valid: the call reaches the device check and must report an error, not compute on the CPU
    assert _fwd(lib, [FAKE] * 6) in (6, 7)
    assert _fwd(lib, [FAKE] * 6, name="lora_delta_fwd_bf16") in (6, 7)


def test_describe(lib):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    d = json.loads(ld.lora_delta_describe())
    assert "canonical pairwise" in d["numeric_profile"] and d["arch"] == "sm_103a"


def test_python_binding_fails_without_library(tmp_path, monkeypatch):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    monkeypatch.setattr(ld, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ld, "_LIB", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        ld.library()


def test_grouped_calls_host_checks(lib):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    def fsite(M=64, K=128, N=96, ptr=FAKE, **kw):
        s = dict(x=ptr, a=ptr, b=ptr, alpha=2.0, M=M, K=K, N=N, delta_y=ptr, u=ptr)
        s.update(kw)
        return ld.FwdSite(**s)

    def bsite(M=64, K=128, N=96, ptr=FAKE, **kw):
        s = dict(dy=ptr, x=ptr, a=ptr, b=ptr, u=ptr, alpha=2.0, M=M, K=K, N=N, dx=ptr, da=ptr, db=ptr, du=ptr)
        s.update(kw)
        return ld.BwdSite(**s)

    def arr(cls, sites):
        a = (cls * len(sites))()
        for i, s in enumerate(sites):
            a[i] = s
        return a

    f = lib.lora_delta_fwd_grouped
    g = lib.lora_delta_bwd_grouped
    big = 1 << 30
    # workspace: one control block plus every site's partial sums
    control = 256 + 65536
    two = arr(ld.FwdSite, [fsite(), fsite(M=300, K=264, N=136)])
    assert lib.lora_delta_fwd_grouped_workspace_size(two, 2, 8) == \
        ld.lora_delta_fwd_workspace_size(64, 128, 96, 8) + ld.lora_delta_fwd_workspace_size(300, 264, 136, 8) - control
    btwo = arr(ld.BwdSite, [bsite(), bsite(M=300, K=264, N=136)])
    assert lib.lora_delta_bwd_grouped_workspace_size(btwo, 2, 16) == \
        ld.lora_delta_bwd_workspace_size(64, 128, 96, 16) + ld.lora_delta_bwd_workspace_size(300, 264, 136, 16) - control
    assert lib.lora_delta_fwd_grouped_workspace_size(two, 5, 8) == 0
    assert lib.lora_delta_fwd_grouped_workspace_size(arr(ld.FwdSite, [fsite(), fsite(K=100)]), 2, 8) == 0
    # errors, each site checked as a single-site call would be
    assert f(None, 1, 8, 0, FAKE, big, None) == 1                                        # LORA_ERR_NULL
    assert f(two, 0, 8, 0, FAKE, big, None) == 2 and f(two, 5, 8, 0, FAKE, big, None) == 2   # count
    assert f(arr(ld.FwdSite, [fsite(), fsite(N=90)]), 2, 8, 0, FAKE, big, None) == 2    # LORA_ERR_SHAPE
    assert f(two, 2, 12, 0, FAKE, big, None) == 4                                       # LORA_ERR_RANK
    assert f(arr(ld.FwdSite, [fsite(), fsite(u=None)]), 2, 8, 0, FAKE, big, None) == 1
    assert f(arr(ld.FwdSite, [fsite(), fsite(x=FAKE + 2)]), 2, 8, 0, FAKE, big, None) == 3
    assert f(two, 2, 8, 0, FAKE, 300, None) == 5                                        # LORA_ERR_WORKSPACE
    assert f(two, 2, 8, 0, None, big, None) == 1
    assert f(arr(ld.FwdSite, [fsite(M=0, ptr=None), fsite(M=0, ptr=None)]), 2, 8, 0, None, 0, None) == 0
    assert g(arr(ld.BwdSite, [bsite(), bsite(db=None)]), 2, 16, FAKE, big, None) == 1
    assert g(arr(ld.BwdSite, [bsite(), bsite(dx=FAKE + 4)]), 2, 16, FAKE, big, None) == 3
    assert g(btwo, 2, 16, FAKE, 1000, None) == 5
    import torch

    if not torch.cuda.is_available():
        # valid arguments reach the device check and fail there: never a CPU computation
        assert f(two, 2, 8, 0, FAKE, big, None) in (6, 7)
        assert g(btwo, 2, 16, FAKE, big, None) in (6, 7)


def test_f32dy_backward_host_checks(lib):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    f = lib.lora_delta_bwd_f32dy
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_float] + [ctypes.c_int64] * 4 + [ctypes.c_void_p] * 5 + \
                 [ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    need = ld.lora_delta_bwd_f32dy_workspace_size(64, 128, 96, 16)
    # the backward's workspace plus the BF16 dV (M x N x 2 bytes, 256-byte rounded)
    assert need == ld.lora_delta_bwd_workspace_size(64, 128, 96, 16) + 64 * 96 * 2
    assert ld.lora_delta_bwd_f32dy_workspace_size(64, 100, 96, 16) == 0
    ok = [FAKE] * 10

    def call(p=ok, M=64, K=128, N=96, R=16, ws=need):
        dy, x, a, b, u, dx, da, db, du, w = p
        return f(dy, x, a, b, u, 2.0, M, K, N, R, dx, da, db, du, w, ws, None)

    assert call(M=0) == 0
    assert call([None] + ok[1:]) == 1
    assert call(K=100) == 2
    assert call(R=12) == 4
    assert call([FAKE + 8] + ok[1:]) == 3
    assert call(ws=need - 256) == 5
    import torch

    if not torch.cuda.is_available():
        assert call() in (6, 7)


def test_exact_mode_host_checks(lib):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    assert ld.lora_delta_exact_slots() == 21
    need = ld.lora_delta_grads_exact_workspace_size(300, 136, 72, 16)
    # segments of the digit kernel: units (64 rows of a 16 x 64 output tile) 3 tiles x 5 = 15 for
    # dA (K = 136), so at most 15 CTAs and 15 + 3 segments; per segment and tile output a 32-byte
    # record and a 21-int64 digit array; the larger gradient's, 256-byte rounded
    assert need == ((18 * 1024 * (32 + 21 * 8) + 255) // 256) * 256
    assert ld.lora_delta_grads_exact_workspace_size(1 << 30, 128, 96, 16) == 0   # M below 2^30
    assert ld.lora_delta_grads_exact_workspace_size(64, 100, 96, 16) == 0
    f = lib.lora_delta_grads_exact
    ok = [FAKE] * 9

    def call(p=ok, M=64, K=128, N=96, R=16, ws=1 << 30):
        dy, x, u, du, da, db, dad, dbd, w = p
        return f(dy, x, u, du, 2.0, M, K, N, R, da, db, dad, dbd, w, ws, None)

    assert call([FAKE] * 4 + [None] * 4 + [FAKE]) == 0          # nothing asked for: a no-op
    assert call([None] + ok[1:]) == 1                            # dB asked for without dy
    assert call(ok[:3] + [None] + ok[4:]) == 1                   # dA asked for without du
    assert call([None, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE]) != 1   # dA alone needs no dy
    assert call(ok[:8] + [None]) == 1                            # workspace
    assert call(K=100) == 2
    assert call(M=1 << 30) == 2
    assert call(R=12) == 4
    assert call(ok[:4] + [FAKE + 4] + ok[5:]) == 3
    assert call(ws=ld.lora_delta_grads_exact_workspace_size(64, 128, 96, 16) - 8) == 5
    assert lib.lora_delta_exact_combine(FAKE, FAKE, -1, FAKE, None) == 2
    assert lib.lora_delta_exact_combine(FAKE, FAKE, 0, FAKE, None) == 0
    assert lib.lora_delta_exact_combine(None, FAKE, 4, FAKE, None) == 1
    assert lib.lora_delta_exact_combine(FAKE, FAKE, 4, None, None) == 1
    assert lib.lora_delta_exact_finalize(FAKE, -1, FAKE, None) == 2
    assert lib.lora_delta_exact_finalize(None, 4, FAKE, None) == 1
    import torch

    if not torch.cuda.is_available():
        assert call() in (6, 7)
        assert call(M=0) in (6, 7)                                # M = 0 still writes zero gradients
        assert lib.lora_delta_exact_finalize(FAKE, 4, FAKE, None) in (6, 7)


def test_exact_f32dy_host_checks(lib):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    f = lib.lora_delta_grads_exact_f32dy
    g = lib.lora_delta_grads_exact_f32dy_workspace_size
    need = int(g(64, 128, 96, 16))
    # the exact pass's scratch plus the BF16 dV (M x N x 2 bytes, 256-byte rounded)
    assert need == ld.lora_delta_grads_exact_workspace_size(64, 128, 96, 16) + 64 * 96 * 2
    assert int(g(64, 100, 96, 16)) == 0
    ok = [FAKE] * 9

    def call(p=ok, M=64, K=128, N=96, R=16, ws=need):
        dy, x, u, du, da, db, dad, dbd, w = p
        return f(dy, x, u, du, 2.0, M, K, N, R, da, db, dad, dbd, w, ws, None)

    assert call([None] + ok[1:]) == 1          # dB asked for without dy
    assert call(ok[:8] + [None]) == 1          # workspace
    assert call(K=100) == 2
    assert call(R=12) == 4
    assert call([FAKE + 4] + ok[1:]) == 3
    assert call(ws=need - 256) == 5
    import torch

    if not torch.cuda.is_available():
        assert call() in (6, 7)


def test_no_base_weight_in_the_signatures():
    """The operator never receives the frozen base weight, so it can neither read nor return a
    gradient for it (page "[DSv4][P5-3] shared_grouped_lora_delta ...", "Acceptance criteria",
    items 2 and 3): the parameters of every compute entry point are the LoRA operands, their
    gradients, shapes, scale, scratch and stream only."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    allowed = {"x", "a", "b", "dy", "u", "du", "alpha", "M", "K", "N", "R", "delta_y", "dx", "da", "db",
               "da_digits", "db_digits", "workspace", "workspace_bytes", "stream", "y_bf16", "sites", "count"}
    for name in ("lora_delta_fwd", "lora_delta_fwd_bf16", "lora_delta_bwd", "lora_delta_bwd_f32dy",
                 "lora_delta_grads_exact", "lora_delta_grads_exact_f32dy", "lora_delta_fwd_noalloc",
                 "lora_delta_fwd_grouped", "lora_delta_bwd_grouped"):
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)", text)
        assert m, name
        params = [re.split(r"[\s*]+", p.strip())[-1] for p in m.group(1).split(",")]
        assert set(params) <= allowed, f"{name}: unexpected parameters {set(params) - allowed}"
    for struct in ("lora_fwd_site", "lora_bwd_site"):
        m = re.search(r"typedef struct " + struct + r"\s*\{(.*?)\}", text, flags=re.S)
        assert m, struct
        fields = re.findall(r"(\w+)\s*;", m.group(1).replace(",", ";"))
        assert set(fields) <= allowed, f"{struct}: unexpected fields {set(fields) - allowed}"


def test_exact_rate_probe_host_checks(lib):
    f = lib.lora_delta_exact_rate_probe
    f.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p]
    f.restype = ctypes.c_int
    n = ctypes.c_int64(0)
    assert f(16, 0x10000, 1 << 20, None, None) == 1            # LORA_ERR_NULL (products)
    assert f(0, 0x10000, 1 << 20, ctypes.byref(n), None) == 2  # LORA_ERR_SHAPE (iters)
    assert f(1 << 31, 0x10000, 1 << 20, ctypes.byref(n), None) == 2
