"""The allocation-free forward entry point (lora_delta_fwd_noalloc).

It is meant for callers that cannot hand the library a workspace because they
may not allocate device memory themselves (for instance code running under an
allocator it does not own). The test calls it through the C ABI, twice in a
row with different inputs, and compares each result with lora_delta_fwd on
the same inputs: the two run the same kernels, so the outputs must agree bit
for bit, the tolerance this suite uses for GPU-to-GPU comparisons.

Kept in a file of its own that sorts last, so a run that stops at the first
failure has run every other test before this one.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib
    from deterministic_arithmetic_gb300 import lora_delta as ld

    build_lib.build()
    lib = ld.library()
    f = lib.lora_delta_fwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float] + [ctypes.c_int64] * 4 + [ctypes.c_void_p] * 3
    f.restype = ctypes.c_int
    lib.lora_delta_fwd_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.lora_delta_fwd_noalloc_status.restype = ctypes.c_int
    return lib


def _noalloc_status(lib):
    code = ctypes.c_int(-1)
    rc = lib.lora_delta_fwd_noalloc_status(ctypes.byref(code))
    return rc, code.value


def _noalloc_fwd(lib, X, A, B, alpha):
    M, K = X.shape
    N, R = B.shape
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=X.device)
    u = torch.zeros((M, R), dtype=torch.bfloat16, device=X.device)
    rc = lib.lora_delta_fwd_noalloc(X.data_ptr(), A.data_ptr(), B.data_ptr(), float(alpha), M, K, N, R,
                                    y.data_ptr(), u.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, f"lora_delta_fwd_noalloc returned {rc}"
    return y, u


def test_noalloc_forward_matches_the_workspace_forward_twice_in_a_row(lib):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    cases = [(S.train(), 0), (S.Workload("ragged", S.Shape(300, 1032, 520, 40, 0.75),
                                         {"x": 1.0, "a": 0.05, "b": 0.2}), 1)]
    for w, seed in cases:                       # two calls in a row, different shapes and inputs
        d = w.generate(seed, only=("x", "a", "b"))
        X, A, B = (G.dev_bf16(d[k]) for k in ("x", "a", "b"))
        y_na, u_na = _noalloc_fwd(lib, X, A, B, w.shape.alpha)
        assert _noalloc_status(lib) == (0, 0)   # no kernel of the call gave up on a wait
        y_ref, u_ref = ld.lora_delta_fwd(X, A, B, w.shape.alpha)
        torch.cuda.synchronize()
        G.assert_bitwise(f"{w.name} delta_y", G.host_f32(y_na), G.host_f32(y_ref))
        G.assert_bitwise(f"{w.name} u", G.host_bits(u_na), G.host_bits(u_ref))


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # M = 2^17 rows at K = 4096, R = 16 needs 32 MiB of partial sums: more than the 16 MiB array.
    # The check happens on the host before any pointer is touched.
    fake = 0x10000
    rc = lib.lora_delta_fwd_noalloc(fake, fake, fake, 1.0, 1 << 17, 4096, 4096, 16, fake, fake, None)
    assert rc == 5                              # LORA_ERR_WORKSPACE
    assert lib.lora_delta_fwd_noalloc(fake, fake, fake, 1.0, 64, 4096, 4096, 12, fake, fake, None) == 4
    assert lib.lora_delta_fwd_noalloc(fake, fake, fake, 1.0, 0, 4096, 4096, 16, fake, fake, None) == 0
