"""The BF16 dY_lora forward (lora_delta_fwd_bf16, the half-size output asked
for in the review thread of page "[DSv4][P5-3] shared_grouped_lora_delta:
CUDA + Triton, both batch-invariant") against the FP32 forward and the oracle.

Its value is the FP32 dY_lora rounded once more to BF16, so: U is bit for bit
the FP32 forward's, dY_lora bit for bit that forward's FP32 output converted
to BF16 (round to nearest even, torch's conversion), and against the oracle
the BF16 tolerance of the precision contract applies (1 ulp, or the BF16
image of the FP32 band). Sub-batches and reruns are bitwise."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import lora_delta as ld  # noqa: E402
from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()


def _fwd_both(d, alpha, rows=None):
    x = d["x"] if rows is None else d["x"][rows]
    X, A, B = G.dev_bf16(x), G.dev_bf16(d["a"]), G.dev_bf16(d["b"])
    M, K = X.shape
    N, R = B.shape
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    y32, u32 = ld.lora_delta_fwd(X, A, B, alpha, workspace=ws)
    y16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y16, u16 = ld.lora_delta_fwd(X, A, B, alpha, delta_y=y16, workspace=ws)
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == 0
    return dict(y32=y32, y16=y16, u32=G.host_bits(u32), u16=G.host_bits(u16))


def _check_against_fp32(name, r):
    G.assert_bitwise(f"{name}: U", r["u16"], r["u32"])
    G.assert_bitwise(f"{name}: dY_lora", G.host_bits(r["y16"]), G.host_bits(r["y32"].to(torch.bfloat16)))


def _check_against_oracle(name, o, d, alpha, r, rows=slice(None), cols=slice(None)):
    u = r["u16"][rows]
    b = d["b"][cols]
    ref = o.delta_y_bf16(u, b, alpha)
    f32, s = o.delta_y(u, b, alpha, want_s=True)
    G.assert_bf16_close(f"{name}: dY_lora", G.host_bits(r["y16"])[rows][:, cols], ref, f32, s)


CASES = [  # (M, K, N, R, alpha): ragged tails, every padded rank, one-tile and many-tile cases
    (64, 128, 96, 8, 2.0), (7, 136, 96, 16, 0.5), (300, 264, 136, 16, 2.0), (129, 512, 264, 32, 2.0),
    (257, 256, 128, 48, 1.5), (600, 2056, 296, 64, 1.0), (1000, 96, 2048, 16, 3.0), (1, 64, 64, 8, 2.0),
]


@pytest.mark.parametrize("M,K,N,R,alpha", CASES)
def test_bf16_output_matches_fp32_output_and_oracle(oracle, M, K, N, R, alpha):
    w = S.Workload("bf16_out", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 1.0})
    d = w.generate(7)
    r = _fwd_both(d, alpha)
    _check_against_fp32("bf16 out", r)
    _check_against_oracle("bf16 out", oracle, d, alpha, r)


def test_bf16_output_integer_inputs_equal_the_oracle_bitwise(oracle):
    """Small-integer inputs: no sum can round, so the BF16 result is the
    oracle's bit for bit."""
    w = S.integers(300, 264, 136, 16, 2.0, bound=2)
    d = w.generate(5)
    r = _fwd_both(d, 2.0)
    ref = oracle.delta_y_bf16(oracle.u(d["x"], d["a"]), d["b"], 2.0)
    G.assert_bitwise("bf16 out", G.host_bits(r["y16"]), ref)


def test_bf16_output_training_shape(oracle):
    """M=8192, K=N=4096, R=16, alpha=2: against the FP32 forward everywhere,
    sampled rows and columns against the oracle, sub-batches and reruns."""
    w = S.train()
    d = w.generate(0)
    alpha = w.shape.alpha
    r = _fwd_both(d, alpha)
    _check_against_fp32("train", r)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(w.shape.M, 16, replace=False))
    cols = np.sort(rng.choice(w.shape.N, 64, replace=False))
    _check_against_oracle("train", oracle, d, alpha, r, rows=rows, cols=cols)
    y_full = G.host_bits(r["y16"])
    for s in (1, 100, 4097):
        for sl in (slice(0, s), slice(w.shape.M - s, w.shape.M)):
            sub = _fwd_both(d, alpha, rows=sl)
            G.assert_bitwise(f"sub-batch {sl}", G.host_bits(sub["y16"]), y_full[sl])
    again = _fwd_both(d, alpha)
    G.assert_bitwise("rerun", G.host_bits(again["y16"]), y_full)
