"""The single-launch forward (lora_delta_fwd_fused) against the three launches
of lora_delta_fwd: the same leaves, trees and rounding points, so every output
must agree bit for bit. Inside the launch the steps are ordered by claimed
work and counters in the workspace's control block; the control words must be
zero again after every call, also when the same workspace serves batches of
other shapes. The oracle check of the forward itself is in test_gpu_parity.py
(lora_delta_fwd); here the two schedules are compared with each other."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import lora_delta as ld  # noqa: E402
from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu

CONTROL = 256 + 65536      # LORA_DELTA_CONTROL_BYTES


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()


def _inputs(M, K, N, R, alpha, seed):
    w = S.Workload("fused", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5})
    d = w.generate(seed, only=("x", "a", "b"))
    return {k: G.dev_bf16(v) for k, v in d.items()}


def _both(t, alpha, y_dtype=torch.float32, ws=None):
    M, K = t["x"].shape
    N, R = t["b"].shape
    ws_ref = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda") if ws is None else ws
    y0 = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    y1 = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    y0, u0 = ld.lora_delta_fwd(t["x"], t["a"], t["b"], alpha, delta_y=y0, workspace=ws_ref)
    y1, u1 = ld.lora_delta_fwd_fused(t["x"], t["a"], t["b"], alpha, delta_y=y1, workspace=ws)
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == 0
    assert not ws[:CONTROL].any().item(), "control block not back at zero"
    return (y0, u0), (y1, u1)


def _same(name, ref, got):
    (y0, u0), (y1, u1) = ref, got
    G.assert_bitwise(f"{name}: delta_y", y1.view(torch.uint8).cpu().numpy(), y0.view(torch.uint8).cpu().numpy())
    G.assert_bitwise(f"{name}: u", G.host_bits(u1), G.host_bits(u0))


SHAPES = [  # (M, K, N, R, alpha): every padded rank, ragged M / K / N, one row, many slices per row tile
    (1, 64, 64, 8, 2.0), (7, 136, 96, 16, 0.5), (300, 1032, 520, 24, 0.75), (129, 512, 264, 32, 2.0),
    (257, 4104, 128, 48, 1.5), (600, 2056, 296, 64, 1.0), (1000, 96, 2048, 16, 3.0), (2048, 5120, 1024, 16, 1.0),
]


@pytest.mark.parametrize("M,K,N,R,alpha", SHAPES)
def test_fused_forward_equals_the_three_launches(M, K, N, R, alpha):
    t = _inputs(M, K, N, R, alpha, 11)
    ref, got = _both(t, alpha)
    _same(f"M{M} K{K} N{N} R{R}", ref, got)


@pytest.mark.parametrize("M,K,N,R,alpha", [(300, 1032, 520, 16, 2.0), (129, 512, 264, 64, 0.5)])
def test_fused_forward_bf16_output(M, K, N, R, alpha):
    t = _inputs(M, K, N, R, alpha, 12)
    ref, got = _both(t, alpha, torch.bfloat16)
    _same("bf16 output", ref, got)


def test_fused_forward_training_shape_and_workspace_reuse():
    """The training shape, then batches of other sizes through the same workspace (the control
    words must be back at zero after each call for the next one to be right)."""
    M, K, N, R, alpha = 8192, 4096, 4096, 16, 2.0
    t = _inputs(M, K, N, R, alpha, 13)
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    for m in (M, 1, 4097, 128, M):
        tm = dict(t, x=t["x"][:m])
        ref, got = _both(tm, alpha, ws=ws)
        _same(f"rows {m}", ref, got)


def test_fused_forward_reruns_and_empty_batch():
    t = _inputs(513, 1024, 520, 32, 2.0, 14)
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(513, 1024, 520, 32), "cuda")
    outs = [ld.lora_delta_fwd_fused(t["x"], t["a"], t["b"], 2.0, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for y, u in outs[1:]:
        G.assert_bitwise("rerun delta_y", y.cpu().numpy(), outs[0][0].cpu().numpy())
        G.assert_bitwise("rerun u", G.host_bits(u), G.host_bits(outs[0][1]))
    y, u = ld.lora_delta_fwd_fused(t["x"][:0], t["a"], t["b"], 2.0, workspace=ws)
    assert y.shape == (0, 520) and u.shape == (0, 32)
    assert not ws[:CONTROL].any().item()


@pytest.mark.parametrize("kind,site", [(1, 9), (2, 10)])
def test_fused_forward_wait_that_runs_out(kind, site):
    """The stall test hook (status word 2) in the single launch: the wait runs out, the status
    names the site, every CTA leaves (the control words are back at zero) and the next call on
    the same workspace is right."""
    M, K, N, R = 640, 1024, 2048, 16
    t = _inputs(M, K, N, R, 2.0, 15)
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    words = ws.view(torch.int32)
    words[2] = kind
    words[3] = 1000
    ld.lora_delta_fwd_fused(t["x"], t["a"], t["b"], 2.0, workspace=ws)
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == (site << 8) | 1
    assert not ws[16:CONTROL].any().item()
    words[0] = 0
    words[2] = 0
    words[3] = 0
    ref, got = _both(t, 2.0, ws=ws)
    _same("after a timeout", ref, got)
    assert np.array_equal(ws[:CONTROL].cpu().numpy(), np.zeros(CONTROL, np.uint8))
