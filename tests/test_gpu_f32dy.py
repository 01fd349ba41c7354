"""The FP32-dY backward (lora_delta_bwd_f32dy: dV = bf16(fp32(dY * alpha)) with a
binary32 dY) against the BF16-dY backward and the oracle.

* dY values that BF16 holds exactly: every output is bit for bit that of the
  BF16-dY backward on the same values.
* General binary32 dY: dV is the oracle's bit for bit (read out exactly through
  dB with one-hot U rows), and the other outputs are within the tolerances of
  the precision contract against the oracle fed the oracle's dV.
* Sub-batches and reruns are bitwise."""
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


def _bwd(dy, x, a, b, u, alpha):
    M, K = x.shape
    N, R = b.shape
    f32 = dy.dtype == torch.float32
    size = ld.lora_delta_bwd_f32dy_workspace_size if f32 else ld.lora_delta_bwd_workspace_size
    ws = ld.new_workspace(size(M, K, N, R), "cuda")
    out = ld.lora_delta_bwd(dy, x, a, b, u, alpha, workspace=ws)
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == 0
    return out


def _inputs(M, K, N, R, alpha, seed):
    w = S.Workload("f32dy", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 1.0})
    d = w.generate(seed)
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    _, u = ld.lora_delta_fwd(t["x"], t["a"], t["b"], alpha, workspace=ws)
    torch.cuda.synchronize()
    return d, t, u


SHAPES = [(64, 128, 96, 8, 2.0), (300, 264, 136, 16, 0.5), (129, 512, 264, 32, 3.0), (257, 256, 128, 64, 1.5),
          (1000, 96, 2048, 16, 2.0)]


@pytest.mark.parametrize("M,K,N,R,alpha", SHAPES)
def test_bf16_representable_dy_matches_the_bf16_backward(M, K, N, R, alpha):
    d, t, u = _inputs(M, K, N, R, alpha, 3)
    ref = _bwd(t["dy"], t["x"], t["a"], t["b"], u, alpha)
    got = _bwd(t["dy"].float(), t["x"], t["a"], t["b"], u, alpha)
    for name, g, r in zip(("dx", "da", "db", "du"), got, ref):
        G.assert_bitwise(name, g.view(torch.uint8).cpu().numpy(), r.view(torch.uint8).cpu().numpy())


@pytest.mark.parametrize("M,K,N,R,alpha", SHAPES)
def test_general_f32_dy_against_the_oracle(oracle, M, K, N, R, alpha):
    d, t, u = _inputs(M, K, N, R, alpha, 4)
    rng = np.random.default_rng(M + N)
    dy32 = (rng.standard_normal((M, N)) * np.exp2(rng.integers(-8, 8, (M, N)))).astype(np.float32)
    dx, da, db, du = _bwd(torch.from_numpy(dy32).cuda(), t["x"], t["a"], t["b"], u, alpha)
    ub = G.host_bits(u)
    dv = oracle.dv_f32(dy32, alpha)
    ref_du, s_du, f_du = oracle.du(dv, d["b"], want_s=True, want_f32=True)
    G.assert_bf16_close("dU", G.host_bits(du), ref_du, f_du, s_du)
    ref_db, s_db = oracle.db(dv, ub, True)
    G.assert_f32_within("dB", G.host_f32(db), ref_db, s_db)
    ref_dx, s_dx = oracle.dx(G.host_bits(du), d["a"], True)
    G.assert_f32_within("dX", G.host_f32(dx), ref_dx, s_dx)
    ref_da, s_da = oracle.da(G.host_bits(du), d["x"], True)
    G.assert_f32_within("dA", G.host_f32(da), ref_da, s_da)


def test_dv_rounding_is_the_oracles_bit_for_bit(oracle):
    """M = R = 16, U = identity: dB[n][r] = dV[r][n] exactly (one nonzero term), so the GPU's
    dV is read out through dB. dY holds every magnitude, midpoints and the double-rounding case."""
    M = R = 16
    K, N = 64, 512
    alpha = float(np.float32(1 - 2.0 ** -24))
    rng = np.random.default_rng(5)
    dy32 = (rng.standard_normal((M, N)) * np.exp2(rng.integers(-60, 60, (M, N)))).astype(np.float32)
    dy32[0, :4] = [1 + 2.0 ** -8 + 2.0 ** -23, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8 + 2.0 ** -23), 2.0 ** -130]
    u = np.zeros((M, R), np.float64)
    np.fill_diagonal(u, 1.0)
    ub = S.to_bf16_bits(u)
    x = S.to_bf16_bits(rng.standard_normal((M, K)))
    a = S.to_bf16_bits(rng.standard_normal((R, K)) * 0.1)
    b = S.to_bf16_bits(rng.standard_normal((N, R)) * 0.1)
    dx, da, db, du = _bwd(torch.from_numpy(dy32).cuda(), G.dev_bf16(x), G.dev_bf16(a), G.dev_bf16(b), G.dev_bf16(ub),
                          alpha)
    dv = oracle.dv_f32(dy32, alpha)
    got = G.host_f32(db).T                                     # [R][N] = dV
    want = dv.view(np.uint16).astype(np.uint32) << 16          # bf16 bits widened to binary32
    G.assert_bitwise("dV through dB", got.astype(np.float32).view(np.uint32), want.view(np.uint32).astype(np.uint32))


def test_f32_dy_training_shape_subbatches_and_reruns():
    w = S.train()
    d = w.generate(0)
    alpha = w.shape.alpha
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    M, N = w.shape.M, w.shape.N
    g = torch.Generator(device="cuda").manual_seed(3)
    dy32 = torch.randn((M, N), generator=g, device="cuda") * 0.1
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, w.shape.K, N, w.shape.R), "cuda")
    _, u = ld.lora_delta_fwd(t["x"], t["a"], t["b"], alpha, workspace=ws)
    full = _bwd(dy32, t["x"], t["a"], t["b"], u, alpha)
    again = _bwd(dy32, t["x"], t["a"], t["b"], u, alpha)
    for name, g1, g2 in zip(("dx", "da", "db", "du"), full, again):
        G.assert_bitwise(f"rerun {name}", g1.view(torch.uint8).cpu().numpy(), g2.view(torch.uint8).cpu().numpy())
    for s in (1, 100, 4097):
        sl = slice(M - s, M)
        sub = _bwd(dy32[sl].contiguous(), t["x"][sl].contiguous(), t["a"], t["b"], u[sl].contiguous(), alpha)
        G.assert_bitwise(f"sub {s} dx", sub[0].view(torch.uint8).cpu().numpy(), full[0][sl].view(torch.uint8).cpu().numpy())
        G.assert_bitwise(f"sub {s} du", sub[3].view(torch.uint8).cpu().numpy(), full[3][sl].view(torch.uint8).cpu().numpy())
