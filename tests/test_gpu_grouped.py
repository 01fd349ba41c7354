"""Grouped calls (lora_delta_fwd_grouped / lora_delta_bwd_grouped: several LoRA
sites of one rank in the launches of a single call, page "[DSv4][P5-3]
shared_grouped_lora_delta: CUDA + Triton, both batch-invariant", section
"Summary") against single-site calls: every output of every site must be bit
for bit the single-site call's on the same arguments (which the parity tests
tie to the oracle), whatever the other sites of the group are."""
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


def _site(M, K, N, R, alpha, seed, kind="std"):
    if kind == "ints":
        w = S.integers(M, K, N, R, alpha, bound=2)
    else:
        w = S.Workload("grouped", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 1.0})
    d = w.generate(seed)
    return {k: G.dev_bf16(v) for k, v in d.items()} | {"alpha": alpha}


def _single(s, y_bf16=False):
    M, K = s["x"].shape
    N, R = s["b"].shape
    y = torch.empty((M, N), dtype=torch.bfloat16 if y_bf16 else torch.float32, device="cuda")
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    y, u = ld.lora_delta_fwd(s["x"], s["a"], s["b"], s["alpha"], delta_y=y, workspace=wf)
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), "cuda")
    g = ld.lora_delta_bwd(s["dy"], s["x"], s["a"], s["b"], u, s["alpha"], workspace=wb)
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(wf) == 0 and ld.lora_delta_device_status(wb) == 0
    return (y, u) + tuple(g)


def _grouped(sites, y_bf16=False):
    fw = ld.lora_delta_fwd_grouped([{k: s[k] for k in ("x", "a", "b", "alpha")} for s in sites], y_bf16=y_bf16)
    bw = ld.lora_delta_bwd_grouped([{"dy": s["dy"], "x": s["x"], "a": s["a"], "b": s["b"], "u": u, "alpha": s["alpha"]}
                                    for s, (_, u) in zip(sites, fw)])
    torch.cuda.synchronize()
    return [f + b for f, b in zip(fw, bw)]


NAMES = ("delta_y", "u", "dx", "da", "db", "du")


def _same(tag, got, want):
    for name, g, w in zip(NAMES, got, want):
        G.assert_bitwise(f"{tag}: {name}", g.view(torch.uint8).cpu().numpy(), w.view(torch.uint8).cpu().numpy())


GROUPS = [  # sites (M, K, N, alpha): ragged tails, different shapes and scales in one group
    [(300, 264, 136, 2.0), (129, 512, 264, 0.5)],
    [(64, 128, 96, 2.0), (1000, 96, 2048, 3.0), (7, 136, 96, 1.0)],
    [(513, 1024, 520, 1.0), (2, 4104, 16, 0.25), (257, 256, 128, 1.5), (600, 2056, 296, 2.0)],
]


@pytest.mark.parametrize("R", [8, 16, 32, 64])
@pytest.mark.parametrize("gi", range(len(GROUPS)))
def test_grouped_equals_single_site_calls(R, gi):
    sites = [_site(M, K, N, R, alpha, seed=10 * gi + i) for i, (M, K, N, alpha) in enumerate(GROUPS[gi])]
    want = [_single(s) for s in sites]
    got = _grouped(sites)
    for i, (g, w) in enumerate(zip(got, want)):
        _same(f"R{R} group {gi} site {i}", g, w)


def test_grouped_bf16_output_and_empty_site():
    sites = [_site(300, 264, 136, 16, 2.0, 1), _site(0, 128, 96, 16, 2.0, 2), _site(129, 512, 264, 16, 0.5, 3)]
    live = [sites[0], sites[2]]
    want = [_single(s, y_bf16=True) for s in live]
    fw = ld.lora_delta_fwd_grouped([{k: s[k] for k in ("x", "a", "b", "alpha")} for s in sites], y_bf16=True)
    torch.cuda.synchronize()
    assert fw[1][0].numel() == 0
    for i, (f, w) in zip((0, 2), zip((fw[0], fw[2]), want)):
        _same(f"bf16 site {i}", f, w[:2])


def test_grouped_integer_inputs_equal_the_oracle(oracle):
    """Integer inputs (no sum can round): every site of a group equals the oracle bit for bit."""
    shapes = [(300, 264, 136), (129, 512, 264)]
    ds = [S.integers(M, K, N, 16, 2.0, bound=2).generate(5 + i) for i, (M, K, N) in enumerate(shapes)]
    sites = [{k: G.dev_bf16(v) for k, v in d.items()} | {"alpha": 2.0} for d in ds]
    got = _grouped(sites)
    for i, d in enumerate(ds):
        f = oracle.fwd(d["x"], d["a"], d["b"], 2.0)
        g = oracle.bwd(d["dy"], d["x"], d["a"], d["b"], f["u"], 2.0)
        y, u, dx, da, db, du = got[i]
        G.assert_bitwise(f"site {i} delta_y", G.host_f32(y), f["delta_y"])
        G.assert_bitwise(f"site {i} u", G.host_bits(u), f["u"])
        for name, t in (("dx", dx), ("da", da), ("db", db)):
            G.assert_bitwise(f"site {i} {name}", G.host_f32(t), g[name])
        G.assert_bitwise(f"site {i} du", G.host_bits(du), g["du"])


def test_mlp_fc1_fc2_grouped():
    """The pages' MLP insertion points (fc1 K5120 -> N17408, fc2 K17408 -> N5120, M4096, R16, alpha 1)
    as one group: bitwise the two single-site calls."""
    sites = []
    for w in (S.mlp_fc1(), S.mlp_fc2()):
        d = w.generate(0)
        sites.append({k: G.dev_bf16(v) for k, v in d.items()} | {"alpha": w.shape.alpha})
    want = [_single(s) for s in sites]
    got = _grouped(sites)
    for i, (g, w) in enumerate(zip(got, want)):
        _same(f"mlp site {i}", g, w)
