"""The schedules on thread-block clusters (lora_delta_set_schedule: the cluster
reductions, and the single cluster launches) against the separate launches: the
same leaves, trees and rounding points, so every output of the forward (U,
dY_lora) and of the backward (dU, dX, dA, dB) must agree bit for bit, whatever
the schedule and the cluster size. The cluster's CTAs exchange
slice partials through the workspace and meet at mbarriers in each other's
shared memory; the control block must be untouched afterwards. The separate
launches, the default schedule, are checked against the oracle in
test_gpu_parity.py; the stall hooks of the cluster backward are exercised by
test_gpu_failure.py with the cluster launches selected."""
import contextlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import lora_delta as ld  # noqa: E402
from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu

CONTROL = 256 + 65536      # LORA_DELTA_CONTROL_BYTES
SEP, RED, ONE, AUTO = ld.SCHEDULE_SEPARATE, ld.SCHEDULE_CLUSTER_REDUCE, ld.SCHEDULE_CLUSTER_SINGLE, ld.SCHEDULE_AUTO
# (schedule, cluster size) pairs compared with the separate launches
VARIANTS = [(RED, 2), (RED, 4), (RED, 8), (ONE, 2), (ONE, 4), (ONE, 8), (AUTO, 0)]


@contextlib.contextmanager
def schedule(sched, cl=0):
    ld.lora_delta_set_schedule(sched, cl)
    try:
        yield
    finally:
        ld.lora_delta_set_schedule(AUTO, 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()
    yield
    ld.lora_delta_set_schedule(AUTO, 0)


def _inputs(M, K, N, R, alpha, seed):
    w = S.Workload("cluster", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5})
    d = w.generate(seed, only=("x", "a", "b"))
    return {k: G.dev_bf16(v) for k, v in d.items()}


def _fwd(t, alpha, sv, y_dtype=torch.float32, ws=None):
    M, K = t["x"].shape
    N, R = t["b"].shape
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda") if ws is None else ws
    y = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    u = torch.full((M, R), float("nan"), dtype=torch.bfloat16, device="cuda")
    with schedule(*sv):
        y, u = ld.lora_delta_fwd(t["x"], t["a"], t["b"], alpha, delta_y=y, u=u, workspace=ws)   # BF16 y: _bf16
        torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == 0
    assert not ws[:CONTROL].any().item(), "control block not at zero"
    return y, u


def _same(name, ref, got):
    (y0, u0), (y1, u1) = ref, got
    G.assert_bitwise(f"{name}: delta_y", y1.view(torch.uint8).cpu().numpy(), y0.view(torch.uint8).cpu().numpy())
    G.assert_bitwise(f"{name}: u", G.host_bits(u1), G.host_bits(u0))


SHAPES = [  # (M, K, N, R, alpha): padded ranks 16 and 32, ragged M / K / N, one row, fewer slices or
    # column tiles than CTAs in a cluster, more slices than CTAs, many row tiles per cluster
    (1, 64, 64, 8, 2.0), (7, 136, 96, 16, 0.5), (300, 1032, 520, 24, 0.75), (129, 512, 264, 32, 2.0),
    (257, 4104, 128, 16, 1.5), (1000, 96, 2048, 16, 3.0), (2048, 5120, 1024, 16, 1.0),
    (640, 17408, 392, 32, 0.5), (9000, 1024, 1032, 8, 2.0),
]


@pytest.mark.parametrize("M,K,N,R,alpha", SHAPES)
def test_cluster_forward_equals_the_separate_launches(M, K, N, R, alpha):
    t = _inputs(M, K, N, R, alpha, 21)
    ref = _fwd(t, alpha, (SEP, 0))
    for sv in VARIANTS:
        _same(f"M{M} K{K} N{N} R{R} schedule {sv}", ref, _fwd(t, alpha, sv))


@pytest.mark.parametrize("M,K,N,R,alpha", [(300, 1032, 520, 16, 2.0), (129, 512, 264, 32, 0.5)])
def test_cluster_forward_bf16_output(M, K, N, R, alpha):
    t = _inputs(M, K, N, R, alpha, 22)
    ref = _fwd(t, alpha, (SEP, 0), torch.bfloat16)
    for sv in ((RED, 4), (ONE, 2), (ONE, 4)):
        _same(f"bf16 output, schedule {sv}", ref, _fwd(t, alpha, sv, torch.bfloat16))


def test_cluster_forward_training_shape_and_workspace_reuse():
    """The training shape, then batches of other sizes through the same workspace."""
    M, K, N, R, alpha = 8192, 4096, 4096, 16, 2.0
    t = _inputs(M, K, N, R, alpha, 23)
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    for m in (M, 1, 4097, 128, M):
        tm = dict(t, x=t["x"][:m])
        ref = _fwd(tm, alpha, (SEP, 0))
        for sv in ((RED, 0), (ONE, 0)):
            _same(f"rows {m} schedule {sv}", ref, _fwd(tm, alpha, sv, ws=ws))


def test_cluster_forward_reruns_and_empty_batch():
    t = _inputs(513, 1024, 520, 32, 2.0, 24)
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(513, 1024, 520, 32), "cuda")
    with schedule(ONE):
        outs = [ld.lora_delta_fwd(t["x"], t["a"], t["b"], 2.0, workspace=ws) for _ in range(3)]
        torch.cuda.synchronize()
        y0, u0 = ld.lora_delta_fwd(t["x"][:0], t["a"], t["b"], 2.0, workspace=ws)
    for y, u in outs[1:]:
        G.assert_bitwise("rerun delta_y", y.cpu().numpy(), outs[0][0].cpu().numpy())
        G.assert_bitwise("rerun u", G.host_bits(u), G.host_bits(outs[0][1]))
    assert y0.shape == (0, 520) and u0.shape == (0, 32)
    assert not ws[:CONTROL].any().item()


def test_schedule_setting():
    assert ld.lora_delta_schedule() == (AUTO, 0)      # the automatic choice by default
    for bad in ((4, 0), (-1, 0), (RED, 1), (ONE, 3), (ONE, 16)):
        with pytest.raises(ld.LoraDeltaError):
            ld.lora_delta_set_schedule(*bad)
    assert ld.lora_delta_schedule() == (AUTO, 0)
    with schedule(RED, 8):
        assert ld.lora_delta_schedule() == (RED, 8)
    assert ld.lora_delta_schedule() == (AUTO, 0)


@pytest.mark.parametrize("sched", [RED, ONE])
@pytest.mark.parametrize("kind,site", [(1, 9), (2, 10)])
def test_cluster_forward_wait_that_runs_out(kind, site, sched):
    """The stall test hook (status word 2): the X / A producer (kind 1) or the b producer (kind 2)
    waits on a barrier that nothing completes; the wait runs out, the status names the site, the
    peers' waits for the stalled CTA give up too, every CTA leaves, and the next call on the same
    workspace (hook and status words cleared, nothing else reset) is right."""
    M, K, N, R = 640, 1024, 2048, 16
    t = _inputs(M, K, N, R, 2.0, 25)
    ws = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    words = ws.view(torch.int32)
    words[2] = kind
    words[3] = 1000
    with schedule(sched):
        ld.lora_delta_fwd(t["x"], t["a"], t["b"], 2.0, workspace=ws)
        torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == (site << 8) | 1
    assert not ws[16:CONTROL].any().item()
    assert torch.ones(4, device="cuda").sum().item() == 4.0    # the context is still usable
    words[0] = 0
    words[2] = 0
    words[3] = 0
    _same("after a timeout", _fwd(t, 2.0, (SEP, 0)), _fwd(t, 2.0, (sched, 0), ws=ws))
    assert np.array_equal(ws[:CONTROL].cpu().numpy(), np.zeros(CONTROL, np.uint8))


# ------------------------------------------------------------------ backward
def _bwd_inputs(M, K, N, R, alpha, seed):
    w = S.Workload("cluster-bwd", S.Shape(M, K, N, R, alpha),
                   {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 0.1})
    d = w.generate(seed)
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    _, t["u"] = ld.lora_delta_fwd(t["x"], t["a"], t["b"], alpha)
    return t


def _bwd(t, alpha, sv, ws=None):
    M, K = t["x"].shape
    N, R = t["b"].shape
    ws = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), "cuda") if ws is None else ws
    outs = dict(dx=torch.full((M, K), float("nan"), device="cuda"), da=torch.full((R, K), float("nan"), device="cuda"),
                db=torch.full((N, R), float("nan"), device="cuda"),
                du=torch.full((M, R), float("nan"), dtype=torch.bfloat16, device="cuda"))
    with schedule(*sv):
        dx, da, db, du = ld.lora_delta_bwd(t["dy"], t["x"], t["a"], t["b"], t["u"], alpha, workspace=ws, **outs)
        torch.cuda.synchronize()
    assert ld.lora_delta_device_status(ws) == 0
    assert not ws[:CONTROL].any().item(), "control block not at zero"
    return dict(dx=dx, da=da, db=db, du=du)


def _same_bwd(name, ref, got):
    for k in ("dx", "da", "db"):
        G.assert_bitwise(f"{name}: {k}", got[k].view(torch.uint8).cpu().numpy(), ref[k].view(torch.uint8).cpu().numpy())
    G.assert_bitwise(f"{name}: du", G.host_bits(got["du"]), G.host_bits(ref["du"]))


BWD_SHAPES = [  # (M, K, N, R, alpha): R 8 and 16, ragged M / K / N, one row, chunks with one row tile,
    # fewer slices / column tiles than CTAs, more chunks than clusters, non-power-of-two alpha
    (1, 64, 64, 8, 2.0), (7, 136, 96, 16, 0.5), (300, 1032, 520, 16, 0.75), (129, 512, 264, 8, 2.0),
    (257, 4104, 136, 16, 1.5), (1000, 96, 2048, 16, 3.0), (2048, 5120, 1024, 16, 1.0),
    (640, 1024, 17408, 16, 0.5), (12000, 1032, 1024, 16, 2.0),
    # more than 8 dU slices with 256-row units (four lanes per value in the rows step; clusters
    # of 4 and 8, and the automatic schedule, take 256-row units here, clusters of 2 128-row ones)
    (7500, 256, 4616, 16, 2.0),
]


@pytest.mark.parametrize("M,K,N,R,alpha", BWD_SHAPES)
def test_cluster_backward_equals_the_separate_launches(M, K, N, R, alpha):
    t = _bwd_inputs(M, K, N, R, alpha, 31)
    ref = _bwd(t, alpha, (SEP, 0))
    for sv in VARIANTS:
        _same_bwd(f"M{M} K{K} N{N} R{R} schedule {sv}", ref, _bwd(t, alpha, sv))


def test_cluster_backward_training_shape_and_workspace_reuse():
    M, K, N, R, alpha = 8192, 4096, 4096, 16, 2.0
    t = _bwd_inputs(M, K, N, R, alpha, 32)
    ws = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), "cuda")
    for m in (M, 1, 4097, 256, M):
        tm = dict(t, x=t["x"][:m], dy=t["dy"][:m], u=t["u"][:m])
        ref = _bwd(tm, alpha, (SEP, 0))
        for sv in ((RED, 0), (ONE, 0)):
            _same_bwd(f"rows {m} schedule {sv}", ref, _bwd(tm, alpha, sv, ws=ws))


def test_cluster_backward_reruns():
    t = _bwd_inputs(1500, 2048, 1032, 16, 2.0, 33)
    ws = ld.new_workspace(ld.lora_delta_bwd_workspace_size(1500, 2048, 1032, 16), "cuda")
    for sv in ((RED, 0), (ONE, 0)):
        ref = _bwd(t, 2.0, sv, ws=ws)
        for _ in range(2):
            _same_bwd(f"rerun {sv}", ref, _bwd(t, 2.0, sv, ws=ws))


def test_launch_plan():
    """lora_delta_plan reports the schedule a call takes and its launch count: the automatic
    schedule keeps the forward's separate launches and takes the backward's cluster reductions
    where its 256-row chunks give at least three quarters of the SMs a CTA."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    big = 256 * ((3 * nsm + 15) // 16) + 256     # enough 256-row chunks for clusters of 4
    assert ld.lora_delta_plan(False, 8192, 4096, 4096, 16) == (SEP, 3)
    assert ld.lora_delta_plan(True, big, 4096, 4096, 16) == (RED, 3)
    assert ld.lora_delta_plan(True, 256, 4096, 4096, 16) == (SEP, 4)
    assert ld.lora_delta_plan(True, 4096, 5120, 17408, 16) == (SEP, 4)     # too few 256-row chunks
    assert ld.lora_delta_plan(True, big, 4096, 4096, 32) == (SEP, 6)       # rank above 16: separate
    assert ld.lora_delta_plan(False, 0, 4096, 4096, 16) == (SEP, 0)
    with schedule(ONE, 4):
        assert ld.lora_delta_plan(False, 8192, 4096, 4096, 32) == (ONE, 1)
        assert ld.lora_delta_plan(False, 8192, 4096, 4096, 64) == (SEP, 3)   # rank above 32: separate
        assert ld.lora_delta_plan(True, 300, 1032, 520, 16) == (ONE, 2)
    with schedule(RED, 2):
        assert ld.lora_delta_plan(False, 8192, 4096, 4096, 16) == (RED, 2)
        assert ld.lora_delta_plan(True, 8192, 4096, 4096, 16) == (RED, 3)
        assert ld.lora_delta_plan(True, 8192, 4096, 1 << 20, 16) == (SEP, 4)   # a CTA's share too large
    with pytest.raises(ld.LoraDeltaError):
        ld.lora_delta_plan(True, 8192, 4095, 4096, 16)                      # K not a multiple of 8
