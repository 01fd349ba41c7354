"""Failure detection without a GPU fault.

Every wait inside the kernels is bounded; when one runs out, the kernel writes
(site << 8) | 1 into word 0 of the workspace's status block, every role of the
CTA stops working, in-flight copies and tensor-core operations are drained,
TMEM is freed and the kernel returns. Here a test hook in the status block
(word 2: a kernel kind; word 3: a 1 ms wait limit) makes the producer warp of
one kernel wait on an mbarrier that nothing completes, so that wait runs out
in every CTA. The test checks that the call returns, that the status block
names the site, that the CUDA context stays usable, and that the next call on
the same workspaces (hook words and the status word cleared, nothing else
reset) gives bit for bit the results of a call on fresh workspaces.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu

CONTROL = 256 + 65536      # LORA_DELTA_CONTROL_BYTES: status block and control words


# (kernel kind, workspace holding the hook, rank, site of the stall wait)
CASES = [
    (1, "fwd", 16, 9),    # down-projection, U partials
    (2, "fwd", 16, 10),   # up-projection, dY_lora
    (2, "bwd", 16, 10),   # dX expansion
    (3, "bwd", 16, 39),   # fused dU + dB pass
    (4, "bwd", 16, 29),   # dA chunk partials
    (1, "bwd", 32, 9),    # dU partials with the dV transform (ranks above 16)
    (4, "bwd", 32, 29),   # dB / dA chunk partials (ranks above 16)
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()


def _step(t, alpha, wf, wb):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    y, u = ld.lora_delta_fwd(t["x"], t["a"], t["b"], alpha, workspace=wf)
    dx, da, db, du = ld.lora_delta_bwd(t["dy"], t["x"], t["a"], t["b"], u, alpha, workspace=wb)
    torch.cuda.synchronize()
    return dict(y=y, u=u, dx=dx, da=da, db=db, du=du)


@pytest.fixture(params=[0, 1, 2], ids=["separate", "cluster-reduce", "cluster-single"])
def schedule(request):
    """Every schedule of the passes: the separate launches (default), the cluster reductions and
    the single cluster launches (forward R <= 32, backward R <= 16), whose producers honour the same
    stall hooks and sites."""
    from deterministic_arithmetic_gb300 import lora_delta as ld

    ld.lora_delta_set_schedule(request.param, 0)
    yield request.param
    ld.lora_delta_set_schedule(ld.SCHEDULE_AUTO, 0)


@pytest.mark.parametrize("kind,where,R,site", CASES)
def test_a_wait_that_runs_out_is_reported_and_leaves_nothing_behind(kind, where, R, site, schedule):
    from deterministic_arithmetic_gb300 import lora_delta as ld

    M, K, N, alpha = 640, 1024, 2048, 2.0
    w = S.Workload("fail", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 1.0})
    d = w.generate(2)
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    ref = _step(t, alpha, ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda"),
                ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), "cuda"))

    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), "cuda")
    hooked, other = (wf, wb) if where == "fwd" else (wb, wf)
    words = hooked.view(torch.int32)
    words[2] = kind          # stall this kind of kernel
    words[3] = 1000          # after 1 ms
    _step(t, alpha, wf, wb)  # returns: the kernels give up instead of hanging
    assert ld.lora_delta_device_status(hooked) == (site << 8) | 1
    assert ld.lora_delta_device_status(other) == 0
    assert int(hooked.view(torch.int32)[2].item()) == kind     # hook words are read, never written
    assert not hooked[16:CONTROL].any().item()                  # control words back at zero
    assert torch.ones(4, device="cuda").sum().item() == 4.0    # the context is still usable

    words[0] = 0             # the caller reads and clears the code ...
    words[2] = 0             # ... and takes the hooks out; nothing else is reset
    words[3] = 0
    got = _step(t, alpha, wf, wb)
    assert ld.lora_delta_device_status(wf) == 0 and ld.lora_delta_device_status(wb) == 0
    for k in ref:
        G.assert_bitwise(k, got[k].view(torch.uint8).cpu().numpy(), ref[k].view(torch.uint8).cpu().numpy())


def test_control_block_is_zero_after_every_call(schedule):
    """The kernels write status word 0 only, and only on a timeout, and leave the control words
    at zero: after normal calls of several shapes the whole control block is zero."""
    from deterministic_arithmetic_gb300 import lora_delta as ld

    M, K, N, R = 1000, 512, 1024, 16
    w = S.Workload("blk", S.Shape(M, K, N, R, 2.0), {"x": 1.0, "a": K ** -0.5, "b": 0.25, "dy": 1.0})
    t = {k: G.dev_bf16(v) for k, v in w.generate(1).items()}
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), "cuda")
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), "cuda")
    for m in (M, 1, 129, M):
        tm = dict(t, x=t["x"][:m], dy=t["dy"][:m])
        _step(tm, 2.0, wf, wb)
        assert not wf[:CONTROL].any().item() and not wb[:CONTROL].any().item(), m
    assert np.array_equal(wf[:CONTROL].cpu().numpy(), np.zeros(CONTROL, np.uint8))
