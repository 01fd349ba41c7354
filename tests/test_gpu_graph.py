"""The C ABI under CUDA-graph capture and on concurrent streams.

Every call only enqueues kernels on the caller's stream (no synchronisation,
allocation or host read of device data), so a training framework can capture
it in a CUDA graph and replay it with new input contents in the same buffers.
A replay must give the bits of an eager call on those inputs. Two independent
problems on two streams, each with its own workspace, must give the bits of the
same calls made one after the other."""
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


def _inputs(M, K, N, R, seed):
    w = S.Workload("graph", S.Shape(M, K, N, R, 2.0), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 0.1})
    return {k: G.dev_bf16(v) for k, v in w.generate(seed).items()}


class Buffers:
    """Inputs, outputs and workspaces of one fwd + bwd, allocated once (as a captured graph needs)."""

    def __init__(self, M, K, N, R):
        dev = "cuda"
        bf, f4 = torch.bfloat16, torch.float32
        self.x, self.dy = torch.empty((M, K), dtype=bf, device=dev), torch.empty((M, N), dtype=bf, device=dev)
        self.a, self.b = torch.empty((R, K), dtype=bf, device=dev), torch.empty((N, R), dtype=bf, device=dev)
        self.y, self.u = torch.empty((M, N), dtype=f4, device=dev), torch.empty((M, R), dtype=bf, device=dev)
        self.dx, self.da = torch.empty((M, K), dtype=f4, device=dev), torch.empty((R, K), dtype=f4, device=dev)
        self.db, self.du = torch.empty((N, R), dtype=f4, device=dev), torch.empty((M, R), dtype=bf, device=dev)
        self.wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M, K, N, R), dev)
        self.wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M, K, N, R), dev)

    def load(self, t):
        for k in ("x", "dy", "a", "b"):
            getattr(self, k).copy_(t[k])

    def step(self, stream, fused=False):
        fwd = ld.lora_delta_fwd_fused if fused else ld.lora_delta_fwd
        fwd(self.x, self.a, self.b, 2.0, delta_y=self.y, u=self.u, workspace=self.wf, stream=stream)
        ld.lora_delta_bwd(self.dy, self.x, self.a, self.b, self.u, 2.0, dx=self.dx, da=self.da, db=self.db, du=self.du,
                          workspace=self.wb, stream=stream)

    def outputs(self):
        return {k: getattr(self, k).view(torch.uint8).cpu().numpy().copy() for k in ("y", "u", "dx", "da", "db", "du")}


def _eager(t, M, K, N, R, fused=False):
    b = Buffers(M, K, N, R)
    b.load(t)
    b.step(torch.cuda.current_stream(), fused)
    torch.cuda.synchronize()
    return b.outputs()


def _same(name, got, want):
    for k in want:
        G.assert_bitwise(f"{name}: {k}", got[k], want[k])


@pytest.mark.parametrize("M,K,N,R,fused", [(300, 1032, 520, 16, False), (513, 2048, 4096, 32, False),
                                           (640, 1024, 2048, 16, True)])
def test_graph_replay_equals_eager_calls(M, K, N, R, fused):
    buf = Buffers(M, K, N, R)
    inputs = [_inputs(M, K, N, R, s) for s in (21, 22)]
    buf.load(inputs[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        buf.step(side, fused)                      # warm-up outside the capture (first-call set-up)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        buf.step(torch.cuda.current_stream(), fused)
    for i, t in enumerate(inputs + inputs[:1]):    # new contents in the captured buffers, then the first again
        buf.load(t)
        graph.replay()
        torch.cuda.synchronize()
        assert ld.lora_delta_device_status(buf.wf) == 0 and ld.lora_delta_device_status(buf.wb) == 0
        _same(f"replay {i}", buf.outputs(), _eager(t, M, K, N, R, fused))


def test_grouped_calls_in_a_graph():
    M, R = 257, 16
    shapes = [(1032, 2056), (2056, 1032)]
    ts = [_inputs(M, K, N, R, 30 + i) for i, (K, N) in enumerate(shapes)]
    dev = "cuda"
    outs = [dict(y=torch.empty((M, N), dtype=torch.float32, device=dev), u=torch.empty((M, R), dtype=torch.bfloat16, device=dev),
                 dx=torch.empty((M, K), dtype=torch.float32, device=dev), da=torch.empty((R, K), dtype=torch.float32, device=dev),
                 db=torch.empty((N, R), dtype=torch.float32, device=dev), du=torch.empty((M, R), dtype=torch.bfloat16, device=dev))
            for K, N in shapes]
    fw = [dict(x=t["x"], a=t["a"], b=t["b"], alpha=2.0, delta_y=o["y"], u=o["u"]) for t, o in zip(ts, outs)]
    bw = [dict(dy=t["dy"], x=t["x"], a=t["a"], b=t["b"], u=o["u"], alpha=2.0, dx=o["dx"], da=o["da"], db=o["db"],
               du=o["du"]) for t, o in zip(ts, outs)]
    wf = ld.new_workspace(64 << 20, dev)
    wb = ld.new_workspace(64 << 20, dev)

    def step(stream):
        ld.lora_delta_fwd_grouped(fw, workspace=wf, stream=stream)
        ld.lora_delta_bwd_grouped(bw, workspace=wb, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = [{k: v.view(torch.uint8).cpu().numpy().copy() for k, v in o.items()} for o in outs]
    for o in outs:
        for v in o.values():
            v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(torch.cuda.current_stream())
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert ld.lora_delta_device_status(wf) == 0 and ld.lora_delta_device_status(wb) == 0
    for i, (o, w) in enumerate(zip(outs, want)):
        _same(f"site {i}", {k: v.view(torch.uint8).cpu().numpy() for k, v in o.items()}, w)


def test_two_streams_two_workspaces():
    shapes = [(513, 2048, 1032, 16), (300, 1032, 4096, 64)]
    ts = [_inputs(*sh, 40 + i) for i, sh in enumerate(shapes)]
    want = [_eager(t, *sh) for t, sh in zip(ts, shapes)]
    bufs = [Buffers(*sh) for sh in shapes]
    for b, t in zip(bufs, ts):
        b.load(t)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):                              # interleaved enqueues on the two streams
        for b, s in zip(bufs, streams):
            with torch.cuda.stream(s):
                b.step(s)
    torch.cuda.synchronize()
    for i, (b, w) in enumerate(zip(bufs, want)):
        assert ld.lora_delta_device_status(b.wf) == 0 and ld.lora_delta_device_status(b.wb) == 0
        _same(f"stream {i}", b.outputs(), w)
    assert np.array_equal(bufs[0].wf[:256 + 65536].cpu().numpy(), np.zeros(256 + 65536, np.uint8))
