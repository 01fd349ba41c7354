"""The multi-process host path of bench.py (one process per GPU, launched by
torch.distributed.run) on the CPU: two gloo ranks on 127.0.0.1 set up the
process group, meet at the barrier and agree on the max-over-ranks time; the
reference arm's non-zero ranks leave without work. The operator itself has no
exchange step (replicas only), so this is all the N > 1 path does."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    import bench

    w, r, local = bench.dist_setup()
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 * (rank + 1), w)
    # the reference arm: only rank 0 measures and prints
    class _Args:
        steps, warmup, gpus, reference_budget_s = 1, 0, world, 1.0
    out = bench.run_reference(_Args, w, r) if r != 0 else "skipped"
    bench.barrier(w)
    torch.distributed.destroy_process_group()
    q.put((r, w, local, m, out))


def test_two_gloo_ranks_share_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(i, 2, port, q)) for i in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == r[0] for r in res)
    assert all(r[3] == 3.0 for r in res)          # max over ranks of 1.5 and 3.0
    assert res[1][4] is None                       # rank 1 of the reference arm returns at once
