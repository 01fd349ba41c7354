"""The multi-process host path of bench.py (one process per GPU, launched by
torch.distributed.run) on the CPU: two gloo ranks on 127.0.0.1 set up the
process group, meet at the barrier and agree on the max-over-ranks time; the
reference arm's non-zero ranks leave without work. The operator itself has no
exchange step (replicas only), so this is all the N > 1 path of the bench does.
The exact mode's digit arrays compose across ranks by one int64 sum all-reduce
(page "det-train", "API": det_all_reduce); that composition runs here over
gloo on the exact oracle's digit arrays, for 2 and 3 ranks."""
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


def _exact_worker(rank, world, port, q):
    """One rank of a data-parallel exact dB/dA reduction: the digit arrays of this rank's rows
    (computed by the exact oracle: this test runs without a GPU), one int64 sum all-reduce over
    gloo, then normalised -- the composition of the det-train page's det_all_reduce."""
    import sys

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch.distributed as dist

    from oracle.exact_mode import ExactOracle
    from deterministic_arithmetic_gb300 import synthetic as S

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    rng = np.random.default_rng(7)
    M, P, Q = 37, 3, 5
    left = S.to_bf16_bits(rng.standard_normal((M, P)) * np.exp2(rng.integers(-30, 30, (M, P))))
    right = S.to_bf16_bits(rng.standard_normal((M, Q)) * np.exp2(rng.integers(-30, 30, (M, Q))))
    eo = ExactOracle()
    cuts = np.linspace(0, M, world + 1).astype(int)
    mine = eo.digits(left[cuts[rank]:cuts[rank + 1]], right[cuts[rank]:cuts[rank + 1]])
    t = torch.from_numpy(mine.copy())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    summed = eo.combine(t.numpy(), np.zeros_like(t.numpy())).reshape(mine.shape)
    whole = eo.digits(left, right)
    dist.destroy_process_group()
    q.put((rank, bool(np.array_equal(summed, whole)),
           bool(np.array_equal(eo.finalize(summed).view(np.uint32), eo.exact_matmul(left, right).view(np.uint32)))))


@pytest.mark.parametrize("world", [2, 3])
def test_exact_digit_arrays_all_reduce_across_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exact_worker, args=(i, world, port, q)) for i in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == list(range(world))
    assert all(r[1] and r[2] for r in res), res
