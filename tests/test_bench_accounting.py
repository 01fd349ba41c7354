"""The benchmark's byte accounting (the numerator of every roofline fraction it
reports), checked on the CPU against a count made from the operator's tensors:
each tensor counted once per kernel that must stream it, without the bench's
per-kernel split."""
import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def tensor_count(M, K, N, R):
    """Bytes of one forward + backward step (R <= 16 kernels), tensor by tensor."""
    bf, f4 = 2, 4
    x, dy = M * K * bf, M * N * bf                 # inputs streamed from HBM
    a, b = R * K * bf, N * R * bf                  # weights
    u = du = M * R * bf                            # BF16 rows
    dy_lora, dx = M * N * f4, M * K * f4           # FP32 outputs
    da, db = R * K * f4, N * R * f4
    return (2 * x        # down (U) and the dX + dA pass read x
            + dy         # one pass over dY for dU and dB
            + dy_lora + dx
            + 3 * u      # written by the rows, read by up and by the dU + dB pass
            + 2 * du     # written by the rows, read by the dX + dA pass
            + 2 * a      # down and the dX + dA pass
            + 2 * b      # up and the dU + dB pass
            + da + db)   # the combine's outputs


@pytest.mark.parametrize("M,K,N,R", [(8192, 4096, 4096, 16), (4096, 5120, 17408, 16), (4096, 17408, 5120, 8), (1, 64, 64, 16)])
def test_step_bytes_match_a_count_of_the_tensors(bench, M, K, N, R):
    assert bench.step_bytes(M, K, N, R) == tensor_count(M, K, N, R)


def test_training_shape_total(bench):
    # 2 reads of the 64 MiB x, the 64 MiB dY, two 128 MiB FP32 outputs, and 1.3 + 1.0 MB of rows and weights
    assert bench.step_bytes(8192, 4096, 4096, 16) == 472_121_344


def test_every_schedule_moves_the_same_bytes(bench):
    """Each schedule's kernels, with the bytes the bench attributes to them, add up to the
    step total (a fused kernel moves the union of its parts' bytes, counted once)."""
    M, K, N, R = 8192, 4096, 4096, 16
    total = bench.step_bytes(M, K, N, R)
    for _, sched, _, kf, kbw in bench.SCHEDULES:
        f, bw, kb = bench.schedule_kernels(sched, sched, M, K, N, R)
        assert (f, bw) == (kf, kbw)
        assert sum(kb[k] for k in f + bw) == total, sched


def test_traffic_table_names_kernels_of_the_default_step(bench):
    M, K, N, R = 8192, 4096, 4096, 16
    _, _, kb = bench.schedule_kernels(0, 1, M, K, N, R)
    names = set(bench.SCHEDULES[1][3]) | set(bench.SCHEDULES[1][4]) | set(bench.KERNELS_FWD)
    assert set(bench.NCU_TRAFFIC) <= names
    for k, v in bench.NCU_TRAFFIC.items():
        # DRAM traffic of a streaming launch near its algorithmic bytes (no re-reads): below by
        # the evict-first output lines still in L2 at its end (written back during the next
        # launch), above by those of the launch before it and by scratch partials that reach
        # DRAM (the cluster dU + dB pass: 12.6 MB of dU slice and dB chunk partials)
        if kb[k] > 10_000_000:
            assert 0.85 * kb[k] <= v["bytes"] <= 1.25 * kb[k], k
