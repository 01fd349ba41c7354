"""The invariance sweep's power, on the CPU: its probes (sub-batches of 1, 8, 24
and 100 rows at each end of the batch, compared with the same rows of the full
batch; page "[DSv4][P5-3] shared_grouped_lora_delta ...", section "Batch
invariance") must catch a reduction whose order depends on the batch size, at
the production-like sweep shapes, and must pass one whose order does not.

The page's lesson is that an M-dependent kernel went unnoticed at 128 x 64.
Here the M-dependent operator is planted in a CPU stand-in for U = bf16(X A^T)
with FP32 accumulation in an explicit order (a planted mistake lives on the
CPU, never in a GPU build): the stand-in switches from one sequential sum over
K to blocked sums of 256 once the batch has 2048 rows or more. The GPU sweep
(`tests/test_gpu_parity.py::test_invariance_sweep`) applies the same probes to
the real kernels."""
import numpy as np
import pytest

from deterministic_arithmetic_gb300 import synthetic as S


def _u_rows(x, a, batch_rows, m_dependent):
    """bf16 bits of U for the given rows of a batch of `batch_rows` rows: products exact in
    binary64, accumulated in binary32 in a fixed order -- one sequential sum over K, or, for the
    planted mistake with a batch of 2048 rows or more, sequential sums over blocks of 256
    added sequentially."""
    xv = S.bf16_bits_to_f64(x)
    av = S.bf16_bits_to_f64(a)
    prod = (xv[:, None, :] * av[None, :, :]).astype(np.float32)   # [rows][R][K], exact
    K = prod.shape[2]
    if m_dependent and batch_rows >= 2048:
        blocks = [np.add.accumulate(prod[:, :, k0:k0 + 256], axis=2, dtype=np.float32)[:, :, -1]
                  for k0 in range(0, K, 256)]
        acc = np.add.accumulate(np.stack(blocks, axis=2), axis=2, dtype=np.float32)[:, :, -1]
    else:
        acc = np.add.accumulate(prod, axis=2, dtype=np.float32)[:, :, -1]
    return S.to_bf16_bits(acc.astype(np.float64))


def _sweep_finds_a_difference(M, KN, m_dependent, seeds=2):
    w = S.sweep(M, KN)
    for seed in range(seeds):
        d = w.generate(seed, only=("x", "a"))
        for s in [s for s in S.SWEEP_SUBBATCH if s <= M]:
            for rows in (slice(0, s), slice(M - s, M)):
                full = _u_rows(d["x"][rows], d["a"], M, m_dependent)    # those rows of the full batch
                sub = _u_rows(d["x"][rows], d["a"], s, m_dependent)     # the sub-batch on its own
                if not np.array_equal(full, sub):
                    return True
    return False


@pytest.mark.parametrize("M,KN", S.SWEEP_SHAPES)
def test_sweep_catches_an_m_dependent_order(M, KN):
    found = _sweep_finds_a_difference(M, KN, m_dependent=True)
    if M >= 2048:
        assert found, f"the sweep missed an M-dependent accumulation order at M={M}, K=N={KN}"
    else:
        assert not found   # below the switch the planted operator is M-independent


@pytest.mark.parametrize("M,KN", S.SWEEP_SHAPES)
def test_sweep_passes_an_m_independent_order(M, KN):
    assert not _sweep_finds_a_difference(M, KN, m_dependent=False)
