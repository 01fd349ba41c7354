"""The GPU's FP32 reduction order, bit for bit, against the CPU model of the
canonical tree (oracle/tree_order.py).

The inputs hold one non-zero product per 16-term leaf, so every leaf is an
exact product and the result is fixed by the order in which the leaves are
added. Large leaves cancel in pairs placed far apart on the reduction axis
(leaf j against leaf L-1-j), so the partial sums are far larger than the final
sum and any other order changes the rounding of most outputs: U and dU (BF16,
their sums over K and N run through the slice partials and the rows kernels,
one-thread and four-lane), dA and dB (FP32, their sums over the batch run
through 256-row chunks and the combine kernel). Every comparison is bitwise
(+0 and -0 equal). delta_y and dX reduce over R, a single leaf or a few, whose
internal rounding the model does not cover: their parity is in
test_gpu_parity.py."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import lora_delta as ld  # noqa: E402
from oracle import tree_order as T  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()


def _bf16_values(rng, shape, lo, hi):
    """Random BF16-exact values: sign * 2^e * (1 + i/128), e in [lo, hi]."""
    sign = rng.choice(np.float32([-1.0, 1.0]), shape)
    return (sign * np.exp2(rng.integers(lo, hi + 1, shape)) * (1 + rng.integers(0, 128, shape) / 128)).astype(np.float32)


def _sparse_operand(rng, rows, T_len, shift):
    """(rows, T_len): row m holds one non-zero at offset (7 m + j + shift) mod 16 of each leaf j
    (none where that falls past T_len). So along the other axis each 16-row block of a column
    holds exactly one non-zero too (7 is invertible mod 16). Leaves j < L/2 are mostly large
    values whose mirror leaf L-1-j holds the same value negated; the rest are small."""
    L = T.leaf_count(T_len)
    j = np.arange(L)
    m = np.arange(rows)[:, None]
    k = 16 * j[None, :] + (7 * m + j[None, :] + shift) % 16
    vals = _bf16_values(rng, (rows, L), -6, -2)                # small by default
    half = L // 2
    big = rng.random((rows, half)) < 0.75
    bigv = _bf16_values(rng, (rows, half), 4, 10)
    vals[:, :half] = np.where(big, bigv, vals[:, :half])
    mirror = L - 1 - np.arange(half)
    vals[:, mirror] = np.where(big, -bigv, vals[:, mirror])
    out = np.zeros((rows, L * 16), np.float32)
    np.put_along_axis(out, k, vals, axis=1)
    return out[:, :T_len]


def _leaf_weights(rng, R, T_len):
    """(R, T_len) positive BF16 values, constant over each leaf and mirror-symmetric in the leaf
    index, so a cancelling pair of the sparse operand cancels in every column."""
    L = T.leaf_count(T_len)
    w = np.exp2(rng.integers(-2, 3, (R, L))) * (1 + rng.integers(0, 128, (R, L)) / 128)
    w = np.where(np.arange(L)[None, :] < L // 2, w, w[:, ::-1])
    return np.repeat(w, 16, axis=1)[:, :T_len].astype(np.float32)


def _to_dev(v):
    return torch.from_numpy(np.ascontiguousarray(v)).to("cuda").to(torch.bfloat16)


def _case(M, K, N, R, alpha, seed):
    rng = np.random.default_rng(seed)
    x = _sparse_operand(rng, M, K, 0)
    a = _leaf_weights(rng, R, K)
    dy = _sparse_operand(rng, M, N, 3)
    b = _leaf_weights(rng, R, N).T.copy()
    return dict(x=x, a=a, dy=dy, b=b, alpha=alpha)


def _model(c):
    """U, dU (BF16 bits) and dA, dB (FP32) as the canonical tree adds them."""
    u_bits = T.rnbf_bits(T.tree_matmul_f32(c["x"], c["a"]))
    u = T.bf16_value(u_bits)
    dv = (c["dy"] * np.float32(c["alpha"])).astype(np.float32)    # power-of-two alpha: exact, BF16
    assert np.array_equal(T.bf16_value(T.rnbf_bits(dv)), dv)
    du_bits = T.rnbf_bits(T.tree_matmul_f32(dv, c["b"].T))
    du = T.bf16_value(du_bits)
    db = T.tree_matmul_f32(dv.T, u.T)
    da = T.tree_matmul_f32(du.T, c["x"].T)
    return dict(u=u_bits, du=du_bits, da=da, db=db)


def _dev_inputs(c):
    return {k: _to_dev(c[k]) for k in ("x", "a", "dy", "b")}


def _check(name, got, want):
    if want.dtype == np.uint16:
        bad = G.bf16_ulp_distance(got, want) != 0
    else:
        bad = ~((got == want) | (np.isnan(got) & np.isnan(want)))
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {bad.size} differ from the canonical tree; "
                           f"first at {np.argwhere(bad)[0].tolist()}")


def _sensitivity(c, want):
    """The inputs must make the order matter: adding the same leaves left to right changes
    most of U (else the test would not tell orders apart)."""
    leaves = T.single_product_leaves(c["x"], c["a"])
    seq = np.zeros(leaves.shape[1:], np.float32)
    for leaf in leaves:
        seq = seq + leaf
    return float(np.mean(T.rnbf_bits(seq) != want["u"]))


CASES = [  # (M, K, N, R): slices of U / dU per row (rows kernel), leaves of dA / dB over the batch
    (1035, 17408, 17408, 16),   # U 17 slices, dU 34 slices (four-lane rows); 65 row leaves, ragged
    (520, 17400, 17208, 16),    # ragged K and N: partial last leaf and slice
    (272, 17408, 4096, 64),     # R 64: 68 U slices and 16 dU slices of 256
    (520, 4096, 4096, 16),      # 4 U slices, 8 dU slices (one-thread rows)
    (300, 8200, 2056, 32),      # 9 U slices (one partial block of 8), 3 dU slices
]


@pytest.mark.parametrize("M,K,N,R", CASES)
def test_reduction_order_is_the_canonical_tree(M, K, N, R):
    c = _case(M, K, N, R, 2.0, M + K + N + R)
    want = _model(c)
    assert _sensitivity(c, want) > 0.1
    t = _dev_inputs(c)
    y, u = ld.lora_delta_fwd(t["x"], t["a"], t["b"], c["alpha"])
    dx, da, db, du = ld.lora_delta_bwd(t["dy"], t["x"], t["a"], t["b"], u, c["alpha"])
    torch.cuda.synchronize()
    _check("u", G.host_bits(u), want["u"])
    _check("du", G.host_bits(du), want["du"])
    _check("da", G.host_f32(da), want["da"])
    _check("db", G.host_f32(db), want["db"])


def test_grouped_sites_mixing_few_and_many_slices():
    """fc1- and fc2-like sites in one grouped call: U with 5 and 17 slices, dU with 34 and 10, so
    the rows kernel of one launch sums sites with at most 8 and with more than 8 slices."""
    M, R = 520, 16
    cs = [_case(M, 5120, 17408, R, 2.0, 101), _case(M, 17408, 5120, R, 2.0, 102)]
    wants = [_model(c) for c in cs]
    ts = [_dev_inputs(c) for c in cs]
    fwd = ld.lora_delta_fwd_grouped([dict(x=t["x"], a=t["a"], b=t["b"], alpha=2.0) for t in ts])
    bwd = ld.lora_delta_bwd_grouped([dict(dy=t["dy"], x=t["x"], a=t["a"], b=t["b"], u=u, alpha=2.0)
                                     for t, (_, u) in zip(ts, fwd)])
    torch.cuda.synchronize()
    for i, (want, (_, u), (dx, da, db, du)) in enumerate(zip(wants, fwd, bwd)):
        _check(f"site {i} u", G.host_bits(u), want["u"])
        _check(f"site {i} du", G.host_bits(du), want["du"])
        _check(f"site {i} da", G.host_f32(da), want["da"])
        _check(f"site {i} db", G.host_f32(db), want["db"])


def test_bf16_output_and_fused_forward_give_the_same_u():
    """The BF16-output forward and the single-launch forward form U by the same tree."""
    c = _case(272, 17408, 2048, 16, 2.0, 7)
    want = _model(c)
    t = _dev_inputs(c)
    yb = torch.empty((272, 2048), dtype=torch.bfloat16, device="cuda")
    _, u1 = ld.lora_delta_fwd(t["x"], t["a"], t["b"], 2.0, delta_y=yb)
    _, u2 = ld.lora_delta_fwd_fused(t["x"], t["a"], t["b"], 2.0)
    torch.cuda.synchronize()
    _check("u (bf16 output)", G.host_bits(u1), want["u"])
    _check("u (fused)", G.host_bits(u2), want["u"])
