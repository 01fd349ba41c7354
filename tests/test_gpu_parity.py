"""CUDA path (through the C ABI) against the CPU oracle, batch invariance and
reruns. Every test here needs a GB300 and the built library."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
import gpu_util as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()


def _rows_of(out, rows):
    return {k: (v[rows] if k in ("u", "delta_y", "du", "dx") else v) for k, v in out.items()}


# ------------------------------------------------------------------ parity
def test_tiny_parity(oracle):
    w = S.tiny()
    d = w.generate(0)
    out = G.run(d, w.shape.alpha)
    G.check_parity(oracle, d, w.shape.alpha, out)


@pytest.mark.parametrize("M,K,N,R", [(64, 128, 96, 8), (300, 264, 136, 16), (513, 1024, 520, 32), (129, 200, 72, 64)])
def test_integer_inputs_are_bitwise_equal_to_the_oracle(oracle, M, K, N, R):
    """Small-integer inputs keep every partial sum exact, so no summation order
    can round: the GPU must equal the oracle bit for bit at every boundary."""
    w = S.integers(M, K, N, R, 2.0, bound=2)
    d = w.generate(5)
    out = G.run(d, 2.0)
    f = oracle.fwd(d["x"], d["a"], d["b"], 2.0)
    g = oracle.bwd(d["dy"], d["x"], d["a"], d["b"], f["u"], 2.0)
    for k in ("u", "delta_y"):
        G.assert_bitwise(k, out[k], f[k])
    for k in ("du", "db", "dx", "da"):
        G.assert_bitwise(k, out[k], g[k])


def _fuzz_shapes(n, seed=20261202):
    """Seeded random ragged shapes: M in [1, 900], K and N multiples of 8 up to 1600, ranks 8
    and 16 (dX and dA in one launch) and 24 / 32 (separate launches), alpha 2, 0.5 or 1 (the
    dV pass-through)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 901))
        K, N = (8 * int(v) for v in rng.integers(1, 201, size=2))
        R = (8, 16, 16, 24, 32)[i % 5]
        out.append((M, K, N, R, (2.0, 0.5, 1.0)[i % 3]))
    return out


@pytest.mark.parametrize("M,K,N,R,alpha", _fuzz_shapes(15))
def test_random_ragged_shapes_bitwise_on_integer_inputs(oracle, M, K, N, R, alpha):
    """Small-integer inputs at random ragged shapes (every partial sum exact): every output of
    the forward and the backward equals the oracle bit for bit, whatever the shape's tails,
    unit counts against the SM count, ring-slot counts and launch schedule."""
    w = S.integers(M, K, N, R, alpha, bound=2)
    d = w.generate(7)
    out = G.run(d, alpha)
    f = oracle.fwd(d["x"], d["a"], d["b"], alpha)
    g = oracle.bwd(d["dy"], d["x"], d["a"], d["b"], f["u"], alpha)
    for k in ("u", "delta_y"):
        G.assert_bitwise(k, out[k], f[k])
    for k in ("du", "db", "dx", "da"):
        G.assert_bitwise(k, out[k], g[k])


EDGE = [  # (M, K, N, R, alpha): ragged M / K / N tails, every padded rank, single rows, one-tile and many-tile cases
    (1, 64, 64, 8, 2.0), (7, 136, 96, 16, 0.5), (100, 200, 104, 24, 1.0), (129, 512, 264, 32, 2.0),
    (300, 1032, 520, 40, 0.75), (257, 256, 128, 48, 1.5), (65, 8, 8, 56, 2.0), (600, 2056, 300 - 4, 64, 1.0),
    (1000, 96, 2048, 16, 3.0), (2, 4096 + 8, 16, 8, 0.25),
]


@pytest.mark.parametrize("M,K,N,R,alpha", EDGE)
def test_edge_shapes(oracle, M, K, N, R, alpha):
    w = S.Workload("edge", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": K ** -0.5, "b": R ** -0.5, "dy": 1.0})
    d = w.generate(3)
    out = G.run(d, alpha)
    G.check_parity(oracle, d, alpha, out)


def test_adversarial_same_sign_inputs(oracle):
    """All products positive and a long reduction: rounding errors cannot
    cancel, the worst case for the 1e-6 * sum|ab| bound."""
    M, K, N, R = 256, 17408, 256, 16
    w = S.Workload("pos", S.Shape(M, K, N, R, 1.0), {"x": 1.0, "a": 1.0, "b": 1.0, "dy": 1.0})
    d = w.generate(8)
    for k in d:
        d[k] = d[k] & np.uint16(0x7FFF)          # clear the sign bit: |value|
    out = G.run(d, 1.0)
    worst = G.check_parity(oracle, d, 1.0, out)
    print("worst |err|/S:", worst)


@pytest.mark.parametrize("alpha", [2.0, 0.5, 4096.0, 3.0, -2.0])
def test_dv_rounding_of_every_finite_bf16(oracle, alpha):
    """dV = bf16(dY * alpha) for every finite BF16 value of dY (signed zeros,
    subnormals, values that overflow to infinity). B selects column 16 r of
    each 16-column block for output column r and dY is zero elsewhere, so
    dU[m][r] = dV[m][16 r] exactly: dU shows dV bit for bit. Powers of two take
    the kernels' packed BF16 multiply, 3 and -2 the FP32 form."""
    R = 16
    pats = np.arange(65536, dtype=np.uint32)
    pats = pats[(pats & 0x7F80) != 0x7F80].astype(np.uint16)          # finite patterns only
    M = -(-pats.size // R)
    N, K = 16 * R, 64
    dy = np.zeros((M, N), np.uint16)
    flat = np.zeros(M * R, np.uint16)
    flat[: pats.size] = pats
    dy[:, 0::16] = flat.reshape(M, R)
    b = np.zeros((N, R), np.uint16)
    b[16 * np.arange(R), np.arange(R)] = 0x3F80                      # 1.0
    w = S.Workload("dv", S.Shape(M, K, N, R, alpha), {"x": 1.0, "a": 0.125, "b": 1.0, "dy": 1.0})
    d = w.generate(0)
    d.update(dy=dy, b=b)
    out = G.run(d, alpha)
    ref = oracle.du(oracle.dv(dy, alpha), b)
    got = out["du"]
    finite = (ref & 0x7F80) != 0x7F80
    zero = ((ref & 0x7FFF) == 0) & ((got & 0x7FFF) == 0)            # +0 and -0 equal (sum of a -0 and +0s)
    assert np.array_equal(got[finite & ~zero], ref[finite & ~zero])
    nan = finite == False  # noqa: E712
    ref_nan = nan & ((ref & 0x7F) != 0)
    assert np.array_equal(got[nan] & 0x7F80, ref[nan] & 0x7F80)   # non-finite where the oracle is
    assert np.array_equal((got[ref_nan] & 0x7F) != 0, np.ones(int(ref_nan.sum()), bool))
    inf = nan & ~ref_nan
    assert np.array_equal(got[inf], ref[inf])                       # same infinities, same signs


def test_power_of_two_alpha_with_out_of_range_weights(oracle):
    """alpha = 2^12 with a few entries of b at 2^118 (alpha * b would leave the
    BF16 range): the stages that meet them must take dV = bf16(dY * alpha)
    itself, not alpha * b; dU, dB, dX and dA against the oracle as usual."""
    M, K, N, R, alpha = 512, 256, 1024, 16, 4096.0
    w = S.Workload("pow2big", S.Shape(M, K, N, R, alpha), {"x": 2.0 ** -10, "a": 256 ** -0.5, "b": 0.25, "dy": 2.0 ** -16})
    d = w.generate(9)
    b = d["b"].copy()
    b[[3, 200, 515, 1000], [0, 7, 15, 4]] = 0x7AC0                    # 2^118 * 1.5
    d["b"] = b
    out = G.run(d, alpha)
    G.check_parity(oracle, d, alpha, out)


def test_reruns_are_bitwise_identical():
    w = S.sweep(2048, 1024)
    d = w.generate(1)
    a = G.run(d, w.shape.alpha)
    b = G.run(d, w.shape.alpha)
    for k in a:
        G.assert_bitwise(k, a[k], b[k])


def test_alpha_scaling_and_zero_weights():
    w = S.tiny()
    d = w.generate(2)
    base = G.run(d, 1.0)
    two = G.run(d, 2.0)
    G.assert_bitwise("u", two["u"], base["u"])
    for k in ("delta_y", "db", "dx", "da"):
        G.assert_bitwise(k, two[k], (base[k] * np.float32(2.0)).astype(np.float32))
    zb = dict(d, b=np.zeros_like(d["b"]))
    out = G.run(zb, 2.0)
    for k in ("delta_y", "dx", "da"):
        assert not np.any(out[k]), k
    assert not np.any(out["du"] & 0x7FFF) and np.any(out["db"])
    za = dict(d, a=np.zeros_like(d["a"]))
    out = G.run(za, 2.0)
    assert not np.any(out["u"] & 0x7FFF) and not np.any(out["delta_y"]) and not np.any(out["db"])


# -------------------------------------------------------- batch invariance
def _check_subbatches(d, alpha, full, sizes):
    M = d["x"].shape[0]
    for s in sizes:
        for rows in (slice(0, s), slice(M - s, M)):
            sub = G.run(d, alpha, rows=rows)
            ref = _rows_of(full, rows)
            for k in ("u", "delta_y", "du", "dx"):
                G.assert_bitwise(f"{k} rows {rows.start}:{rows.stop}", sub[k], ref[k])


def test_ragged_tails_are_stable_across_reruns():
    """Batches whose last 128-row tile is partly empty, run several times:
    warps whose rows lie past M skip their stores, which must not disturb the
    staging of the rows before them (every run bit-identical to the full batch)."""
    w = S.Workload("ragged", S.Shape(4224, 512, 4096, 16, 2.0), {"x": 1.0, "a": 512 ** -0.5, "b": 0.25, "dy": 1.0})
    d = w.generate(4)
    full = G.run(d, w.shape.alpha)
    for s in (4097, 4098, 4100, 4160, 4223):
        for _ in range(3):
            sub = G.run(d, w.shape.alpha, rows=slice(0, s))
            for k in ("u", "delta_y", "du", "dx"):
                G.assert_bitwise(f"{k} rows 0:{s}", sub[k], full[k][:s])


def test_shared_workspace_across_shapes():
    """One pair of workspaces reused by calls of different batch sizes: every
    call equals a call with fresh workspaces bit for bit (nothing a call leaves
    in the scratch is read by the next), and the status block stays zero."""
    from deterministic_arithmetic_gb300 import lora_delta as ld

    w = S.Workload("shared", S.Shape(2304, 1024, 2048, 16, 2.0), {"x": 1.0, "a": 1024 ** -0.5, "b": 0.25, "dy": 1.0})
    d = w.generate(6)
    M0, K, N, R = 2304, 1024, 2048, 16
    wf = ld.new_workspace(ld.lora_delta_fwd_workspace_size(M0, K, N, R), "cuda")
    wb = ld.new_workspace(ld.lora_delta_bwd_workspace_size(M0, K, N, R), "cuda")
    A, B = G.dev_bf16(d["a"]), G.dev_bf16(d["b"])
    for m in (2304, 37, 1000, 2304, 1, 640):
        X, DY = G.dev_bf16(d["x"][:m]), G.dev_bf16(d["dy"][:m])
        y, u = ld.lora_delta_fwd(X, A, B, 2.0, workspace=wf)
        dx, da, db, du = ld.lora_delta_bwd(DY, X, A, B, u, 2.0, workspace=wb)
        torch.cuda.synchronize()
        control = 256 + 65536      # status block and control words: zero after every call
        assert not wf[:control].any().item() and not wb[:control].any().item(), m
        ref = G.run(d, 2.0, rows=slice(0, m))
        got = dict(u=G.host_bits(u), delta_y=G.host_f32(y), du=G.host_bits(du), dx=G.host_f32(dx),
                   da=G.host_f32(da), db=G.host_f32(db))
        for k in got:
            G.assert_bitwise(f"{k} m={m}", got[k], ref[k])


def test_tiny_batch_invariance():
    w = S.tiny()
    d = w.generate(0)
    full = G.run(d, w.shape.alpha)
    _check_subbatches(d, w.shape.alpha, full, (1, 7, 32, 64))


@pytest.mark.parametrize("M,KN", S.SWEEP_SHAPES)
def test_invariance_sweep(oracle, M, KN):
    """5 seeds x sub-batch sizes {1, 8, 24, 100, M}: every row boundary (U,
    delta_y, dU, dX) bitwise equal to the full batch's rows; dA/dB by rerun.
    Parity against the oracle on the first seed."""
    w = S.sweep(M, KN)
    for seed in range(5):
        d = w.generate(seed)
        full = G.run(d, w.shape.alpha)
        if seed == 0:
            G.check_parity(oracle, d, w.shape.alpha, full)
        sizes = [s for s in S.SWEEP_SUBBATCH if s <= M] + [M]
        _check_subbatches(d, w.shape.alpha, full, sizes)
        again = G.run(d, w.shape.alpha)
        for k in ("da", "db"):
            G.assert_bitwise(k, again[k], full[k])


# ------------------------------------------------------ full-size workloads
def test_training_step_full_size(oracle):
    """M=8192, K=N=4096, R=16, alpha=2 (the benchmark's workload): every
    element of every boundary against the oracle, sub-batch invariance, reruns."""
    w = S.train()
    d = w.generate(0)
    out = G.run(d, w.shape.alpha)
    worst = G.check_parity(oracle, d, w.shape.alpha, out)
    print("training step: worst |err|/S and band counts:", worst)
    _check_subbatches(d, w.shape.alpha, out, (1, 100, 4097))
    again = G.run(d, w.shape.alpha)
    for k in out:
        G.assert_bitwise(k, again[k], out[k])


@pytest.mark.parametrize("site", ["fc1", "fc2"])
def test_mlp_insertion_points(oracle, site):
    w = S.mlp_fc1() if site == "fc1" else S.mlp_fc2()
    d = w.generate(0)
    out = G.run(d, w.shape.alpha)
    worst = G.check_parity(oracle, d, w.shape.alpha, out)     # every element of every boundary
    print(f"{site}: worst |err|/S and band counts:", worst)
    _check_subbatches(d, w.shape.alpha, out, (8,))
    # acceptance criteria of the same page: the gradients are finite and not all zero, at both
    # insertion points
    for k in ("delta_y", "dx", "da", "db"):
        v = out[k]
        assert np.isfinite(v).all(), f"{site}: {k} has a non-finite value"
        assert np.count_nonzero(v) > v.size // 2, f"{site}: {k} is mostly zero"
    for k in ("u", "du"):
        assert ((out[k] & 0x7F80) != 0x7F80).all(), f"{site}: {k} has an infinite or NaN value"


@pytest.mark.parametrize("M", [1, 8, 64])
def test_decode_batches(oracle, M):
    w = S.decode(M)
    d = w.generate(0)
    out = G.run(d, w.shape.alpha)
    ref_u, s_u, f_u = oracle.u(d["x"], d["a"], want_s=True, want_f32=True)
    G.assert_bf16_close("U", out["u"], ref_u, f_u, s_u)
    y, sy = oracle.delta_y(out["u"], d["b"], w.shape.alpha, True)
    G.assert_f32_within("delta_y", out["delta_y"], y, sy)
    if M == 64:
        G.check_parity(oracle, d, w.shape.alpha, out)
    # decode rows are the leading rows of the 64-row batch (same flat streams): same bits
    if M < 64:
        w64 = S.decode(64)
        d64 = w64.generate(0)
        assert np.array_equal(d64["x"][:M], d["x"]) and np.array_equal(d64["dy"][:M], d["dy"])
        big = G.run(d64, w64.shape.alpha)
        for k in ("u", "delta_y", "du", "dx"):
            G.assert_bitwise(k, out[k], big[k][:M])
