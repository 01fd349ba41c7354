"""Exact mode of the weight gradients (lora_delta_grads_exact, page "det-train",
section "Method") against the exact-mode oracle: bitwise, everywhere.

* dA and dB (FP32) and their digit arrays equal the oracle's bit for bit, for
  ranks 8-64, ragged K, N and M, alpha of both kinds (power of two or not), and
  inputs over a wide exponent range (products far from one another, which take
  the kernel's direct path as well as its register window).
* The closed-form sums of the oracle's pins (cancellation, ties, overflow,
  subnormals, IEEE specials) come out exact on the GPU.
* Factors far below their column's largest, subnormal ones and zeros, few or many
  per 64 rows, take the kernel's exact side paths with the same bits.
* Row shards' digit arrays, added with lora_delta_exact_combine in any grouping,
  equal the whole batch's; so does their plain int64 sum (what an all-reduce
  leaves) once normalised; finalize gives the same FP32 bits; any row order gives
  the same bits; reruns are bitwise.
* The full training shape (M=8192, K=N=4096, R=16): sampled columns against the
  oracle, and every output equal to the correctly rounded binary64 sum where that
  sum is exact."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_arithmetic_gb300 import lora_delta as ld  # noqa: E402
from deterministic_arithmetic_gb300 import synthetic as S  # noqa: E402
from oracle.exact_mode import ExactOracle  # noqa: E402
import gpu_util as G  # noqa: E402
import pins_exact as PE  # noqa: E402

pytestmark = pytest.mark.gpu
EO = ExactOracle()


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_arithmetic_gb300 import build_lib

    build_lib.build()


def _inputs(M, K, N, R, seed, wide=False):
    """x, dy, u, du as bf16 bits: the training distributions, or (wide) magnitudes
    spread over 2^-60 .. 2^60 with exact zeros."""
    rng = np.random.default_rng(seed)
    if wide:
        def g(shape):
            v = rng.standard_normal(shape) * np.exp2(rng.integers(-60, 60, shape))
            v[rng.random(shape) < 0.05] = 0.0
            return S.to_bf16_bits(v)
        return dict(x=g((M, K)), dy=g((M, N)), u=g((M, R)), du=g((M, R)))
    w = S.Workload("exact", S.Shape(M, K, N, R, 1.0), {"x": 1.0, "dy": 0.1})
    d = w.generate(seed, only=("x", "dy"))
    d["u"] = S.to_bf16_bits(rng.standard_normal((M, R)) * 4.0)
    d["du"] = S.to_bf16_bits(rng.standard_normal((M, R)) * 0.05)
    return d


def _gpu(d, alpha, want=("da", "db", "da_digits", "db_digits")):
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    out = ld.lora_delta_grads_exact(t["dy"], t["x"], t["u"], t["du"], alpha, want=want)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _bits_equal(name, got, want):
    g = np.ascontiguousarray(got)
    w = np.ascontiguousarray(want)
    assert g.shape == w.shape, f"{name}: shape {g.shape} != {w.shape}"
    if g.dtype == np.float32:
        nan = np.isnan(g) & np.isnan(w)
        g, w = np.where(nan, 0, g.view(np.uint32)), np.where(nan, 0, w.view(np.uint32))
    bad = np.argwhere(g != w)
    assert bad.size == 0, f"{name}: {len(bad)} elements differ, first at {tuple(bad[0])}: " \
                          f"{got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


SHAPES = [(300, 136, 72, 16, 2.0), (129, 64, 200, 8, 0.3), (70, 520, 24, 24, -1.5), (257, 72, 64, 64, 0.5),
          (1, 8, 8, 32, 1.0)]


@pytest.mark.parametrize("wide", [False, True], ids=["train-like", "wide-exponents"])
@pytest.mark.parametrize("M,K,N,R,alpha", SHAPES)
def test_bitwise_equal_to_the_oracle(oracle, M, K, N, R, alpha, wide):
    d = _inputs(M, K, N, R, seed=M + K + N + R, wide=wide)
    out = _gpu(d, alpha)
    dv = oracle.dv(d["dy"], alpha)
    _bits_equal("dA digits", out["da_digits"], EO.digits(d["du"], d["x"]))
    _bits_equal("dB digits", out["db_digits"], EO.digits(d["u"], dv, transpose=True))
    da, db = EO.grads(dv, d["x"], d["u"], d["du"])
    _bits_equal("dA", out["da"], da)
    _bits_equal("dB", out["db"], db)


def test_closed_forms():
    """Every closed-form case of the oracle's pins on one diagonal: case c sits in
    column c of du and of x, so dA[c][c] is its sum."""
    cases = PE.CLOSED_FORMS
    R = K = 32
    assert len(cases) <= R
    M = max(1, max(len(p) for _, p, _ in cases))
    du = np.zeros((M, R)); x = np.zeros((M, K))
    for c, (_, products, _) in enumerate(cases):
        for m, (a, b) in enumerate(products):
            du[m, c], x[m, c] = a, b
    d = dict(du=S.to_bf16_bits(du), x=S.to_bf16_bits(x))
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    u = torch.zeros((M, R), dtype=torch.bfloat16, device="cuda")
    out = ld.lora_delta_grads_exact(None, t["x"], u, t["du"], 1.0, want=("da", "da_digits"))
    torch.cuda.synchronize()
    da = out["da"].cpu().numpy()
    for c, (name, _, want) in enumerate(cases):
        PE._same(f"GPU {name}", da[c, c], want)
    _bits_equal("dA digits (whole matrix)", out["da_digits"].cpu().numpy(), EO.digits(d["du"], d["x"]))
    _bits_equal("dA (whole matrix)", da, EO.exact_matmul(d["du"], d["x"]))


def test_row_shards_compose(oracle):
    M, K, N, R, alpha = 700, 264, 136, 16, 2.0
    d = _inputs(M, K, N, R, seed=5, wide=True)
    whole = _gpu(d, alpha)
    cuts = [0, 1, 130, 131, 512, M]
    parts = [_gpu({k: v[a:b] for k, v in d.items()}, alpha, want=("da_digits", "db_digits"))
             for a, b in zip(cuts[:-1], cuts[1:])]
    for key, fp in (("da_digits", "da"), ("db_digits", "db")):
        dev = [torch.from_numpy(p[key]).cuda() for p in parts]
        acc = dev[0].clone()
        for p in dev[1:]:                                    # left fold, in place
            ld.lora_delta_exact_combine(acc, p, out=acc)
        tree = ld.lora_delta_exact_combine(ld.lora_delta_exact_combine(dev[0], dev[1]),
                                           ld.lora_delta_exact_combine(dev[2], ld.lora_delta_exact_combine(dev[3],
                                                                                                           dev[4])))
        fin = ld.lora_delta_exact_finalize(acc)
        torch.cuda.synchronize()
        _bits_equal(f"{key}: left fold", acc.cpu().numpy(), whole[key])
        _bits_equal(f"{key}: tree", tree.cpu().numpy(), whole[key])
        _bits_equal(f"{fp}: finalize", fin.cpu().numpy(), whole[fp])
        _bits_equal(f"{fp}: oracle finalize", EO.finalize(acc.cpu().numpy()), whole[fp])


def test_row_order_and_reruns():
    M, K, N, R, alpha = 513, 128, 64, 16, 0.3
    d = _inputs(M, K, N, R, seed=9, wide=True)
    a = _gpu(d, alpha)
    b = _gpu(d, alpha)
    perm = np.random.default_rng(1).permutation(M)
    c = _gpu({k: v[perm] for k, v in d.items()}, alpha)
    for key in a:
        _bits_equal(f"{key}: rerun", b[key], a[key])
        _bits_equal(f"{key}: permuted rows", c[key], a[key])


def test_empty_batch_and_partial_outputs():
    K, N, R = 64, 32, 8
    x = torch.zeros((0, K), dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros((0, N), dtype=torch.bfloat16, device="cuda")
    u = torch.zeros((0, R), dtype=torch.bfloat16, device="cuda")
    out = ld.lora_delta_grads_exact(dy, x, u, u, 1.0, want=("da", "db", "db_digits"))
    torch.cuda.synchronize()
    assert (out["da"].view(torch.int32) == 0).all() and (out["db"].view(torch.int32) == 0).all()
    assert (out["db_digits"] == 0).all()
    # only dB asked for: x and du may be absent
    d = _inputs(40, K, N, R, seed=2)
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    only_b = ld.lora_delta_grads_exact(t["dy"], None, t["u"], None, 0.5, want=("db",))
    torch.cuda.synchronize()
    full = _gpu(d, 0.5)
    _bits_equal("dB alone", only_b["db"].cpu().numpy(), full["db"])
    assert set(only_b) == {"db"}


def test_training_shape_sampled(oracle):
    """M=8192, K=N=4096, R=16, alpha=2, the training distributions: 24 sampled
    columns of dA and of dB against the oracle; every output against the binary64
    sum rounded to FP32 where no binary64 rounding occurred (|sum| bounds), and
    within half an FP32 ulp of the binary64 sum elsewhere."""
    w = S.train()
    M, K, N, R, alpha = w.shape.M, w.shape.K, w.shape.N, w.shape.R, w.shape.alpha
    d = w.generate(0, only=("x", "dy"))
    rng = np.random.default_rng(3)
    d["u"] = S.to_bf16_bits(rng.standard_normal((M, R)) * 4.0)
    d["du"] = S.to_bf16_bits(rng.standard_normal((M, R)) * 0.05)
    out = _gpu(d, alpha, want=("da", "db"))
    again = _gpu(d, alpha, want=("da", "db"))
    _bits_equal("dA rerun", again["da"], out["da"])
    _bits_equal("dB rerun", again["db"], out["db"])
    cols = np.sort(rng.choice(K, 24, replace=False))
    _bits_equal("dA sampled", out["da"][:, cols], EO.exact_matmul(d["du"], d["x"][:, cols]))
    dv = oracle.dv(d["dy"], alpha)
    ncol = np.sort(rng.choice(N, 24, replace=False))
    _bits_equal("dB sampled", out["db"][ncol], EO.exact_matmul(d["u"], dv[:, ncol], transpose=True))
    # every output: the correctly rounded exact sum is within half an FP32 ulp of the binary64 sum
    # plus the binary64 sum's own error bound (M products, each exact)
    for name, left, right, got in (("dA", d["du"], d["x"], out["da"]), ("dB", d["u"], dv, out["db"].T)):
        L = S.bf16_bits_to_f64(left); Rt = S.bf16_bits_to_f64(right)
        ref = L.T @ Rt
        bound = M * 2.0 ** -52 * (np.abs(L).T @ np.abs(Rt))
        g = got.astype(np.float64)
        half_ulp = np.spacing(np.abs(got).astype(np.float32)).astype(np.float64) / 2
        assert np.all(np.abs(g - ref) <= half_ulp + bound + 2.0 ** -149), f"{name}: not the rounded exact sum"
        assert math.isfinite(float(np.abs(g).max()))


def test_raw_digit_sums_normalise_to_the_whole():
    """What an int64 sum all-reduce of the ranks' digit arrays leaves (a plain sum, not
    normalised), normalised by lora_delta_exact_combine(a, None): the whole batch's digits."""
    M, K, N, R, alpha = 300, 72, 64, 16, 0.5
    d = _inputs(M, K, N, R, seed=12, wide=True)
    whole = _gpu(d, alpha, want=("da_digits", "db_digits"))
    cuts = [0, 100, 101, M]
    parts = [_gpu({k: v[a:b] for k, v in d.items()}, alpha, want=("da_digits", "db_digits"))
             for a, b in zip(cuts[:-1], cuts[1:])]
    for key in ("da_digits", "db_digits"):
        raw = sum(torch.from_numpy(p[key]) for p in parts).cuda()
        norm = ld.lora_delta_exact_combine(raw, None, out=raw)
        torch.cuda.synchronize()
        _bits_equal(f"{key}: summed and normalised", norm.cpu().numpy(), whole[key])


@pytest.mark.parametrize("frac", [0.002, 0.02, 0.1], ids=["few-small", "more-small", "past-the-list"])
def test_small_factors_take_the_exact_side_path(oracle, frac):
    """The training distributions with a sprinkling of factors far below their column's
    largest (2^-24 .. 2^-60 of it), subnormal ones, and exact zeros: a few of them per 64 rows
    go through the listed one-by-one path, more than the list holds through the general one.
    Bitwise equal to the oracle either way."""
    M, K, N, R, alpha = 640, 136, 200, 16, 0.75
    rng = np.random.default_rng(int(frac * 1e4))
    d = _inputs(M, K, N, R, seed=33)
    for key in ("x", "dy", "u", "du"):
        v = S.bf16_bits_to_f64(d[key])
        pick = rng.random(v.shape) < frac
        v[pick] *= np.exp2(-rng.integers(24, 60, v.shape))[pick]
        v[rng.random(v.shape) < frac / 4] = 2.0 ** -130 * rng.integers(-100, 100)   # subnormal (or zero)
        v[rng.random(v.shape) < frac] = 0.0
        d[key] = S.to_bf16_bits(v)
    out = _gpu(d, alpha)
    dv = oracle.dv(d["dy"], alpha)
    _bits_equal("dA digits", out["da_digits"], EO.digits(d["du"], d["x"]))
    _bits_equal("dB digits", out["db_digits"], EO.digits(d["u"], dv, transpose=True))
    da, db = EO.grads(dv, d["x"], d["u"], d["du"])
    _bits_equal("dA", out["da"], da)
    _bits_equal("dB", out["db"], db)


def test_f32_dy(oracle):
    """lora_delta_grads_exact with a binary32 dY: dB is the exact oracle's on
    dV = bf16(fp32(dy * alpha)) (the FP32-dY backward's dV), bit for bit; dY values BF16 holds
    exactly give the BF16-dY call's bits."""
    M, K, N, R, alpha = 300, 64, 136, 16, 0.3
    d = _inputs(M, K, N, R, seed=21)
    rng = np.random.default_rng(5)
    dy32 = (rng.standard_normal((M, N)) * np.exp2(rng.integers(-20, 20, (M, N)))).astype(np.float32)
    t = {k: G.dev_bf16(v) for k, v in d.items()}
    out = ld.lora_delta_grads_exact(torch.from_numpy(dy32).cuda(), t["x"], t["u"], t["du"], alpha,
                                    want=("da", "db", "db_digits"))
    torch.cuda.synchronize()
    dv = oracle.dv_f32(dy32, alpha)
    _bits_equal("dB digits (f32 dy)", out["db_digits"].cpu().numpy(), EO.digits(d["u"], dv, transpose=True))
    _bits_equal("dB (f32 dy)", out["db"].cpu().numpy(), EO.exact_matmul(d["u"], dv, transpose=True))
    _bits_equal("dA (f32 dy call)", out["da"].cpu().numpy(), EO.exact_matmul(d["du"], d["x"]))
    # BF16-representable binary32 dY: the same bits as the BF16-dY call
    dyb = S.bf16_bits_to_f64(d["dy"]).astype(np.float32)
    a = ld.lora_delta_grads_exact(torch.from_numpy(dyb).cuda(), t["x"], t["u"], t["du"], alpha, want=("db",))
    b = ld.lora_delta_grads_exact(t["dy"], t["x"], t["u"], t["du"], alpha, want=("db",))
    torch.cuda.synchronize()
    _bits_equal("dB: f32 dy holding BF16 values", a["db"].cpu().numpy(), b["db"].cpu().numpy())


def test_rate_probe_runs_and_counts_its_products():
    """The multiply-add rate probe (the exact mode's measured roofline): the launch performs the
    number of multiply-adds it reports (two CTAs of 512 threads per SM, 8 chains per thread) and
    writes every thread's sum."""
    from deterministic_arithmetic_gb300 import lora_delta as ld

    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(ld.library().lora_delta_exact_rate_probe_sink_bytes(), dtype=torch.uint8, device="cuda")
    assert sink.numel() == 2 * nsm * 512 * 8
    n = ld.lora_delta_exact_rate_probe(16, sink=sink)
    torch.cuda.synchronize()
    assert n == 2 * nsm * 512 * 8 * 16
    assert sink.view(torch.int64).ne(0).all().item()
