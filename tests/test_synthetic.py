"""The seeded input generator (deterministic_arithmetic_gb300/synthetic.py), which
serves the oracle and the GPU path alike: every array is a pure function of
(seed, tensor name, shape); a stream's values do not depend on how many are
drawn, so a smaller batch is the leading rows of a larger one; the streams of
different tensors and seeds differ; the normals have mean 0 and variance 1 and
the scaled workloads the variances they name; the BF16 cast rounds to nearest
even and the reverse map is exact."""
import numpy as np

from deterministic_arithmetic_gb300 import synthetic as S


def test_pure_function_of_seed_name_and_count():
    a = S.normal_f64(3, "x", 1000)
    assert np.array_equal(a, S.normal_f64(3, "x", 1000))
    assert not np.array_equal(a, S.normal_f64(4, "x", 1000))
    assert not np.array_equal(a, S.normal_f64(3, "dy", 1000))
    # the first values of a longer draw are the values of a shorter one (odd counts included)
    assert np.array_equal(S.normal_f64(3, "x", 4097)[:777], S.normal_f64(3, "x", 777))
    ints = S.small_ints(1, "a", 500, 3)
    assert np.array_equal(ints, S.small_ints(1, "a", 500, 3))
    assert set(np.unique(ints)) <= set(range(-3, 4)) and len(np.unique(ints)) == 7


def test_normal_moments():
    z = S.normal_f64(0, "x", 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.var() - 1.0) < 5e-3
    assert abs(np.mean(z ** 4) - 3.0) < 0.05       # Gaussian kurtosis
    assert np.isfinite(z).all()


def test_workload_shapes_and_scales():
    w = S.Workload("t", S.Shape(512, 256, 128, 16, 2.0), {"x": 1.0, "a": 256 ** -0.5, "b": 0.25, "dy": 0.1})
    d = w.generate(0)
    assert d["x"].shape == (512, 256) and d["a"].shape == (16, 256)
    assert d["b"].shape == (128, 16) and d["dy"].shape == (512, 128)
    for k, var in (("x", 1.0), ("a", 1 / 256), ("b", 0.0625), ("dy", 0.01)):
        v = S.bf16_bits_to_f64(d[k])
        assert abs(v.var() / var - 1.0) < 0.1, (k, v.var(), var)
    # a smaller batch is the leading rows of a larger one
    small = S.Workload("t", S.Shape(64, 256, 128, 16, 2.0), w.std).generate(0)
    assert np.array_equal(small["x"], d["x"][:64]) and np.array_equal(small["dy"], d["dy"][:64])


def test_bf16_cast_rounds_to_nearest_even_and_maps_back_exactly():
    vals = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20, -(1 + 2.0 ** -8),
                     2.0 ** -133, 3.4e38, 0.0, -0.0])
    bits = S.to_bf16_bits(vals)
    back = S.bf16_bits_to_f64(bits)
    assert back[0] == 1.0 and back[1] == 1.0                  # tie to even
    assert back[2] == 1 + 2.0 ** -6                           # tie to even (up)
    assert back[3] == 1 + 2.0 ** -7                           # above the midpoint
    assert back[4] == -1.0
    assert back[5] == 2.0 ** -133                             # the least subnormal
    assert np.isinf(back[6])                                  # past the BF16 range
    assert bits[7] == 0x0000 and bits[8] == 0x8000
    every = np.arange(1 << 16, dtype=np.uint16)
    finite = (every & 0x7F80) != 0x7F80
    assert np.array_equal(S.to_bf16_bits(S.bf16_bits_to_f64(every[finite])), every[finite])
