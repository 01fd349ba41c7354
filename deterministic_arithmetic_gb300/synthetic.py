"""Seeded synthetic inputs for the LoRA delta operator.

This module generates inputs and nothing else: it holds none of the
operator's arithmetic, so both the CUDA path's tests/benchmark and the CPU
oracle can take their operands from it.

Generator: splitmix64 in counter mode (output i of stream ``key`` is the
splitmix64 finaliser applied to ``key + (i + 1) * 0x9E3779B97F4A7C15``),
mapped to standard normals by the Box-Muller transform in binary64, scaled,
then converted to bfloat16 by torch's round-to-nearest-even cast. Every array
is a pure function of (seed, tensor name, shape), identical on any host.

Workloads follow the shapes and value distributions of the pages: the
per-GEMM LoRA profile of page "Independent from-scratch Qwen-14B step
reimplementation ..." (section "Finding 2": M=8192, K=N=4096, R=16), the
invariance sweep and insertion points of page "[DSv4][P5-3]
shared_grouped_lora_delta ..." (sections "Batch invariance", "Summary") and
the 17408 x 5120 projection width of the page "Eine reale Projektion als
feste Vergleichsaufgabe". "N(0, s)" in a workload description means variance
s (standard deviation sqrt(s)).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TENSOR_IDS = {"x": 1, "a": 2, "b": 3, "dy": 4}
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, name: str) -> np.uint64:
    base = np.array([(int(seed) & 0xFFFFFFFF) * 0x100 + _TENSOR_IDS.get(name, 0xFF)], np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + _GOLDEN)[0]


def _stream(key: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GOLDEN)


def normal_f64(seed: int, name: str, count: int) -> np.ndarray:
    """``count`` standard normals (binary64) from the named stream."""
    key = _key(seed, name)
    out = np.empty(count, np.float64)
    npairs = (count + 1) // 2
    two53 = 2.0 ** -53
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        raw = _stream(key, 2 * p0, 2 * (p1 - p0))
        u1 = ((raw[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * two53   # (0, 1]
        u2 = (raw[1::2] >> np.uint64(11)).astype(np.float64) * two53          # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * (p1 - p0), np.float64)
        z[0::2] = r * np.cos(2.0 * math.pi * u2)
        z[1::2] = r * np.sin(2.0 * math.pi * u2)
        lo = 2 * p0
        hi = min(count, 2 * p1)
        out[lo:hi] = z[: hi - lo]
    return out


def small_ints(seed: int, name: str, count: int, bound: int) -> np.ndarray:
    """``count`` integers uniform in [-bound, bound] (binary64 values)."""
    key = _key(seed, name)
    raw = _stream(key, 0, count)
    return (raw % np.uint64(2 * bound + 1)).astype(np.int64).astype(np.float64) - bound


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of ``values`` via torch's RNE cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact binary64 values of bfloat16 bit patterns (a bit move, no rounding)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class Shape:
    M: int
    K: int
    N: int
    R: int
    alpha: float


@dataclass(frozen=True)
class Workload:
    """One workload: shape plus the standard deviations of X, A, B, dY."""

    name: str
    shape: Shape
    std: dict = field(default_factory=dict)
    kind: str = "normal"            # "normal" or "ints" (small integers)
    int_bounds: dict = field(default_factory=dict)

    def generate(self, seed: int = 0, only: tuple = ("x", "a", "b", "dy")) -> dict:
        """bf16 bit patterns for x[M,K], a[R,K], b[N,R], dy[M,N]."""
        s = self.shape
        shapes = {"x": (s.M, s.K), "a": (s.R, s.K), "b": (s.N, s.R), "dy": (s.M, s.N)}
        out = {}
        for name in only:
            shp = shapes[name]
            n = shp[0] * shp[1]
            if self.kind == "ints":
                v = small_ints(seed, name, n, self.int_bounds.get(name, 3))
            else:
                v = normal_f64(seed, name, n) * self.std.get(name, 1.0)
            out[name] = to_bf16_bits(v).reshape(shp)
        return out


def _std_pages(K: int, R: int, dy_var: float = 1.0) -> dict:
    return {"x": 1.0, "a": 1.0 / math.sqrt(K), "b": 1.0 / math.sqrt(R), "dy": math.sqrt(dy_var)}


def _std_scaled(K: int, R: int) -> dict:
    return {"x": 1.0 / math.sqrt(K), "a": 1.0 / math.sqrt(K), "b": 1.0 / math.sqrt(R), "dy": 1.0}


def tiny() -> Workload:
    """M=64, K=128, N=96, R=8, alpha=2; X, dY ~ N(0,1); A ~ N(0,1/K); B ~ N(0,1/R)."""
    return Workload("tiny M64 K128 N96 R8", Shape(64, 128, 96, 8, 2.0), _std_pages(128, 8))


SWEEP_SHAPES = ((128, 64), (512, 512), (2048, 1024), (4096, 2048))
SWEEP_SUBBATCH = (1, 8, 24, 100)  # plus M itself


def sweep(M: int, KN: int) -> Workload:
    """Invariance sweep: R=8, alpha=0.5, K=N; X, A, B, dY ~ N(0,1) scaled by
    1/sqrt(K), 1/sqrt(K), 1/sqrt(R), 1."""
    return Workload(f"sweep M{M} K=N{KN} R8", Shape(M, KN, KN, 8, 0.5), _std_scaled(KN, 8))


def train() -> Workload:
    """LoRA training step: M=8192, K=N=4096, R=16, alpha=2; X ~ N(0,1),
    A ~ N(0,1/4096), B ~ N(0,1/16), dY ~ N(0,1e-2)."""
    return Workload("train M8192 K4096 N4096 R16", Shape(8192, 4096, 4096, 16, 2.0), _std_pages(4096, 16, 1e-2))


def mlp_fc1() -> Workload:
    """MLP fc1 delta: M=4096, K=5120 -> N=17408, R=16, alpha=1, drawn as train."""
    return Workload("fc1 M4096 K5120 N17408 R16", Shape(4096, 5120, 17408, 16, 1.0), _std_pages(5120, 16, 1e-2))


def mlp_fc2() -> Workload:
    """MLP fc2 delta: M=4096, K=17408 -> N=5120, R=16, alpha=1, drawn as train."""
    return Workload("fc2 M4096 K17408 N5120 R16", Shape(4096, 17408, 5120, 16, 1.0), _std_pages(17408, 16, 1e-2))


def decode(M: int) -> Workload:
    """Decode-like skinny batch: M in {1, 8, 64}, K=5120, N=17408, R=64, alpha=1;
    N(0,1) scaled by 1/sqrt(K), 1/sqrt(K), 1/sqrt(R), 1."""
    return Workload(f"decode M{M} K5120 N17408 R64", Shape(M, 5120, 17408, 64, 1.0), _std_scaled(5120, 64))


def integers(M: int, K: int, N: int, R: int, alpha: float = 2.0, bound: int = 3) -> Workload:
    """Small-integer inputs: every product and partial sum is an integer well
    inside binary32's 24-bit significand, so no summation order can round."""
    return Workload(f"ints M{M} K{K} N{N} R{R}", Shape(M, K, N, R, alpha), kind="ints",
                    int_bounds={"x": bound, "a": 2, "b": 2, "dy": bound})
