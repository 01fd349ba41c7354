"""CPU model of the GPU path's FP32 reduction order.

TEST INFRASTRUCTURE ONLY: the test suite is the only caller. It shares nothing
with the CUDA library and imports nothing from it.

The f64 oracle (``oracle.oracle``) fixes what each sum is; this module fixes
in which order the GPU path adds its FP32 terms, so that tests can compare the
GPU's bits with a model of that order, not only with a tolerance. The order is
the reduction of page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton,
both batch-invariant", sections "Agreement with the oracle" and "Provenance":
FP32 accumulation over a fixed tree of fixed-size leaves, no split-K, no
atomics, whose children are contiguous shards of the reduction axis. Here:

* a **leaf** is the FP32 dot product of 16 consecutive terms of the reduction
  axis (the last leaf is padded with zeros);
* leaves are added by the **canonical pairwise tree over the leaf index**: at
  level l, node i takes node i + 2^l when i is a multiple of 2^(l+1) and that
  node exists; a node without a partner passes up unchanged. Each addition is
  FP32 round-to-nearest-even.

The tensor core's rounding inside a leaf of several non-zero products is not
modelled; ``single_product_leaves`` builds the leaves of inputs whose every
leaf holds at most one non-zero product, where each leaf is that product (a
BF16 x BF16 product has at most 16 significant bits and is exact in FP32), so
the model is exact for such inputs and the whole result is fixed by the tree.
"""
from __future__ import annotations

import numpy as np

LEAF = 16


def canonical_tree_f32(leaves: np.ndarray, axis: int = -1) -> np.ndarray:
    """FP32 canonical pairwise tree over ``axis`` (the leaf index), level by level."""
    v = np.moveaxis(np.asarray(leaves, dtype=np.float32), axis, 0).copy()
    n = v.shape[0]
    if n == 0:
        return np.zeros(v.shape[1:], np.float32)
    step = 1
    while step < n:
        left = np.arange(0, n, 2 * step)
        left = left[left + step < n]
        v[left] = v[left] + v[left + step]          # float32 + float32: one RN-even rounding
        step *= 2
    return v[0]


def leaf_count(n_terms: int) -> int:
    return (n_terms + LEAF - 1) // LEAF


def single_product_leaves(left: np.ndarray, right: np.ndarray) -> np.ndarray:
    """Leaves of sum_t left[i, t] * right[j, t] for all (i, j), for inputs with at most one
    non-zero product per 16-term leaf (checked). ``left`` (I, T) and ``right`` (J, T) hold BF16
    values (any float dtype); returns (leaf_count(T), I, J) float32: leaf l of (i, j) is the one
    non-zero product among t in [16 l, 16 l + 16), else zero."""
    left = np.asarray(left, dtype=np.float64)
    right = np.asarray(right, dtype=np.float64)
    T = left.shape[1]
    L = leaf_count(T)
    pad = L * LEAF - T

    def blocks(v):                                  # (rows, T) -> (L, rows, 16)
        v = np.concatenate([v, np.zeros((v.shape[0], pad))], axis=1) if pad else v
        return v.reshape(v.shape[0], L, LEAF).transpose(1, 0, 2)

    lb, rb = blocks(left), blocks(right)
    count = (lb != 0).astype(np.float64) @ (rb != 0).astype(np.float64).transpose(0, 2, 1)
    if count.max(initial=0) > 1:
        raise ValueError("a leaf holds more than one non-zero product")
    out = lb @ rb.transpose(0, 2, 1)                # one non-zero term per sum: exact in binary64
    out32 = out.astype(np.float32)
    if not np.array_equal(out32.astype(np.float64), out):
        raise ValueError("a product is not exact in FP32")
    return out32


def rnbf_bits(v: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of float32 values, round to nearest even (finite values)."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    return ((b + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """float32 values of BF16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def tree_matmul_f32(left: np.ndarray, right: np.ndarray) -> np.ndarray:
    """sum_t left[i, t] * right[j, t] for all (i, j), added as the GPU path adds it: the canonical
    tree over single-product leaves. left (I, T), right (J, T); returns (I, J) float32."""
    return canonical_tree_f32(single_product_leaves(left, right), axis=0)
