"""The CPU model of the FP32 reduction order (oracle/tree_order.py) against its pins.

The model is pinned to facts outside itself: hand-worked sums whose FP32 result
depends on the pairing (each worked out below from IEEE round-to-nearest-even),
a recursive statement of the same tree, exact sums where no addition rounds,
torch's own float32 -> bfloat16 conversion, and the leaf builder's checks. Each
alternative order that a plausible mistake would give (left to right, right to
left, halves split in the middle, the unpaired node joined on the wrong side)
fails at least one pin."""
import numpy as np
import pytest

from oracle import tree_order as T

E = np.float32(2.0 ** -24)          # half an FP32 ulp of 1.0


def tree(v):
    return T.canonical_tree_f32(np.asarray(v, np.float32))


# (leaves, expected FP32 sum under the canonical tree). In FP32, 1 + 2^-24 is a tie that rounds
# to 1 (even), while 2^-24 + 2^-24 = 2^-23 is exact and 1 + 2^-23 is representable.
WORKED = [
    ([1, 0, E, E], 1 + 2 * E),            # (1+0) + (E+E): the two halves meet first
    ([1, E, E, 0], 1),                    # (1+E) + (E+0) = 1 + E -> 1
    ([E, E, 1], 1 + 2 * E),               # (E+E) + 1: node 2 has no partner at level 0
    ([1, 0, 0, E, E, 0], 1),              # ((1+0)+(0+E)) + (E+0): the last pair joins at level 2
    ([E, E, E, E, 1, 0, 0], 1 + 4 * E),   # ((E+E)+(E+E)) + ((1+0)+0)
    ([1, 0, E, 0, E], 1),                 # ((1+0)+(E+0)) + E = (1+E) + E -> 1 + E -> 1
]


@pytest.mark.parametrize("leaves,want", WORKED)
def test_worked_sums(leaves, want):
    got = tree(leaves)
    assert got.dtype == np.float32 and got == np.float32(want), (leaves, float(got), float(want))


def _recursive(v):
    """The same tree stated top-down: the first child holds the largest power of two of leaves
    that is smaller than the count, the second child the rest."""
    n = len(v)
    if n == 1:
        return np.float32(v[0])
    p = 1
    while 2 * p < n:
        p *= 2
    return np.float32(_recursive(v[:p]) + _recursive(v[p:]))


@pytest.mark.parametrize("n", [1, 2, 3, 5, 7, 8, 13, 17, 34, 64, 65, 100, 1088])
def test_level_by_level_equals_recursive_split(n):
    rng = np.random.default_rng(n)
    v = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
    assert tree(v).view(np.uint32) == _recursive(v).view(np.uint32)


def test_axis_and_batch():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((7, 37, 3)) * np.exp2(rng.integers(-20, 20, (7, 37, 3)))).astype(np.float32)
    got = T.canonical_tree_f32(v, axis=1)
    for i in range(7):
        for j in range(3):
            assert got[i, j].view(np.uint32) == _recursive(v[i, :, j]).view(np.uint32)


def test_exact_when_nothing_rounds():
    rng = np.random.default_rng(6)
    v = rng.integers(-2 ** 12, 2 ** 12, (50, 1000)).astype(np.float32)   # every partial sum < 2^24
    assert np.array_equal(T.canonical_tree_f32(v, axis=1), v.astype(np.int64).sum(axis=1).astype(np.float32))


def test_zero_padding_on_the_right_is_neutral():
    rng = np.random.default_rng(7)
    for n in (3, 9, 34, 100):
        v = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
        for pad in (1, 5, 64):
            assert tree(np.concatenate([v, np.zeros(pad, np.float32)])) == tree(v)


def _left_to_right(v):
    s = np.float32(0)
    for x in v:
        s = np.float32(s + np.float32(x))
    return s


def _right_to_left(v):
    return _left_to_right(list(v)[::-1])


def _mid_split(v):
    n = len(v)
    if n == 1:
        return np.float32(v[0])
    h = (n + 1) // 2
    return np.float32(_mid_split(v[:h]) + _mid_split(v[h:]))


def _odd_node_first(v):
    """Pairs taken from the right end, so the unpaired node sits on the left."""
    v = [np.float32(x) for x in v]
    while len(v) > 1:
        out = []
        if len(v) % 2:
            out.append(v[0])
            v = v[1:]
        out += [np.float32(v[i] + v[i + 1]) for i in range(0, len(v), 2)]
        v = out
    return v[0]


@pytest.mark.parametrize("wrong", [_left_to_right, _right_to_left, _mid_split, _odd_node_first])
def test_each_other_order_fails_a_worked_sum(wrong):
    assert any(wrong([np.float32(x) for x in leaves]) != np.float32(want) for leaves, want in WORKED)


def test_rnbf_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-60, 60, 200000))).astype(np.float32)
    ties = (np.arange(1, 2000, dtype=np.uint32) << 15).view(np.float32) * np.float32(1.0)   # low half 0x8000
    v = np.concatenate([v, ties, -ties, np.float32([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8])])
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(T.rnbf_bits(v), want)
    assert T.rnbf_bits(np.float32([1 + 2 ** -8]))[0] == 0x3F80       # tie to even: down to 1.0
    assert T.rnbf_bits(np.float32([1 + 3 * 2 ** -8]))[0] == 0x3F82   # tie to even: up to 1 + 2^-6
    assert np.array_equal(T.bf16_value(T.rnbf_bits(np.float32([1.5, -3.25]))), np.float32([1.5, -3.25]))


def test_single_product_leaves():
    left = np.zeros((2, 40), np.float32)
    right = np.zeros((3, 40), np.float32)
    left[0, 3], left[0, 20], left[0, 39] = 1.5, -2.0, 0.75      # leaves 0, 1, 2 (the last one ragged)
    left[1, 17] = 3.0
    right[:, :] = np.arange(1, 4, dtype=np.float32)[:, None]
    got = T.single_product_leaves(left, right)
    assert got.shape == (3, 2, 3)
    assert np.array_equal(got[:, 0, 1], np.float32([3.0, -4.0, 1.5]))
    assert np.array_equal(got[:, 1, 2], np.float32([0.0, 9.0, 0.0]))
    two = left.copy()
    two[0, 4] = 1.0                                            # a second product in leaf 0
    with pytest.raises(ValueError):
        T.single_product_leaves(two, right)
    with pytest.raises(ValueError):                            # 2^-160: below FP32's range, not exact
        T.single_product_leaves(np.float32([[2.0 ** -120]]), np.float32([[2.0 ** -40]]))


def test_tree_matmul_of_integers_is_the_exact_product():
    rng = np.random.default_rng(9)
    M, K = 37, 16 * 9 + 5
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        for j in range(T.leaf_count(K)):
            k = 16 * j + (7 * m + j) % 16
            if k < K:
                x[m, k] = rng.integers(-64, 64)
    a = rng.integers(-64, 64, (5, K)).astype(np.float32)
    assert np.array_equal(T.tree_matmul_f32(x, a), (x.astype(np.int64) @ a.astype(np.int64).T).astype(np.float32))
