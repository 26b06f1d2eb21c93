"""Pins for the RoPE-with-tree-positions oracle (oracle.attention.rope and
tree_positions; positions are the prefix length plus the node depth, SwiftSpec
summary §3.3): closed forms, norm preservation, the relative-position
property, and sequential positions on a chain."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import tree as T


def test_position_zero_is_the_identity():
    x = np.random.default_rng(0).normal(size=(3, 2, 8))
    assert np.allclose(A.rope(x, [0, 0, 0], 10000.0), x, atol=0, rtol=0)


def test_two_dimensions_turn_by_the_position():
    x = np.array([[[1.0, 0.0]]])
    for pos in (1, 7, 1234):
        y = A.rope(x, [pos], 10000.0)[0, 0]
        assert y[0] == pytest.approx(math.cos(pos), abs=1e-12) and y[1] == pytest.approx(math.sin(pos), abs=1e-12)


def test_pairs_keep_their_norms():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 3, 16))
    y = A.rope(x, rng.integers(0, 40000, size=5), 500000.0)
    for j in range(8):
        assert np.allclose(np.hypot(y[..., j], y[..., j + 8]), np.hypot(x[..., j], x[..., j + 8]), atol=1e-12)


def test_scores_depend_on_the_position_difference_only():
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=(1, 1, 64)), rng.normal(size=(1, 1, 64))
    for a, b, c in [(5, 2, 100), (33000, 32990, -32000), (7, 7, 1)]:
        s1 = float(A.rope(q, [a], 10000.0).ravel() @ A.rope(k, [b], 10000.0).ravel())
        s2 = float(A.rope(q, [a + c], 10000.0).ravel() @ A.rope(k, [b + c], 10000.0).ravel())
        assert s1 == pytest.approx(s2, rel=1e-9, abs=1e-9)


def test_tree_positions_are_prefix_plus_depth():
    parent = [-1, 0, 1, 0, 3, 3, -1]
    pos = A.tree_positions(parent, 7, 100)
    assert pos.tolist() == [100 + T.depth(parent, i) for i in range(7)] == [100, 101, 102, 101, 102, 102, 100]
    # a chain's positions are sequential, as in ordinary decoding
    assert A.tree_positions(list(range(-1, 9)), 10, 37).tolist() == list(range(37, 47))


def test_bf16_rounding_is_nearest_even():
    assert A.round_bf16(np.array([1.0, -2.5, 0.0]) ).tolist() == [1.0, -2.5, 0.0]
    one_ulp = 2.0 ** -7                                  # bf16 spacing just above 1
    assert A.round_bf16(np.array([1.0 + one_ulp * 0.5]))[0] == 1.0            # tie: to even (1.0)
    assert A.round_bf16(np.array([1.0 + one_ulp * 1.5]))[0] == 1.0 + 2 * one_ulp   # tie: to even (1 + 2 ulp)
    assert A.round_bf16(np.array([1.0 + one_ulp * 0.51]))[0] == 1.0 + one_ulp
    x = np.random.default_rng(3).normal(size=1000) * 100
    r = A.round_bf16(x)
    assert np.all(r.astype(np.float32).view(np.uint32) & 0xFFFF == 0)
    assert np.all(np.abs(r - x) <= 2.0 ** -8 * np.abs(x) + 1e-30)   # half a unit of the 8-bit significand
