"""Pins of the rotary-embedding oracle (oracle/rope.py) to the pages
("Chapter 15 -- matrix formulas", section 15.6; "Chapter 31 -- attention
backprop", section 5): the 2-D rotation itself, R_i^T R_j = R((j - i) w) (the
rotated score depends on the position difference only), orthogonality, and
the backward being the rotation by the opposite angle (checked by finite
differences, with a negative control that uses the forward rotation)."""
import math

import numpy as np

from oracle.rope import frequencies, rope


def test_single_block_is_a_column_vector_rotation():
    # d = 2: one block with w_0 = 1; (1, 0) at position 1 turns to (cos 1, sin 1).
    y = rope(np.array([[1.0, 0.0]]), [1], base=10000.0)
    np.testing.assert_allclose(y, [[math.cos(1.0), math.sin(1.0)]], rtol=0, atol=1e-15)
    y = rope(np.array([[0.0, 1.0]]), [2], base=10000.0)
    np.testing.assert_allclose(y, [[-math.sin(2.0), math.cos(2.0)]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(frequencies(8, 100.0), [1.0, 100 ** -0.25, 100 ** -0.5, 100 ** -0.75], rtol=1e-15)


def test_score_depends_on_position_difference_only():
    rng = np.random.default_rng(1)
    d = 16
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for i, j, shift in ((3, 10, 57), (40, 2, -11), (0, 0, 1000)):
        a = float(rope(q[None], [i])[0] @ rope(k[None], [j])[0])
        b = float(rope(q[None], [i + shift])[0] @ rope(k[None], [j + shift])[0])
        c = float(q @ rope(k[None], [j - i])[0])          # q^T R((j - i) w) k
        assert abs(a - b) < 1e-12 and abs(a - c) < 1e-12


def test_orthogonal_and_inverse():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((5, 3, 8))
    pos = [0, 1, 7, 100, 4096]
    Y = rope(X, pos)
    np.testing.assert_allclose(np.linalg.norm(Y, axis=-1), np.linalg.norm(X, axis=-1), rtol=1e-14)
    np.testing.assert_allclose(rope(Y, pos, inverse=True), X, rtol=0, atol=1e-13)


def _fd_gradient(g, X, pos):
    h, out = 1e-6, np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        p, m = X.copy(), X.copy()
        p[idx] += h
        m[idx] -= h
        out[idx] = (np.sum(g * rope(p, pos)) - np.sum(g * rope(m, pos))) / (2 * h)
    return out


def test_backward_is_the_opposite_rotation():
    rng = np.random.default_rng(3)
    X, g = rng.standard_normal((3, 2, 6)), rng.standard_normal((3, 2, 6))
    pos = [2, 5, 9]
    fd = _fd_gradient(g, X, pos)
    assert np.max(np.abs(fd - rope(g, pos, inverse=True))) < 1e-7
    # negative control: the forward rotation is not the gradient map
    assert np.max(np.abs(fd - rope(g, pos))) > 1e-2
