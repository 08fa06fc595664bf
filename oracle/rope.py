"""fp64 rotary position embedding.

TEST INFRASTRUCTURE ONLY, under the same rules as the rest of ``oracle/``.

What it computes ("Chapter 15 -- matrix formulas", section 15.6: rotate the
2-D blocks of q and k by position-dependent angles before the dot product,
q~_i = R_i q_i, k~_j = R_j k_j, with R_i^T R_j = R((j - i) w); "Chapter 31 --
attention backprop", section 5: the backward rotates the upstream gradient by
the opposite angle).  Block k of a row is its pair of components (2k, 2k+1)
and turns by a = pos * w_k, w_k = base^(-2k/d) (the pages fix only "position
times a fixed frequency"; the frequency schedule is the plainest common
reading and is a parameter).  Column-vector rotation R(a) = [[cos, -sin],
[sin, cos]].  Angles are exact in double precision.

Pinned by ``tests/test_oracle_rope_pins.py``.
"""
from __future__ import annotations

import numpy as np


def frequencies(d: int, base: float) -> np.ndarray:
    """w_k = base^(-2k/d), k < d/2."""
    return np.power(float(base), -2.0 * np.arange(d // 2) / d)


def rope(X, positions, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotate every row of X [tokens][heads][d] (or [tokens][d]) at positions [tokens]."""
    X = np.asarray(X, dtype=np.float64)
    squeeze = X.ndim == 2
    if squeeze:
        X = X[:, None, :]
    T, H, d = X.shape
    a = np.asarray(positions, dtype=np.float64)[:, None] * frequencies(d, base)[None, :]   # [T][d/2]
    if inverse:
        a = -a
    c, s = np.cos(a)[:, None, :], np.sin(a)[:, None, :]
    x0, x1 = X[..., 0::2], X[..., 1::2]
    Y = np.empty_like(X)
    Y[..., 0::2] = x0 * c - x1 * s
    Y[..., 1::2] = x0 * s + x1 * c
    return Y[:, 0, :] if squeeze else Y
