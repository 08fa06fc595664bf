"""fp64 projections on either side of attention.

TEST INFRASTRUCTURE ONLY, under the same rules as the rest of ``oracle/``:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it, and it never imports the product library.

What it computes ("Appendix A.10 -- Attention matrices and backpropagation",
row-vector convention, X [n][d], W_Q, W_K [d][d_h], W_V [d][d_v]):

* eq. A.10.10:  Q = X W_Q,  K = X W_K,  V = X W_V.
* eq. A.10.11:  G_{W_Q} = X^T G_Q (the same for K and V), and
  G_X = G_Q W_Q^T + G_K W_K^T + G_V W_V^T, summed over the branches that
  share X (for cross-attention the query input gets only the query branch and
  the key/value input the other two).

The matrix products are numpy's (a library primitive); everything is fp64.
Pinned by ``tests/test_oracle_proj_pins.py``: worked example 1 of "Computing
attention term by term" run through the projections, and central finite
differences of the whole module (projections + attention) on every
coordinate of X and of each W, with a negative control that drops two of the
three branches of G_X.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np


def proj_forward(X, W) -> np.ndarray:
    """Y = X W (eq. A.10.10): X [n][d], W [d][out]."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


def proj_grad_weight(X, G) -> np.ndarray:
    """G_W = X^T G (eq. A.10.11): X [n][d], G [n][out] -> [d][out]."""
    return np.asarray(X, dtype=np.float64).T @ np.asarray(G, dtype=np.float64)


def proj_grad_input(branches: Sequence[Tuple[np.ndarray, np.ndarray]]) -> np.ndarray:
    """G_X = sum over the (G_b, W_b) branches that share X of G_b W_b^T (eq. A.10.11)."""
    total = None
    for G, W in branches:
        term = np.asarray(G, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T
        total = term if total is None else total + term
    return total


def _heads(Y, n, H, d):
    """[n][H*d] (token-major) -> [1][H][n][d] (the attention oracle's layout)."""
    return np.ascontiguousarray(Y.reshape(n, H, d).transpose(1, 0, 2)[None])


def _tokens(Z):
    """[1][H][n][d] -> [n][H*d]."""
    _, H, n, d = Z.shape
    return np.ascontiguousarray(Z[0].transpose(1, 0, 2).reshape(n, H * d))


def module_forward(orc, p, Xq, Xkv, Wq, Wk, Wv, scale: Optional[float] = None):
    """Projections then attention for one batch element (p.B == 1): queries
    from Xq [n_q][d], keys and values from Xkv [n_k][d] (the same array for
    self-attention).  Returns (Q, K, V, O, LSE) in the attention oracle's
    layout."""
    Q = _heads(proj_forward(Xq, Wq), p.nq, p.Hq, p.dh)
    K = _heads(proj_forward(Xkv, Wk), p.nk, p.Hkv, p.dh)
    V = _heads(proj_forward(Xkv, Wv), p.nk, p.Hkv, p.dv)
    O, LSE = orc.forward(p, Q, K, V, scale=scale)
    return Q, K, V, O, LSE


def module_backward(orc, p, Xq, Xkv, Wq, Wk, Wv, G, scale: Optional[float] = None, self_attention=True):
    """Gradients of sum(G * O) through attention and the projections.

    Returns (dXq, dXkv, dWq, dWk, dWv); for self-attention dXq is the whole
    input gradient (all three branches) and dXkv is None."""
    Q, K, V, _O, _L = module_forward(orc, p, Xq, Xkv, Wq, Wk, Wv, scale=scale)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G, scale=scale)
    gq, gk, gv = _tokens(dQ), _tokens(dK), _tokens(dV)
    dWq, dWk, dWv = proj_grad_weight(Xq, gq), proj_grad_weight(Xkv, gk), proj_grad_weight(Xkv, gv)
    if self_attention:
        return proj_grad_input([(gq, Wq), (gk, Wk), (gv, Wv)]), None, dWq, dWk, dWv
    return proj_grad_input([(gq, Wq)]), proj_grad_input([(gk, Wk), (gv, Wv)]), dWq, dWk, dWv
