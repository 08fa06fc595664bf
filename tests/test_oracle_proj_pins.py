"""Pins of the projection oracle (oracle/projections.py) to the pages.

* Worked example 1 of "Computing attention term by term" starts from
  projections: X = I, W_Q = sqrt(2) ln(3) I, W_K = I, W_V = diag(2, 4).  Run
  through the projections and the attention oracle, it must give the page's
  O and J = 15/2, and with X = I the weight gradients are the page's
  dQ, dK and dV themselves (eq. A.10.11, G_W = X^T G).
* Central finite differences (fp64, steps 1e-5 and 1e-6, bound 1e-7) of the
  whole module (projections + attention) on every coordinate of X and of each
  W, for self-attention (shared X: G_X sums three branches) and for
  cross-attention (query input one branch, key/value input two).
* Negative control: keeping only the value branch of G_X ("the branches must
  be added; the value branch computed last must not overwrite the others",
  same page) fails the finite-difference check.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest

from oracle import Problem
from oracle.projections import module_backward, module_forward, proj_grad_input, proj_grad_weight

GOLDEN = Path(__file__).resolve().parent / "golden"


def _expr(v):
    return float(eval(v, {"sqrt": math.sqrt, "log": math.log}))   # fixture expressions only


def test_worked_example_1_through_the_projections(orc):
    fx = json.loads((GOLDEN / "worked_example_1.json").read_text())
    a = math.sqrt(2) * math.log(3)
    X = np.eye(2)
    Wq, Wk, Wv = a * np.eye(2), np.eye(2), np.diag([2.0, 4.0])
    p = Problem(1, 1, 1, 2, 2, 2, 2)
    G = np.array([[[[1.0, 0.0], [0.0, 2.0]]]])
    _Q, _K, _V, O, _L = module_forward(orc, p, X, X, Wq, Wk, Wv, scale=1 / math.sqrt(2))
    expO = np.array([[_expr(v) for v in row] for row in fx["expected"]["O"]])
    np.testing.assert_allclose(O[0, 0], expO, rtol=0, atol=1e-13)
    assert abs(float(np.sum(O * G)) - _expr(fx["expected"]["J"])) < 1e-13
    _dX, _n, dWq, dWk, dWv = module_backward(orc, p, X, X, Wq, Wk, Wv, G, scale=1 / math.sqrt(2))
    for key, got in (("dQ", dWq), ("dK", dWk), ("dV", dWv)):
        exp = np.array([[_expr(v) for v in row] for row in fx["expected"][key]])
        np.testing.assert_allclose(got, exp, rtol=0, atol=1e-13, err_msg=key)


def _fd_module(orc, p, Xq, Xkv, Ws, G, self_attention, grad_fn):
    """Largest |central FD - analytic| over every coordinate of the inputs."""
    def loss(xq, xkv, wq, wk, wv):
        _Q, _K, _V, O, _L = module_forward(orc, p, xq, xq if self_attention else xkv, wq, wk, wv)
        return float(np.sum(O * G))

    analytic = grad_fn(Xq, Xkv, *Ws)
    inputs = [Xq, Xkv] + list(Ws)
    names = ["Xq", "Xkv", "Wq", "Wk", "Wv"]
    worst = {}
    for h in (1e-5, 1e-6):
        for f, x in enumerate(inputs):
            if analytic[f] is None:
                continue
            for idx in np.ndindex(x.shape):
                plus = [a.copy() for a in inputs]
                minus = [a.copy() for a in inputs]
                plus[f][idx] += h
                minus[f][idx] -= h
                fd = (loss(*plus) - loss(*minus)) / (2 * h)
                worst[names[f]] = max(worst.get(names[f], 0.0), abs(fd - analytic[f][idx]))
    return worst


@pytest.mark.parametrize("causal", [False, True])
def test_fd_self_attention_shared_input(orc, causal):
    rng = np.random.default_rng(21 + causal)
    n, d, dh, dv = 3, 4, 2, 3
    p = Problem(1, 1, 1, n, n, dh, dv, causal=causal)
    X = rng.standard_normal((n, d))
    Ws = [rng.standard_normal((d, dh)) * 0.7, rng.standard_normal((d, dh)) * 0.7, rng.standard_normal((d, dv))]
    G = rng.standard_normal((1, 1, n, dv))

    def grads(xq, _xkv, wq, wk, wv):
        dX, _n, dWq, dWk, dWv = module_backward(orc, p, xq, xq, wq, wk, wv, G)
        return [dX, None, dWq, dWk, dWv]

    worst = _fd_module(orc, p, X, X, Ws, G, True, grads)
    assert max(worst.values()) < 1e-7, worst


def test_fd_cross_attention_two_inputs(orc):
    rng = np.random.default_rng(31)
    nq, nk, d, dh, dv = 2, 4, 3, 2, 2
    p = Problem(1, 2, 1, nq, nk, dh, dv)   # two query heads sharing one KV head
    Xq, Xkv = rng.standard_normal((nq, d)), rng.standard_normal((nk, d))
    Ws = [rng.standard_normal((d, 2 * dh)) * 0.7, rng.standard_normal((d, dh)) * 0.7, rng.standard_normal((d, dv))]
    G = rng.standard_normal((1, 2, nq, dv))

    def grads(xq, xkv, wq, wk, wv):
        return list(module_backward(orc, p, xq, xkv, wq, wk, wv, G, self_attention=False))

    worst = _fd_module(orc, p, Xq, Xkv, Ws, G, False, grads)
    assert max(worst.values()) < 1e-7, worst


def test_negative_control_value_branch_alone_fails_fd(orc):
    rng = np.random.default_rng(22)
    n, d, dh, dv = 3, 4, 2, 3
    p = Problem(1, 1, 1, n, n, dh, dv)
    X = rng.standard_normal((n, d))
    Ws = [rng.standard_normal((d, dh)) * 0.7, rng.standard_normal((d, dh)) * 0.7, rng.standard_normal((d, dv))]
    G = rng.standard_normal((1, 1, n, dv))
    from oracle.projections import _tokens

    def grads_value_only(xq, _xkv, wq, wk, wv):
        dX, _n, dWq, dWk, dWv = module_backward(orc, p, xq, xq, wq, wk, wv, G)
        Q, K, V, _O, _L = module_forward(orc, p, xq, xq, wq, wk, wv)
        _dQ, _dK, dV, _D, _C = orc.backward(p, Q, K, V, G)
        return [proj_grad_input([(_tokens(dV), wv)]), None, dWq, dWk, dWv]

    worst = _fd_module(orc, p, X, X, Ws, G, True, grads_value_only)
    assert worst["Xq"] > 1e-3, worst


def test_weight_gradient_is_a_token_sum():
    """G_W = X^T G equals the sum over tokens of outer products x_t g_t^T."""
    rng = np.random.default_rng(5)
    X, G = rng.standard_normal((7, 3)), rng.standard_normal((7, 2))
    outer = sum(np.outer(X[t], G[t]) for t in range(7))
    np.testing.assert_allclose(proj_grad_weight(X, G), outer, rtol=1e-14, atol=1e-14)
