"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Every test here checks the oracle against something other than itself: the
worked examples printed on "Computing attention term by term" (fixtures under
tests/golden/), closed forms, invariants stated in "Appendix A.10 -- Attention
matrices and backpropagation" and "Chapter 31 -- attention backprop", central
finite differences, and negative controls that break the oracle on purpose
and must be caught.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest

import oracle
from oracle import Oracle, Problem

GOLDEN = Path(__file__).parent / "golden"


def _ev(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt, "log": math.log}))


def _arr(x):
    if isinstance(x, list):
        return np.array([_arr(e) for e in x], dtype=np.float64)
    return _ev(x)


def _fixture(name):
    fx = json.loads((GOLDEN / name).read_text())
    out = {"scale": _ev(fx["scale"]), "d": fx["d"]}
    out["inputs"] = {k: _arr(v) for k, v in fx["inputs"].items()}
    out["expected"] = {k: _arr(v) for k, v in fx["expected"].items()}
    return out


def _single(x):
    return x[None, None]


def _example(orc, name):
    fx = _fixture(name)
    I = fx["inputs"]
    n, d = I["Q"].shape
    p = Problem(1, 1, 1, n, I["K"].shape[0], d, I["V"].shape[1])
    S, A, dA, dS = orc.dense(p, _single(I["Q"]), _single(I["K"]), _single(I["V"]),
                             _single(I["G"]), scale=fx["scale"])
    O, LSE = orc.forward(p, _single(I["Q"]), _single(I["K"]), _single(I["V"]), scale=fx["scale"])
    dQ, dK, dV, D, C = orc.backward(p, _single(I["Q"]), _single(I["K"]), _single(I["V"]),
                                    _single(I["G"]), scale=fx["scale"])
    got = dict(S=S[0, 0], A=A[0, 0], dA=dA[0, 0], dS=dS[0, 0], O=O[0, 0], LSE=LSE[0, 0],
               dQ=dQ[0, 0], dK=dK[0, 0], dV=dV[0, 0], c=C[0, 0], D=D[0, 0])
    got["J"] = float(np.sum(got["O"] * I["G"]))
    return fx["expected"], got


@pytest.mark.parametrize("name", ["worked_example_1.json", "worked_example_2.json"])
def test_worked_examples(orc, name):
    exp, got = _example(orc, name)
    for key, val in exp.items():
        np.testing.assert_allclose(got[key], val, rtol=0, atol=1e-13, err_msg=key)
    # c_i (A.10.7) and rowsum(G*O) agree exactly in real arithmetic.
    np.testing.assert_allclose(got["D"], exp["c"], rtol=0, atol=1e-13)


def test_worked_example_2_query_gradient_is_exactly_zero(orc):
    _exp, got = _example(orc, "worked_example_2.json")
    assert np.all(got["dQ"] == 0.0)
    assert np.any(got["dK"] != 0.0)


def test_transpose_check(orc):
    fx = _fixture("transpose_check.json")
    Q, K = fx["inputs"]["Q"], fx["inputs"]["K"]
    p = Problem(1, 1, 1, 2, 2, 2, 2)
    S, _A, _, _ = orc.dense(p, _single(Q), _single(K), _single(np.zeros((2, 2))), scale=fx["scale"])
    np.testing.assert_array_equal(S[0, 0], fx["expected"]["QKt"])
    assert not np.array_equal(S[0, 0], fx["expected"]["wrong_QK"])
    # The log-sum-exp rows differ between the two orientations as well.
    _O, LSE = orc.forward(p, _single(Q), _single(K), _single(np.eye(2)), scale=1.0)
    np.testing.assert_allclose(LSE[0, 0], [math.log(math.e + math.e ** 4), math.log(1 + math.e)],
                               rtol=1e-14)


def _random_problem(rng, p, scale_qk=1.0):
    Q = rng.standard_normal((p.B, p.Hq, p.nq, p.dh)) * scale_qk
    K = rng.standard_normal((p.B, p.Hkv, p.nk, p.dh)) * scale_qk
    V = rng.standard_normal((p.B, p.Hkv, p.nk, p.dv))
    G = rng.standard_normal((p.B, p.Hq, p.nq, p.dv))
    return Q, K, V, G


def test_two_position_jacobian_closed_form(orc):
    """n_k = 2: dS row = a(1-a)(u-v) * [1, -1] (end of worked example 2)."""
    rng = np.random.default_rng(7)
    p = Problem(1, 2, 1, 5, 2, 3, 4)
    Q, K, V, G = _random_problem(rng, p)
    _S, A, _dA, dS = orc.dense(p, Q, K, V, G)
    for r in range(p.Hq):
        dA = G[0, r] @ V[0, 0].T            # upstream weight gradient, eq. A.10.6
        a = A[0, r, :, 0]
        u, v = dA[:, 0], dA[:, 1]
        expect = a * (1 - a) * (u - v)
        np.testing.assert_allclose(dS[0, r, :, 0], expect, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dS[0, r, :, 1], -expect, rtol=1e-12, atol=1e-15)
    # u == v (identical value rows): the score gradient vanishes.
    V2 = np.repeat(V[:, :, :1, :], 2, axis=2)
    _S, _A, _dA, dS2 = orc.dense(p, Q, K, V2, G)
    np.testing.assert_allclose(dS2, 0.0, atol=1e-15)


MASKS = [
    dict(name="full", nq=4, nk=4),
    dict(name="causal", nq=4, nk=4, causal=True),
    dict(name="causal_offset", nq=3, nk=5, causal=True),            # offset n_k - n_q = 2
    dict(name="causal_offset0", nq=3, nk=5, causal=True, offset=0),
    dict(name="padded", nq=4, nk=4, kv_len=(3, 2)),
    dict(name="causal_padded", nq=4, nk=4, causal=True, kv_len=(4, 2)),
    dict(name="cross", nq=2, nk=4, kv_len=(3, 4)),
]


def _mk(spec, B=2, Hq=2, Hkv=1, dh=3, dv=2):
    return Problem(B, Hq, Hkv, spec["nq"], spec["nk"], dh, dv, causal=spec.get("causal", False),
                   offset=spec.get("offset"), kv_len=spec.get("kv_len"))


def _fd_max_error(o: Oracle, p: Problem, seed: int):
    """Central differences of L = sum(O * G) on every coordinate of Q, K and V."""
    rng = np.random.default_rng(seed)
    Q, K, V, G = _random_problem(rng, p)
    dQ, dK, dV, _D, _C = o.backward(p, Q, K, V, G)
    analytic = [dQ, dK, dV]

    def loss(q, k, v):
        O, _ = o.forward(p, q, k, v)
        return float(np.sum(O * G))

    worst = 0.0
    for h in (1e-5, 1e-6):
        for field in range(3):
            base = [Q, K, V]
            x = base[field]
            for idx in np.ndindex(x.shape):
                plus = [a.copy() for a in base]
                minus = [a.copy() for a in base]
                plus[field][idx] += h
                minus[field][idx] -= h
                fd = (loss(*plus) - loss(*minus)) / (2 * h)
                worst = max(worst, abs(fd - analytic[field][idx]))
    return worst


@pytest.mark.parametrize("spec", MASKS, ids=[m["name"] for m in MASKS])
def test_finite_differences_every_coordinate(orc, spec):
    """Central FD (eps 1e-5 and 1e-6, fp64) on all of Q, K, V; threshold 1e-7."""
    p = _mk(spec)
    assert _fd_max_error(orc, p, seed=11) < 1e-7


def _causal_locality(o: Oracle):
    """Chapter 31 section 6: causal mask, only query row 0 enters the loss."""
    p = Problem(1, 1, 1, 4, 4, 3, 2, causal=True, offset=0)
    rng = np.random.default_rng(3)
    Q, K, V, G = _random_problem(rng, p)
    G[:, :, 1:, :] = 0.0
    dQ, dK, dV, _D, _C = o.backward(p, Q, K, V, G)
    ok = True
    ok &= bool(np.all(dQ[0, 0, 1:] == 0.0))
    ok &= bool(np.allclose(dK, 0.0, atol=1e-15))
    ok &= bool(np.allclose(dV[0, 0, 0], G[0, 0, 0], atol=1e-15))
    ok &= bool(np.allclose(dV[0, 0, 1:], 0.0, atol=1e-15))
    return ok


def test_causal_future_gradients_zero(orc):
    assert _causal_locality(orc)


@pytest.fixture(scope="module")
def mutated(tmp_path_factory):
    d = tmp_path_factory.mktemp("oracle_mutants")
    return {m: Oracle(oracle.build(mutation=m, out_dir=d)) for m in (1, 2)}


def test_negative_control_drop_row_term_fails_fd(mutated):
    """Chapter 31 section 8: without the row term c_i the FD check must fail."""
    p = _mk(MASKS[0])
    assert _fd_max_error(mutated[1], p, seed=11) > 1e-3


def test_negative_control_drop_mask_fails_locality(mutated):
    """Chapter 31 section 8: without the mask the causal-gradient test must fail."""
    assert not _causal_locality(mutated[2])


def test_invariants_random(orc):
    """A rows are convex weights, O lies in the hull of visible V rows, rows of
    dS sum to zero, dS vanishes off the visible set, and rowsum(G*O) = c_i."""
    rng = np.random.default_rng(5)
    p = Problem(2, 4, 2, 37, 53, 8, 5, causal=True, offset=16, kv_len=(40, 23))
    Q, K, V, G = _random_problem(rng, p, scale_qk=2.0)
    S, A, _dA, dS = orc.dense(p, Q, K, V, G)
    O, LSE = orc.forward(p, Q, K, V)
    _dQ, _dK, _dV, D, C = orc.backward(p, Q, K, V, G)
    visible = ~np.isnan(S)
    assert np.all(A >= 0)
    assert np.all(A[~visible] == 0)
    np.testing.assert_allclose(A.sum(-1), 1.0, atol=1e-13)
    assert np.all(dS[~visible] == 0)
    np.testing.assert_allclose(dS.sum(-1), 0.0, atol=1e-13)
    np.testing.assert_allclose(D, C, rtol=1e-12, atol=1e-13)
    group = p.Hq // p.Hkv
    for b in range(p.B):
        for r in range(p.Hq):
            Vh = V[b, r // group]
            for i in range(p.nq):
                vis = visible[b, r, i]
                lo = Vh[vis].min(0) - 1e-12
                hi = Vh[vis].max(0) + 1e-12
                assert np.all(O[b, r, i] >= lo) and np.all(O[b, r, i] <= hi)
                # LSE is the log of the visible exponential sum.
                s = S[b, r, i][vis]
                assert abs(LSE[b, r, i] - (s.max() + math.log(np.exp(s - s.max()).sum()))) < 1e-12


def test_visible_set_matches_definition(orc):
    """The visible set is {j : j <= i + offset (causal), j < kv_len[b]}."""
    p = Problem(2, 1, 1, 5, 7, 2, 2, causal=True, offset=1, kv_len=(6, 3))
    rng = np.random.default_rng(2)
    Q, K, V, _G = _random_problem(rng, p)
    S, _A, _, _ = orc.dense(p, Q, K, V)
    for b, L in enumerate(p.kv_len):
        for i in range(p.nq):
            for j in range(p.nk):
                assert (not np.isnan(S[b, 0, i, j])) == (j <= i + 1 and j < L)
    assert orc.visible_pairs(p) == int((~np.isnan(S)).sum())


def test_single_visible_key_closed_form(orc):
    """kv_len = 1: A = e_0, so O_i = v_0, LSE_i = S_i0, dS = 0, dQ = dK = 0, dV_0 = sum G."""
    p = Problem(1, 2, 1, 3, 4, 3, 2, kv_len=(1,))
    rng = np.random.default_rng(4)
    Q, K, V, G = _random_problem(rng, p)
    O, LSE = orc.forward(p, Q, K, V)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G)
    s = 1 / math.sqrt(p.dh)
    for r in range(p.Hq):
        np.testing.assert_array_equal(O[0, r], np.broadcast_to(V[0, 0, 0], O[0, r].shape))
        np.testing.assert_allclose(LSE[0, r], s * (Q[0, r] @ K[0, 0, 0]), rtol=1e-14)
    assert np.all(dQ == 0) and np.all(dK == 0)
    np.testing.assert_allclose(dV[0, 0, 0], G[0].sum(axis=(0, 1)), rtol=1e-13)
    assert np.all(dV[0, 0, 1:] == 0)


def test_permutation_equivariance_without_mask(orc):
    """Chapter 15 section 15.6: without a mask, permuting query rows permutes O
    and dQ rows; permuting key/value rows together leaves O unchanged and
    permutes dK, dV rows."""
    rng = np.random.default_rng(9)
    p = Problem(1, 2, 1, 6, 5, 4, 3)
    Q, K, V, G = _random_problem(rng, p)
    O, _ = orc.forward(p, Q, K, V)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G)
    pq = rng.permutation(p.nq)
    pk = rng.permutation(p.nk)
    O2, _ = orc.forward(p, Q[:, :, pq], K, V)
    dQ2, dK2, dV2, _, _ = orc.backward(p, Q[:, :, pq], K, V, G[:, :, pq])
    np.testing.assert_allclose(O2, O[:, :, pq], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dQ2, dQ[:, :, pq], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dK2, dK, rtol=1e-12, atol=1e-14)
    O3, _ = orc.forward(p, Q, K[:, :, pk], V[:, :, pk])
    dQ3, dK3, dV3, _, _ = orc.backward(p, Q, K[:, :, pk], V[:, :, pk], G)
    np.testing.assert_allclose(O3, O, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dK3, dK[:, :, pk], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dV3, dV[:, :, pk], rtol=1e-12, atol=1e-14)


def test_gqa_heads_read_their_group_and_gradients_sum(orc):
    """Appendix A.10 section A.10.5: query head r reads KV head g(r) = r // (Hq/Hkv);
    dK, dV of a KV head are the sums over the query heads that share it."""
    rng = np.random.default_rng(13)
    p = Problem(2, 4, 2, 5, 6, 3, 2, causal=True, kv_len=(6, 4))
    Q, K, V, G = _random_problem(rng, p)
    O, _ = orc.forward(p, Q, K, V)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G)
    acc_k = np.zeros_like(dK)
    acc_v = np.zeros_like(dV)
    for b in range(p.B):
        for r in range(p.Hq):
            h = r // 2
            single = Problem(1, 1, 1, p.nq, p.nk, p.dh, p.dv, causal=True, kv_len=(p.kv_len[b],))
            args = (Q[b:b + 1, r:r + 1], K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1])
            o1, _ = orc.forward(single, *args)
            np.testing.assert_allclose(o1[0, 0], O[b, r], rtol=1e-14, atol=1e-15)
            q1, k1, v1, _, _ = orc.backward(single, *args, G[b:b + 1, r:r + 1])
            np.testing.assert_allclose(q1[0, 0], dQ[b, r], rtol=1e-13, atol=1e-15)
            acc_k[b, h] += k1[0, 0]
            acc_v[b, h] += v1[0, 0]
    np.testing.assert_allclose(dK, acc_k, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dV, acc_v, rtol=1e-12, atol=1e-14)


def test_empty_rows_are_detected_and_refused(orc):
    """A.10.2 is undefined on an empty visible set; Chapter 31 section 3 rejects it."""
    bad = Problem(1, 1, 1, 3, 3, 2, 2, causal=True, offset=-1)
    assert orc.first_empty_row(bad) == 0
    Q = np.ones((1, 1, 3, 2)); K = np.ones((1, 1, 3, 2)); V = np.ones((1, 1, 3, 2))
    with pytest.raises(ValueError):
        orc.forward(bad, Q, K, V)
    assert orc.first_empty_row(Problem(2, 1, 1, 3, 3, 2, 2, kv_len=(3, 0))) == 3
    assert orc.first_empty_row(Problem(1, 1, 1, 3, 3, 2, 2, causal=True)) == -1


def test_sampled_rows_equal_full(orc):
    """The row-selected entry points give the same numbers as the full ones."""
    rng = np.random.default_rng(21)
    p = Problem(2, 4, 2, 19, 23, 8, 6, causal=True, kv_len=(20, 9))
    Q, K, V, G = _random_problem(rng, p)
    O, LSE = orc.forward(p, Q, K, V)
    dQ, dK, dV, D, C = orc.backward(p, Q, K, V, G)
    rows = np.array([0, 5, 18, 19, 77, 151])
    keys = np.array([0, 8, 9, 22, 45, 91])
    Os, Ls = orc.forward(p, Q, K, V, rows=rows)
    dQs, dKs, dVs, Ds, Cs = orc.backward(p, Q, K, V, G, q_rows=rows, k_rows=keys)
    np.testing.assert_array_equal(Os, O.reshape(-1, p.dv)[rows])
    np.testing.assert_array_equal(Ls, LSE.reshape(-1)[rows])
    np.testing.assert_array_equal(dQs, dQ.reshape(-1, p.dh)[rows])
    np.testing.assert_array_equal(Ds, D.reshape(-1)[rows])
    np.testing.assert_array_equal(dKs, dK.reshape(-1, p.dh)[keys])
    np.testing.assert_array_equal(dVs, dV.reshape(-1, p.dv)[keys])
