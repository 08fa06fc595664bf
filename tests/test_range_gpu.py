"""Parity at input scales far outside the fp16 range.

The forward's P V product and every backward product run on fp16 operands,
each tile re-encoded with its own power of two.  "Appendix A.10" eqs.
A.10.1-A.10.9 hold for any real inputs, and the pages restrict no magnitude,
so gradients of 1e-9 or values of 1e5 must come out as accurately as unit
ones.  Every case scales the seeded inputs by exact powers of two (exact in
bf16), runs the CUDA path and the fp64 oracle on the same scaled inputs,
multiplies the outputs back by the known power of two and compares them
element by element at the usual tolerance (|gpu - ref| <= 1e-2 + 2e-2 |ref|,
LSE 1e-3): without the rescaling the absolute 1e-2 would hide any error in
a tiny output.

Scalings: dO x 2^-20 and x 2^-30 (dQ, dK, dV scale with dO); V x 2^17 (O,
dQ, dK scale with V); Q, K x 2^-10 (dQ, dK scale with K, Q at fixed dS);
mixed magnitudes inside one CTA (a query tile's dO, or a key tile's V,
scaled alone, so the per-tile exponents differ; each output is compared at
the scale of the terms that dominate it, since the fp16 weights' rounding
error grows with those terms); an all-zero dO head; and a tile beyond 2^46,
which saturates and must be reported as ATTN_ERR_RANGE.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import Workload, make_inputs

from _attn_cases import LSE_ATOL, assert_close, f64, problem_of, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from exact_scaled_dot_gb300 import build as b
    b.build()
    import exact_scaled_dot_gb300 as esd
    esd.load()
    assert torch.cuda.is_available(), "a CUDA device is required"
    esd.attn_clear_status()
    yield
    assert esd.attn_get_status() == 0


GQA = Workload("range_gqa", B=2, Hq=4, Hkv=2, nq=300, nk=300, dh=128, dv=128, causal=True,
               kv_len_range=(150, 300), seed=91)
CROSS = Workload("range_cross_dv64", B=1, Hq=2, Hkv=1, nq=200, nk=500, dh=128, dv=64, kv_len_range=(200, 500),
                 seed=92)


def _oracle(orc, w, inp):
    p = problem_of(w, inp)
    Q, K, V, G = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    O, LSE = orc.forward(p, Q, K, V)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G)
    return dict(O=O, LSE=LSE, dQ=dQ, dK=dK, dV=dV)


def _compare(res, ref, mult):
    """Outputs times mult[name] (a scalar or an array broadcast over rows)
    against the oracle's times the same factor."""
    assert res.status == 0, f"device status {res.status}"
    for name in ("O", "dQ", "dK", "dV"):
        m = mult.get(name, 1.0)
        assert_close(f64(getattr(res, name)) * m, ref[name] * m, f"{name} x {m if np.isscalar(m) else 'rows'}")
    assert_close(f64(res.LSE), ref["LSE"], "LSE", atol=LSE_ATOL, rtol=0.0)


@pytest.mark.parametrize("w", [GQA, CROSS], ids=lambda w: w.name)
@pytest.mark.parametrize("case", ["dO_2^-20", "dO_2^-30", "V_2^17", "QK_2^-10"])
def test_power_of_two_rescaled_inputs(orc, w, case):
    inp = make_inputs(w)
    if case == "dO_2^-20":
        inp.dO.mul_(2.0 ** -20)
        mult = dict(dQ=2.0 ** 20, dK=2.0 ** 20, dV=2.0 ** 20)
    elif case == "dO_2^-30":
        inp.dO.mul_(2.0 ** -30)
        mult = dict(dQ=2.0 ** 30, dK=2.0 ** 30, dV=2.0 ** 30)
    elif case == "V_2^17":
        inp.V.mul_(2.0 ** 17)
        mult = dict(O=2.0 ** -17, dQ=2.0 ** -17, dK=2.0 ** -17)
    else:
        inp.Q.mul_(2.0 ** -10)
        inp.K.mul_(2.0 ** -10)
        mult = dict(dQ=2.0 ** 10, dK=2.0 ** 10)
    res = run_gpu(w, inp)
    _compare(res, _oracle(orc, w, inp), mult)


def test_mixed_query_tile_magnitudes(orc):
    """Inside one CTA the steps carry different exponents: query rows
    128..255 get dO x 2^-12.  dQ_i is linear in dO_i, so those rows of dQ are
    compared after x 2^12; dK and dV are dominated by the unit rows."""
    w = GQA
    inp = make_inputs(w)
    inp.dO[:, :, 128:256, :] *= 2.0 ** -12
    res = run_gpu(w, inp)
    row = np.ones((1, 1, w.nq, 1))
    row[:, :, 128:256, :] = 2.0 ** 12
    _compare(res, _oracle(orc, w, inp), dict(dQ=row))


def test_mixed_key_tile_magnitudes(orc):
    """Key rows 128..255 get V x 2^10, so the forward's key tiles carry
    different exponents.  Every output that these keys feed grows by 2^10 and
    is compared after x 2^-10: O and dQ of the rows that see them (rows >= 128,
    causal with key lengths >= 150), and dK (every key's gradient collects
    dS terms of those rows); dV = A^T dO does not involve V."""
    w = GQA
    inp = make_inputs(w)
    inp.V[:, :, 128:256, :] *= 2.0 ** 10
    res = run_gpu(w, inp)
    row = np.ones((1, 1, w.nq, 1))
    row[:, :, 128:, :] = 2.0 ** -10
    _compare(res, _oracle(orc, w, inp), dict(O=row, dQ=row, dK=2.0 ** -10))


def test_zero_gradient_head(orc):
    """One query head with dO = 0: its dQ rows are exactly zero, the other
    heads are unaffected (all-zero tiles carry no exponent of their own)."""
    w = GQA
    inp = make_inputs(w)
    inp.dO[:, 1] = 0
    inp.Q[:, 2] = 0
    res = run_gpu(w, inp)
    _compare(res, _oracle(orc, w, inp), {})
    assert int(torch.count_nonzero(res.dQ[:, 1])) == 0


@pytest.mark.parametrize("what", ["V", "dO"])
def test_saturating_tile_is_reported(what):
    """A tile whose largest magnitude is 2^52 (above the 2^46 the clamped
    exponents reach) saturates in fp16: the call must record ATTN_ERR_RANGE
    in the status word, and later calls run normally once it is cleared."""
    import exact_scaled_dot_gb300 as esd
    w = GQA
    inp = make_inputs(w)
    getattr(inp, what)[0, 0, 0, 0] = 2.0 ** 52
    res = run_gpu(w, inp)
    assert res.status == esd.ATTN_ERR_RANGE
    esd.attn_clear_status()
    clean = make_inputs(w)
    again = run_gpu(w, clean)
    assert again.status == 0
