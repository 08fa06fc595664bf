"""GPU-vs-oracle parity of the CUDA forward and backward (through the C ABI).

Small problems are compared element by element; they span several 128-row
tiles and a ragged tail.  The five full-size workloads are compared on
sampled rows that the oracle computes one by one.  Tolerances:
|gpu - ref| <= 1e-2 + 2e-2 |ref| for O, dQ, dK, dV and 1e-3 absolute for LSE.
"""
import math

import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import WORKLOAD_ORDER, WORKLOADS, Workload, make_inputs

from _attn_cases import compare_full, compare_sampled, f64, problem_of, run_gpu

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


SMALL = {
    # name: workload (seed fixed per case)
    "single_head_full": WORKLOADS["single_head_full"],
    "mha_causal_ragged": Workload("mha_causal_ragged", B=2, Hq=2, Hkv=2, nq=300, nk=300, dh=128, dv=128,
                                  causal=True, seed=11),
    "gqa_causal_padded": Workload("gqa_causal_padded", B=2, Hq=4, Hkv=2, nq=333, nk=333, dh=128, dv=128,
                                  causal=True, kv_len_range=(140, 333), seed=12),
    "cross_padded_peaked": Workload("cross_padded_peaked", B=2, Hq=2, Hkv=2, nq=200, nk=700, dh=128, dv=64,
                                    kv_len_range=(300, 700), sigma_qk=3.0, seed=13),
    "cross_padded_peaked_2": Workload("cross_padded_peaked_2", B=2, Hq=2, Hkv=2, nq=256, nk=1024, dh=128, dv=64,
                                      kv_len_range=(512, 1024), sigma_qk=3.0, seed=99),
    "mqa_chunked_prefill": Workload("mqa_chunked_prefill", B=1, Hq=4, Hkv=1, nq=130, nk=520, dh=128, dv=128,
                                    causal=True, seed=14),
    "d64_causal_gqa": Workload("d64_causal_gqa", B=1, Hq=4, Hkv=1, nq=257, nk=257, dh=64, dv=64, causal=True,
                               seed=15),
    "d64_full_cross": Workload("d64_full_cross", B=3, Hq=2, Hkv=1, nq=100, nk=390, dh=64, dv=64,
                               kv_len_range=(1, 390), seed=16),
    "explicit_offset_zero": Workload("explicit_offset_zero", B=1, Hq=2, Hkv=2, nq=150, nk=400, dh=128, dv=128,
                                     causal=True, offset=0, seed=17),
    "more_queries_than_keys": Workload("more_queries_than_keys", B=1, Hq=1, Hkv=1, nq=300, nk=50, dh=128, dv=64,
                                       seed=18),
    "single_row": Workload("single_row", B=1, Hq=1, Hkv=1, nq=1, nk=1, dh=64, dv=64, causal=True, seed=19),
    "causal_large_offset": Workload("causal_large_offset", B=2, Hq=2, Hkv=1, nq=129, nk=260, dh=128, dv=128,
                                    causal=True, offset=5000, kv_len_range=(129, 260), seed=20),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_elementwise(orc, name):
    w = SMALL[name]
    inp = make_inputs(w)
    res = run_gpu(w, inp)
    compare_full(w, inp, res, orc)


def test_small_second_seed(orc):
    w = SMALL["gqa_causal_padded"]
    inp = make_inputs(w, seed=2012)
    compare_full(w, inp, run_gpu(w, inp), orc)


def test_key_length_one(orc):
    """kv_len = 1 for every batch element: A = e_0, O_i = v_0 exactly, and dQ, dK
    vanish up to rounding (dP and D are summed in different orders on the GPU,
    so dS is of the order of 1e-7 rather than exactly 0)."""
    w = Workload("kv1", B=2, Hq=2, Hkv=1, nq=140, nk=200, dh=128, dv=128, kv_len_range=(1, 1), seed=21)
    inp = make_inputs(w)
    res = run_gpu(w, inp)
    compare_full(w, inp, res, orc)
    for b in range(w.B):
        for r in range(w.Hq):
            assert torch.equal(res.O[b, r], inp.V[b, 0, 0].to(res.O.device).expand(w.nq, w.dv))
    assert float(res.dQ.float().abs().max()) <= 1e-4 and float(res.dK.float().abs().max()) <= 1e-4


def test_nan_in_key_padding_does_not_leak(orc):
    """Key rows beyond kv_len may hold anything (here NaN); results must equal
    the oracle's, which never reads them."""
    w = Workload("nan_pad", B=2, Hq=2, Hkv=1, nq=200, nk=300, dh=128, dv=128, causal=True,
                 kv_len_range=(130, 250), seed=22)
    inp = make_inputs(w)
    for b, L in enumerate(inp.kv_len.tolist()):
        inp.K[b, :, L:, :] = float("nan")
        inp.V[b, :, L:, :] = float("nan")
    res = run_gpu(w, inp)
    # The oracle never looks at padded rows; give it zeros there to be sure.
    clean = make_inputs(w)
    for b, L in enumerate(clean.kv_len.tolist()):
        clean.K[b, :, L:, :] = 0
        clean.V[b, :, L:, :] = 0
    compare_full(w, clean, res, orc)


def test_transpose_orientation_on_gpu(orc):
    """The asymmetric pair Q=[[1,2],[0,1]], K=[[1,0],[2,1]] ("Computing attention
    term by term", section I), zero-padded to d = 64, scale 1: the log-sum-exp rows
    must follow Q K^T = [[1,4],[0,1]], not [[5,2],[2,1]]."""
    w = Workload("transpose", B=1, Hq=1, Hkv=1, nq=2, nk=2, dh=64, dv=64, seed=0)
    inp = make_inputs(w)
    inp.Q.zero_(); inp.K.zero_(); inp.V.zero_()
    inp.Q[0, 0, 0, :2] = torch.tensor([1.0, 2.0]); inp.Q[0, 0, 1, :2] = torch.tensor([0.0, 1.0])
    inp.K[0, 0, 0, :2] = torch.tensor([1.0, 0.0]); inp.K[0, 0, 1, :2] = torch.tensor([2.0, 1.0])
    inp.V[0, 0, :, :2] = torch.eye(2)
    res = run_gpu(w, inp, scale=1.0)
    lse = f64(res.LSE)[0, 0]
    np.testing.assert_allclose(lse, [math.log(math.e + math.e ** 4), math.log(1 + math.e)], atol=1e-3)
    compare_full(w, inp, res, orc, scale=1.0)


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_full_size_sampled(orc, name):
    """Each full-size workload at its own seed, in the launch configuration the
    benchmark times, compared on sampled rows."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    res = run_gpu(w, inp)
    if name == "single_head_full":
        compare_full(w, inp, res, orc)
    else:
        compare_sampled(w, inp, res, orc)


def test_visible_pairs_closed_form_matches_oracle(orc):
    """The library's closed-form pair count (used to classify tiles and to count
    FLOPs) agrees with the oracle's pair-by-pair count."""
    import exact_scaled_dot_gb300 as esd
    for w in list(SMALL.values())[:6]:
        inp = make_inputs(w)
        kv = None if inp.kv_len is None else inp.kv_len.tolist()
        got = esd.attn_visible_pairs(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal,
                                     causal_offset=w.causal_offset if w.causal else None, kv_len=kv)
        assert got == orc.visible_pairs(problem_of(w, inp))
