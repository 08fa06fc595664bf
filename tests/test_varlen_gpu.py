"""GPU-vs-oracle parity of the packed variable-length entry points
(attn_fwd_varlen, attn_bwd_varlen): token-major tensors, per-sequence query
and key lengths, causal masks aligned bottom-right inside each sequence.

The reference is the fp64 oracle run once per sequence (a B = 1 problem with
that sequence's lengths and default offset len_k - len_q), its outputs packed
back to the token-major layout; every output element is compared (O, dQ, dK,
dV within 1e-2 + 2e-2 |ref|, LSE within 1e-3).  Outputs start as NaN, so an
element the kernels fail to write fails the comparison.  The cases cover
lengths around the 128-row tiles, a single token, cross-length sequences, MQA
chunks over a history, a sequence with no queries (its keys get dK = dV = 0),
d_v = 64 with a peaked softmax, and a single sequence checked against the
padded [B][H][n][d] entry points.
"""
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, make_varlen_inputs

from _attn_cases import LSE_ATOL, assert_close, assert_same_sum, f64, varlen_reference

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


CASES = {
    "mixed_causal_gqa": VarlenWorkload("mixed_causal_gqa", B=4, Hq=8, Hkv=2, dh=128, dv=128, causal=True,
                                       lens_q=(1, 127, 300, 513), seed=61),
    "cross_lengths_full": VarlenWorkload("cross_lengths_full", B=3, Hq=4, Hkv=4, dh=128, dv=128,
                                         lens_q=(200, 129, 64), lens_k=(700, 5, 333), seed=62),
    "mqa_chunks_over_history": VarlenWorkload("mqa_chunks_over_history", B=3, Hq=8, Hkv=1, dh=128, dv=128,
                                              causal=True, lens_q=(16, 100, 1), lens_k=(600, 100, 1000), seed=63),
    "zero_query_sequence_d64": VarlenWorkload("zero_query_sequence_d64", B=3, Hq=4, Hkv=2, dh=64, dv=64,
                                              causal=True, lens_q=(130, 0, 77), lens_k=(130, 40, 77), seed=64),
    "dv64_peaked": VarlenWorkload("dv64_peaked", B=2, Hq=4, Hkv=2, dh=128, dv=64, lens_q=(257, 64),
                                  lens_k=(400, 1000), sigma_qk=3.0, seed=65),
    "drawn_lengths": VarlenWorkload("drawn_lengths", B=5, Hq=4, Hkv=1, dh=128, dv=128, causal=True,
                                    len_range=(1, 400), seed=66),
}


def _run(w: VarlenWorkload, inp, dev="cuda:0"):
    import exact_scaled_dot_gb300 as esd
    Q, K, V, G = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    nan = float("nan")
    O = torch.full((Q.shape[0], w.Hq, w.dv), nan, dtype=torch.bfloat16, device=dev)
    O_lo = torch.full_like(O, nan)
    LSE = torch.full((w.Hq, Q.shape[0]), nan, dtype=torch.float32, device=dev)
    esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=w.causal, O=O, LSE=LSE, O_lo=O_lo)
    dQ, dK, dV = (torch.full_like(x, nan) for x in (Q, K, V))
    esd.attn_bwd_varlen(Q, K, V, O, G, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=w.causal, dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    return O, LSE, dQ, dK, dV


@pytest.mark.parametrize("name", list(CASES))
def test_varlen_matches_oracle(orc, name):
    w = CASES[name]
    inp = make_varlen_inputs(w)
    O, LSE, dQ, dK, dV = _run(w, inp)
    rO, rL, rdQ, rdK, rdV = varlen_reference(w, inp, orc)
    assert_close(f64(O), rO, "O")
    assert_close(f64(LSE), rL, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(dQ), rdQ, "dQ")
    assert_close(f64(dK), rdK, "dK")
    assert_close(f64(dV), rdV, "dV")


def test_zero_query_sequence_gets_zero_key_gradients():
    w = CASES["zero_query_sequence_d64"]
    inp = make_varlen_inputs(w)
    _O, _L, _dQ, dK, dV = _run(w, inp)
    k0, k1 = inp.cu_k[1], inp.cu_k[2]
    assert torch.count_nonzero(dK[k0:k1]).item() == 0
    assert torch.count_nonzero(dV[k0:k1]).item() == 0


def test_single_sequence_equals_padded_layout():
    """One packed sequence is the [S][H][d] layout: the same numbers as the
    padded entry points on the [1][H][S][d] transpose (O, LSE bit for bit: the same
    kernels visit the same tiles in the same order)."""
    import exact_scaled_dot_gb300 as esd
    w = VarlenWorkload("one", B=1, Hq=4, Hkv=2, dh=128, dv=128, causal=True, lens_q=(700,), seed=67)
    inp = make_varlen_inputs(w)
    O, LSE, dQ, dK, dV = _run(w, inp)
    dev = "cuda:0"
    to_pad = lambda x: x.to(dev).transpose(0, 1).unsqueeze(0).contiguous()  # noqa: E731
    Qp, Kp, Vp, Gp = (to_pad(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    O2, L2, Olo2 = esd.attn_fwd(Qp, Kp, Vp, causal=True)
    dQ2, dK2, dV2 = esd.attn_bwd(Qp, Kp, Vp, O2, Gp, L2, O_lo=Olo2, causal=True)
    torch.cuda.synchronize()
    back = lambda x: x[0].transpose(0, 1)  # noqa: E731
    assert torch.equal(O, back(O2))
    assert torch.equal(LSE, L2[0])
    assert_same_sum(dK, back(dK2), "dK")
    assert_same_sum(dV, back(dV2), "dV")
    assert_close(f64(dQ), f64(back(dQ2)), "dQ (reduce-add order may differ)", atol=1e-3, rtol=1e-3)
