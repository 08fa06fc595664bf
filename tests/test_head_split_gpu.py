"""The backward's query-head split against the oracle.

When a launch has too few CTAs to fill the GPU (one per batch element, KV
head and 128-key tile) and each KV head has several query heads, the
backward splits a KV head's query heads over several CTAs, each adding its
fp32 share of dK and dV ("Appendix A.10", section A.10.5: the sums over the
group) into workspace sums that a last launch rounds into dK, dV.  Checked:
the split is chosen for small MQA/GQA launches and not for one query head
per KV head; its dQ, dK, dV match the fp64 oracle element by element (the
usual 1e-2 + 2e-2 |ref|), padded and packed, with key padding and ragged
tails; strided gradient outputs receive the rounded sums.
"""
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, Workload, make_inputs, make_varlen_inputs

from _attn_cases import assert_close, compare_full, f64, run_gpu, varlen_reference

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


SPLIT_CASES = [
    Workload("split_mqa_causal", B=1, Hq=8, Hkv=1, nq=700, nk=700, dh=128, dv=128, causal=True, seed=91),
    Workload("split_gqa_padded_dv64", B=2, Hq=8, Hkv=2, nq=300, nk=450, dh=128, dv=64, kv_len_range=(200, 450),
             seed=92),
    Workload("split_mqa_d64", B=1, Hq=4, Hkv=1, nq=257, nk=513, dh=64, dv=64, causal=True, seed=93),
]


def _split_of(w):
    import exact_scaled_dot_gb300 as esd
    return esd.attn_bwd_head_split(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal,
                                   causal_offset=w.causal_offset if w.causal else None)


@pytest.mark.parametrize("w", SPLIT_CASES, ids=lambda w: w.name)
def test_split_matches_oracle(orc, w):
    z = _split_of(w)
    assert z > 1 and (w.Hq // w.Hkv) % z == 0, z
    inp = make_inputs(w)
    compare_full(w, inp, run_gpu(w, inp), orc)


def test_one_query_head_per_kv_head_is_not_split():
    w = Workload("mha_small", B=1, Hq=4, Hkv=4, nq=300, nk=300, dh=128, dv=128, causal=True, seed=94)
    assert _split_of(w) == 1


def test_large_launch_is_not_split():
    # 2 x 8 x 32 = 512 CTAs: more than two per SM
    w = Workload("gqa_large", B=2, Hq=32, Hkv=8, nq=4096, nk=4096, dh=128, dv=128, causal=True, seed=95)
    assert _split_of(w) == 1


def test_split_packed_with_strided_gradients(orc):
    """Packed sequences (one KV head, ragged lengths): the rounded sums land
    in dK, dV views of a fused gradient buffer, and nothing outside them is
    written."""
    import exact_scaled_dot_gb300 as esd
    w = VarlenWorkload("split_packed", B=2, Hq=8, Hkv=1, dh=128, dv=128, causal=True, lens_q=(300, 129), seed=96)
    inp = make_varlen_inputs(w)
    dev = "cuda:0"
    Q, K, V, G = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    O, LSE, O_lo = esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=True)
    T = K.shape[0]
    buf = torch.full((T, 2 * w.dh + 32), 7.0, dtype=torch.bfloat16, device=dev)
    dK = buf[:, :w.dh].view(T, 1, w.dh)
    dV = buf[:, w.dh:2 * w.dh].view(T, 1, w.dv)
    dQ, dK, dV = esd.attn_bwd_varlen(Q, K, V, O, G, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=True, dK=dK, dV=dV)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    assert bool((buf[:, 2 * w.dh:] == 7.0).all())
    _rO, _rL, rdQ, rdK, rdV = varlen_reference(w, inp, orc)
    assert_close(f64(dQ), rdQ, "dQ")
    assert_close(f64(dK), rdK, "dK")
    assert_close(f64(dV), rdV, "dV")
