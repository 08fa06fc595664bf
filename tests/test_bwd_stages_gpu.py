"""The three backward stage calls, run one by one on one workspace, give the
same gradients as the composite attn_bwd (up to the order of fp32 sums:
dQ's always varies between runs, dK's and dV's when the backward splits a
KV head's query heads over several CTAs), and a
workspace reused across two problems carries nothing over."""
import pytest
import torch

from exact_scaled_dot_gb300.inputs import Workload, make_inputs

from _attn_cases import assert_close, assert_same_sum, f64

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


def _staged(w, inp, ws, dev="cuda:0"):
    import exact_scaled_dot_gb300 as esd
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    mask = dict(causal=w.causal, causal_offset=w.causal_offset if w.causal else None, kv_len=kv)
    O, LSE, O_lo = esd.attn_fwd(Q, K, V, **mask)
    shape = esd.make_shape(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    dQ, dK, dV = (torch.full_like(x, float("nan")) for x in (Q, K, V))
    esd.attn_bwd_preprocess(Q, O, dO, ws, shape=shape, O_lo=O_lo)
    esd.attn_bwd_main(K, V, LSE, ws, dK, dV, shape=shape, **mask)
    esd.attn_bwd_finalize(ws, dQ, shape=shape)
    ref = esd.attn_bwd(Q, K, V, O, dO, LSE, O_lo=O_lo, **mask)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    return (dQ, dK, dV), ref


@pytest.mark.parametrize("w", [
    Workload("stages_gqa_causal", B=2, Hq=4, Hkv=2, nq=300, nk=300, dh=128, dv=128, causal=True,
             kv_len_range=(200, 300), seed=71),
    Workload("stages_cross_d64v", B=1, Hq=2, Hkv=1, nq=130, nk=400, dh=128, dv=64, seed=72),
])
def test_stages_equal_composite(w):
    import exact_scaled_dot_gb300 as esd
    inp = make_inputs(w)
    ws = torch.empty((esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv),),
                     dtype=torch.uint8, device="cuda:0")
    (dQ, dK, dV), (rQ, rK, rV) = _staged(w, inp, ws)
    assert_same_sum(dK, rK, "dK")
    assert_same_sum(dV, rV, "dV")
    assert_close(f64(dQ), f64(rQ), "dQ", atol=1e-3, rtol=1e-3)


def test_workspace_reused_across_problems():
    """A workspace filled with garbage by one problem serves the next one."""
    import exact_scaled_dot_gb300 as esd
    a = Workload("ws_first", B=2, Hq=4, Hkv=4, nq=256, nk=256, dh=128, dv=128, causal=True, seed=73)
    b = Workload("ws_second", B=1, Hq=4, Hkv=2, nq=200, nk=333, dh=128, dv=128, causal=True, seed=74)
    need = max(esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv) for w in (a, b))
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda:0")   # NaN patterns everywhere
    _staged(a, make_inputs(a), ws)
    (dQ, dK, dV), (rQ, rK, rV) = _staged(b, make_inputs(b), ws)
    assert_same_sum(dK, rK, "dK")
    assert_same_sum(dV, rV, "dV")
    assert_close(f64(dQ), f64(rQ), "dQ", atol=1e-3, rtol=1e-3)
