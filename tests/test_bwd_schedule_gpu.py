"""The backward main kernel's two schedules against the oracle.

The main kernel does the same work per (batch, KV head, 128-key tile) item
under two schedules: one CTA per item (the grid kernel), or one CTA per SM
taking items from a counter (the persistent kernel, which hides each item's
fixed cost behind its neighbours' steps).  The host picks the persistent one
when the mean item has at most 40 steps (128-query tiles times query heads).
Checked: the choice for long-item and short-item problems (padded and
packed, with and without a rotary), and each schedule's dQ, dK, dV (and the
forward's O, LSE) against the fp64 oracle element by element at the usual
tolerance (1e-2 + 2e-2 |ref|, LSE 1e-3), with key padding, ragged tails and
d = 64.  The persistent kernel also runs items without steps (key tiles past
kv_len: zero dK, dV rows) between items with steps.
"""
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, Workload, make_inputs, make_varlen_inputs

from _attn_cases import LSE_ATOL, assert_close, compare_full, f64, run_gpu, varlen_reference

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


# (workload, persistent): the first two have items of 48 steps (one of them
# GQA, eight query heads per KV head), the others of at most a few (the last
# one also splits its query heads).
PADDED = [
    (Workload("grid_mha_long_queries", B=1, Hq=16, Hkv=16, nq=6144, nk=256, dh=128, dv=128, seed=111), False),
    (Workload("grid_gqa_cross_dv64", B=3, Hq=16, Hkv=2, nq=768, nk=2304, dh=128, dv=64, seed=112), False),
    (Workload("pers_mha_causal_padded", B=2, Hq=4, Hkv=4, nq=640, nk=2048, dh=128, dv=128, causal=True,
              kv_len_range=(1000, 2048), seed=113), True),
    (Workload("pers_cross_short_queries_d64", B=3, Hq=4, Hkv=2, nq=200, nk=1500, dh=64, dv=64,
              kv_len_range=(700, 1500), seed=114), True),
]


def _persistent(w, rotary=None):
    import exact_scaled_dot_gb300 as esd
    return esd.attn_bwd_persistent(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal,
                                   causal_offset=w.causal_offset if w.causal else None,
                                   kv_len=None if w.kv_len_range is None else [w.nk] * w.B, rotary=rotary)


@pytest.mark.parametrize("w,persistent", PADDED, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_schedule_matches_oracle(orc, w, persistent):
    assert _persistent(w) == persistent
    inp = make_inputs(w)
    if w.kv_len_range is not None:
        # the choice with the drawn key lengths (items past kv_len have no steps)
        import exact_scaled_dot_gb300 as esd
        assert esd.attn_bwd_persistent(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal,
                                       causal_offset=w.causal_offset if w.causal else None,
                                       kv_len=inp.kv_len.tolist()) == persistent
    compare_full(w, inp, run_gpu(w, inp), orc)


def test_rotary_keeps_the_choice():
    """A rotary only rules out the query-head split; long items still take
    the grid kernel."""
    import exact_scaled_dot_gb300 as esd
    w = PADDED[0][0]
    pos = torch.zeros((w.B, w.nq), dtype=torch.int32)
    rot = esd.Rotary(pos, torch.zeros((w.B, w.nk), dtype=torch.int32))
    assert _persistent(w, rotary=rot) is False
    assert _persistent(PADDED[2][0], rotary=rot) is True


PACKED = [
    # one key tile per sequence seen by 47-50 query tiles: grid
    (VarlenWorkload("grid_packed_long_queries", B=2, Hq=4, Hkv=4, dh=128, dv=128, lens_q=(6400, 6000),
                    lens_k=(256, 200), seed=115), False),
    # causal self-attention, a few steps per item: persistent
    (VarlenWorkload("pers_packed_causal", B=3, Hq=4, Hkv=4, dh=128, dv=128, causal=True, lens_q=(700, 1, 450),
                    seed=116), True),
]


@pytest.mark.parametrize("w,persistent", PACKED, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_packed_schedule_matches_oracle(orc, w, persistent):
    import exact_scaled_dot_gb300 as esd
    inp = make_varlen_inputs(w)
    if not w.causal:
        # Without a mask the plan of the padded problem with the longest
        # query sequence and these key lengths makes the same choice.
        assert esd.attn_bwd_persistent(w.B, w.Hq, w.Hkv, max(inp.lens_q), max(inp.lens_k), w.dh, w.dv,
                                       kv_len=list(inp.lens_k)) == persistent
    dev = "cuda:0"
    Q, K, V, G = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    O, LSE, O_lo = esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=w.causal)
    dQ, dK, dV = (torch.full_like(x, float("nan")) for x in (Q, K, V))   # every row must be written
    esd.attn_bwd_varlen(Q, K, V, O, G, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=w.causal, dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    rO, rL, rdQ, rdK, rdV = varlen_reference(w, inp, orc)
    assert_close(f64(O), rO, "O")
    assert_close(f64(LSE), rL, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(dQ), rdQ, "dQ")
    assert_close(f64(dK), rdK, "dK")
    assert_close(f64(dV), rdV, "dV")
