"""Stage 1 of the backward (row a5: D_i = sum_l dO_il O_il, the c_i of
"Appendix A.10", eq. A.10.7) checked on its own, in both layouts.

White-box: the checks read the workspace through the library's private
layout (row terms D, then the per-tile bounds, the fp32 dQ accumulator and
the fp16 copies of Q and dO, each block starting on a 256-byte boundary).
Per case:
  * the fp16 copies of Q and dO equal torch's bf16 -> fp16 conversion bit
    for bit (byte work: exact);
  * the dQ accumulator rows are all +0.0 (the workspace starts as 0xFF, NaN);
  * D equals sum_l dO_il (O_il + O_lo_il) restated in fp64 from the same
    device tensors, within the fp32 summation bound 32 * 2^-24 * sum |terms|;
  * with O_lo, D equals the oracle's D (its own fp64 O) within
    1e-2 + 2e-2 |D| (without it, D is that of the bf16 O by definition);
  * each tile bound equals (max_i ||dO_i||_2, max_i |D_i|) over the tile's
    rows, relative 1e-5, and (0, 0) for a tile with no rows.
Cases span ragged last tiles, d_v = 64 and 128, with and without O_lo, and
packed sequences including one of length zero.
"""
import math

import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, Workload, make_inputs, make_varlen_inputs

from _attn_cases import ATOL, RTOL, f64, problem_of

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


def _r256(x):
    return (x + 255) // 256 * 256


def _views(ws, rows, tiles, dh, dv):
    """D [rows], tile bounds [tiles, 2], accumulator [rows * dh], Q16 [rows, dh], dO16 [rows, dv]."""
    off_t = _r256(rows * 4)
    off_a = off_t + _r256(tiles * 8)
    off_q = off_a + _r256(rows * dh * 4)
    off_o = off_q + _r256(rows * dh * 2)
    assert off_o + rows * dv * 2 <= ws.numel()
    D = ws[:rows * 4].view(torch.float32)
    tm = ws[off_t:off_t + tiles * 8].view(torch.float32).reshape(tiles, 2)
    acc = ws[off_a:off_a + rows * dh * 4].view(torch.float32)
    q16 = ws[off_q:off_q + rows * dh * 2].view(torch.float16).reshape(rows, dh)
    do16 = ws[off_o:off_o + rows * dv * 2].view(torch.float16).reshape(rows, dv)
    return D, tm, acc, q16, do16


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def _row_terms(O, O_lo, dO):
    """fp64 D and its fp32 summation bound from the device tensors (last axis = d_v)."""
    Of = O.double() + (O_lo.double() if O_lo is not None else 0.0)
    prod = dO.double() * Of
    return prod.sum(-1), 32.0 * 2.0 ** -24 * prod.abs().sum(-1) + 1e-30


def _tile_bounds(dO_rows, D_rows):
    """(max ||dO_i||, max |D_i|) over one tile's rows (fp64), (0, 0) when empty."""
    if D_rows.numel() == 0:
        return 0.0, 0.0
    return float(dO_rows.double().norm(dim=-1).max()), float(D_rows.double().abs().max())


PADDED = [
    Workload("pre_gqa_causal_tail", B=2, Hq=4, Hkv=2, nq=300, nk=300, dh=128, dv=128, causal=True,
             kv_len_range=(200, 300), seed=81),
    Workload("pre_cross_dv64_tail2", B=1, Hq=2, Hkv=1, nq=130, nk=400, dh=128, dv=64, seed=82),
    Workload("pre_d64_one_row_tail", B=1, Hq=3, Hkv=1, nq=257, nk=257, dh=64, dv=64, causal=True, seed=83),
]


@pytest.mark.parametrize("w", PADDED, ids=lambda w: w.name)
@pytest.mark.parametrize("with_lo", [True, False], ids=["O_lo", "no_O_lo"])
def test_preprocess_padded(orc, w, with_lo):
    import exact_scaled_dot_gb300 as esd
    dev = "cuda:0"
    inp = make_inputs(w)
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    O, LSE, O_lo = esd.attn_fwd(Q, K, V, causal=w.causal, kv_len=kv)
    lo = O_lo if with_lo else None
    shape = esd.make_shape(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    need = esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    esd.attn_bwd_preprocess(Q, O, dO, ws, shape=shape, O_lo=lo)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0

    rows, nqt = w.B * w.Hq * w.nq, math.ceil(w.nq / 128)
    D, tm, acc, q16, do16 = _views(ws, rows, w.B * w.Hq * nqt, w.dh, w.dv)
    assert _same_bits(q16, Q.reshape(rows, w.dh).to(torch.float16))
    assert _same_bits(do16, dO.reshape(rows, w.dv).to(torch.float16))
    assert torch.count_nonzero(acc.view(torch.int32)).item() == 0

    ref, bound = _row_terms(O, lo, dO)
    ref, bound = ref.reshape(rows), bound.reshape(rows)
    err = (D.double() - ref).abs()
    assert bool((err <= bound).all()), f"D vs fp64 restatement: worst excess {float((err - bound).max()):.3e}"

    if with_lo:
        # Without O_lo, D is by definition that of the bf16 O (each element
        # rounded by up to 2^-9 relative), which the restatement above covers;
        # the oracle's D is that of the unrounded O.
        _dq, _dk, _dv, D_orc, _C = orc.backward(problem_of(w, inp),
                                                 *(f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO)), want_dkdv=False)
        got = f64(D).reshape(D_orc.shape)
        assert np.all(np.abs(got - D_orc) <= ATOL + RTOL * np.abs(D_orc)), \
            f"D vs oracle: max err {np.abs(got - D_orc).max():.3e}"

    dO_r, D_r, tm_c = dO.reshape(w.B * w.Hq, w.nq, w.dv), D.reshape(w.B * w.Hq, w.nq), tm.cpu()
    for bh in range(w.B * w.Hq):
        for t in range(nqt):
            i0, i1 = t * 128, min(w.nq, (t + 1) * 128)
            mn, md = _tile_bounds(dO_r[bh, i0:i1], D_r[bh, i0:i1])
            got_mn, got_md = float(tm_c[bh * nqt + t, 0]), float(tm_c[bh * nqt + t, 1])
            assert abs(got_mn - mn) <= 1e-5 * mn + 1e-30 and abs(got_md - md) <= 1e-5 * md + 1e-30, \
                (bh, t, got_mn, mn, got_md, md)


PACKED = [
    VarlenWorkload("pre_packed_mixed", B=4, Hq=4, Hkv=2, dh=128, dv=128, causal=True,
                   lens_q=(1, 127, 300, 129), seed=84),
    VarlenWorkload("pre_packed_zero_len_d64", B=3, Hq=4, Hkv=2, dh=64, dv=64, causal=True,
                   lens_q=(130, 0, 77), lens_k=(130, 40, 77), seed=85),
    VarlenWorkload("pre_packed_dv64", B=2, Hq=2, Hkv=1, dh=128, dv=64, lens_q=(257, 64), lens_k=(400, 100),
                   seed=86),
]


@pytest.mark.parametrize("w", PACKED, ids=lambda w: w.name)
def test_preprocess_packed(w):
    """The packed layout through attn_bwd_varlen: its stage 1 leaves D, the
    bounds and the fp16 copies in the workspace (the main kernel only reads
    them), so they are checked after the whole backward."""
    import exact_scaled_dot_gb300 as esd
    dev = "cuda:0"
    inp = make_varlen_inputs(w)
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    O, LSE, O_lo = esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=w.causal)
    need = esd.attn_bwd_varlen_workspace_bytes(w.Hq, w.Hkv, w.dh, w.dv, inp.cu_q, inp.cu_k, causal=w.causal)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    esd.attn_bwd_varlen(Q, K, V, O, dO, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=w.causal, workspace=ws)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0

    Tq = Q.shape[0]
    lens = [int(inp.cu_q[b + 1]) - int(inp.cu_q[b]) for b in range(w.B)]
    nqt = math.ceil(max(max(lens), 1) / 128)
    rows = Tq * w.Hq
    D, tm, _acc, q16, do16 = _views(ws, rows, w.B * w.Hq * nqt, w.dh, w.dv)
    assert _same_bits(q16, Q.reshape(rows, w.dh).to(torch.float16))
    assert _same_bits(do16, dO.reshape(rows, w.dv).to(torch.float16))

    ref, bound = _row_terms(O, O_lo, dO)                   # [Tq, Hq]
    Dm = D.reshape(w.Hq, Tq).t()                           # D is head-major: [Hq, Tq]
    err = (Dm.double() - ref).abs()
    assert bool((err <= bound).all()), f"D vs fp64 restatement: worst excess {float((err - bound).max()):.3e}"

    tm_c = tm.cpu()
    for b in range(w.B):
        q0 = int(inp.cu_q[b])
        for h in range(w.Hq):
            for t in range(nqt):
                i0, i1 = t * 128, max(t * 128, min(lens[b], (t + 1) * 128))
                mn, md = _tile_bounds(dO[q0 + i0:q0 + i1, h], Dm[q0 + i0:q0 + i1, h])
                got = tm_c[(b * w.Hq + h) * nqt + t]
                assert abs(float(got[0]) - mn) <= 1e-5 * mn + 1e-30, (b, h, t, float(got[0]), mn)
                assert abs(float(got[1]) - md) <= 1e-5 * md + 1e-30, (b, h, t, float(got[1]), md)
