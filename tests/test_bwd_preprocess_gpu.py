"""Stage 1 of the backward (row a5: D_i = sum_l dO_il O_il, the c_i of
"Appendix A.10", eq. A.10.7) checked on its own, in both layouts.

White-box: the checks read the workspace through the library's private
layout (row terms D, then the per-tile bounds, the group exponents, the
main kernel's work counter, the fp32 dQ accumulator and the fp16 copies of
Q and dO, each block starting on a 256-byte boundary).
Per case:
  * each query tile's exponent follows from its largest magnitude M (15 - E
    for M = m 2^E, m in [0.5, 1), rounded down to a multiple of 4, clamped
    to [-30, 30]; 31 for an all-zero tile) and is kept in its record; each
    (batch, KV head) group's exponent is the smallest over its tiles with a
    non-zero entry (0 if there is none), for Q and for dO separately, and
    the fp16 copies of Q and dO equal torch's conversion of the rows times
    2^e_group, bit for bit (byte work: exact);
  * the dQ accumulator rows are all +0.0 (the workspace starts as 0xFF, NaN)
    and the main kernel's work counter is 0;
  * D equals sum_l dO_il (O_il + O_lo_il) restated in fp64 from the same
    device tensors, within the fp32 summation bound 32 * 2^-24 * sum |terms|;
  * with O_lo, D equals the oracle's D (its own fp64 O) within
    1e-2 + 2e-2 |D| (without it, D is that of the bf16 O by definition);
  * each tile bound equals (max_i ||dO_i||_2, max_i |D_i|) over the tile's
    rows, relative 1e-5, and (0, 0) for a tile with no rows.
Cases span ragged last tiles, d_v = 64 and 128, inputs scaled far outside
the fp16 range (2^-30 and 2^20), and packed sequences including one of
length zero.  Without O_lo the stage refuses to run (ATTN_ERR_NULL).
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


def _views(ws, rows, tiles, groups, dh, dv):
    """D [rows], tile records [tiles, 4] (bounds, e_Q, e_dO), group exponents [groups, 2], the main kernel's
    work counter [1], accumulator [rows * dh], Q16 [rows, dh], dO16 [rows, dv]."""
    off_t = _r256(rows * 4)
    off_g = off_t + _r256(tiles * 16)
    off_c = off_g + _r256(groups * 8)
    off_a = off_c + 256
    off_q = off_a + _r256(rows * dh * 4)
    off_o = off_q + _r256(rows * dh * 2)
    assert off_o + rows * dv * 2 <= ws.numel()
    D = ws[:rows * 4].view(torch.float32)
    tm = ws[off_t:off_t + tiles * 16].view(torch.float32).reshape(tiles, 4)
    grp = ws[off_g:off_g + groups * 8].view(torch.float32).reshape(groups, 2)
    ctr = ws[off_c:off_c + 4].view(torch.int32)
    acc = ws[off_a:off_a + rows * dh * 4].view(torch.float32)
    q16 = ws[off_q:off_q + rows * dh * 2].view(torch.float16).reshape(rows, dh)
    do16 = ws[off_o:off_o + rows * dv * 2].view(torch.float16).reshape(rows, dv)
    return D, tm, grp, ctr, acc, q16, do16


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def _tile_exp(x):
    """The exponent of a tile whose entries are x: 15 - E for max |x| = m 2^E,
    m in [0.5, 1), rounded down to a multiple of 4 and clamped to [-30, 30];
    31 for an all-zero tile."""
    m = float(x.abs().max()) if x.numel() else 0.0
    if m == 0.0:
        return 31
    e = 15 - math.frexp(m)[1]
    return max(-30, min(30, 4 * (e // 4)))


def _check_f16_tile(got16, x, e):
    """got16 is the tile x re-encoded as fp16 x 2^e (e = 31: zeros, unscaled)."""
    sc = 1.0 if e == 31 else 2.0 ** e
    assert _same_bits(got16, (x.double() * sc).to(torch.float16))


def _group_exps(tile_exp, B, Hq, Hkv, tiles_of):
    """The exponent every tile of a (batch, KV head) group ends with: the
    smallest per-tile exponent among the group's tiles (heads r of the group,
    tiles t < tiles_of(b)) that are not all zero, or 0 when all are.
    tile_exp[(b, r, t)] -> exponent; returns the same keys."""
    g = Hq // Hkv
    out = {}
    for b in range(B):
        for hk in range(Hkv):
            keys = [(b, r, t) for r in range(hk * g, (hk + 1) * g) for t in range(tiles_of(b))]
            vals = [tile_exp[k] for k in keys if tile_exp[k] != 31]
            e = min(vals) if vals else 0
            out.update({k: e for k in keys})
    return out


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
@pytest.mark.parametrize("mode", ["unit", "scaled", "mixed"])
def test_preprocess_padded(orc, w, mode):
    """mixed: query tiles of one group with different exponents (head 0's dO
    x 2^-12, rows 128.. of Q x 2^8), so the group pass rescales some tiles."""
    import exact_scaled_dot_gb300 as esd
    dev = "cuda:0"
    inp = make_inputs(w)
    gscale = 1.0
    if mode == "scaled":      # exact: powers of two in bf16
        inp.Q.mul_(2.0 ** 20)
        gscale = 2.0 ** -30
        inp.dO.mul_(gscale)
    elif mode == "mixed":
        inp.dO[:, 0] *= 2.0 ** -12
        inp.Q[:, :, 128:] *= 2.0 ** 8
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    O, LSE, O_lo = esd.attn_fwd(Q, K, V, causal=w.causal, kv_len=kv)
    lo = O_lo
    shape = esd.make_shape(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    need = esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    esd.attn_bwd_preprocess(Q, O, dO, ws, shape=shape, O_lo=lo)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0

    rows, nqt = w.B * w.Hq * w.nq, math.ceil(w.nq / 128)
    D, tm, grp, ctr, acc, q16, do16 = _views(ws, rows, w.B * w.Hq * nqt, w.B * w.Hkv, w.dh, w.dv)
    assert int(ctr.item()) == 0   # the main kernel's work counter (the workspace started as 0xFF)
    tm_c, grp_c = tm.cpu(), grp.cpu()
    Qr, dOr = Q.reshape(w.B, w.Hq, w.nq, w.dh), dO.reshape(w.B, w.Hq, w.nq, w.dv)
    q16r, do16r = q16.reshape(w.B, w.Hq, w.nq, w.dh), do16.reshape(w.B, w.Hq, w.nq, w.dv)
    rng = lambda t: slice(t * 128, min(w.nq, (t + 1) * 128))  # noqa: E731
    keys = [(b, r, t) for b in range(w.B) for r in range(w.Hq) for t in range(nqt)]
    tq = {k: _tile_exp(Qr[k[0], k[1], rng(k[2])]) for k in keys}
    to = {k: _tile_exp(dOr[k[0], k[1], rng(k[2])]) for k in keys}
    eq = _group_exps(tq, w.B, w.Hq, w.Hkv, lambda b: nqt)
    eo = _group_exps(to, w.B, w.Hq, w.Hkv, lambda b: nqt)
    g = w.Hq // w.Hkv
    for (b, r, t) in keys:
        rec = tm_c[(b * w.Hq + r) * nqt + t]
        assert (int(rec[2]), int(rec[3])) == (tq[(b, r, t)], to[(b, r, t)]), (b, r, t)
        gr = grp_c[b * w.Hkv + r // g]
        assert (int(gr[0]), int(gr[1])) == (eq[(b, r, t)], eo[(b, r, t)]), (b, r)
        _check_f16_tile(q16r[b, r, rng(t)], Qr[b, r, rng(t)], eq[(b, r, t)])
        _check_f16_tile(do16r[b, r, rng(t)], dOr[b, r, rng(t)], eo[(b, r, t)])
    assert torch.count_nonzero(acc.view(torch.int32)).item() == 0

    ref, bound = _row_terms(O, lo, dO)
    ref, bound = ref.reshape(rows), bound.reshape(rows)
    err = (D.double() - ref).abs()
    assert bool((err <= bound).all()), f"D vs fp64 restatement: worst excess {float((err - bound).max()):.3e}"

    # D against the oracle's (its own fp64 O), at the unit scale of dO.
    _dq, _dk, _dv, D_orc, _C = orc.backward(problem_of(w, inp),
                                             *(f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO)), want_dkdv=False)
    unit = np.full((w.B, w.Hq, 1), 1.0 / gscale)
    if mode == "mixed":
        unit[:, 0] = 2.0 ** 12
    got = f64(D).reshape(D_orc.shape) * unit
    D_orc = D_orc * unit
    assert np.all(np.abs(got - D_orc) <= ATOL + RTOL * np.abs(D_orc)), \
        f"D vs oracle: max err {np.abs(got - D_orc).max():.3e}"

    dO_r, D_r = dO.reshape(w.B * w.Hq, w.nq, w.dv), D.reshape(w.B * w.Hq, w.nq)
    for bh in range(w.B * w.Hq):
        for t in range(nqt):
            i0, i1 = t * 128, min(w.nq, (t + 1) * 128)
            mn, md = _tile_bounds(dO_r[bh, i0:i1], D_r[bh, i0:i1])
            got_mn, got_md = float(tm_c[bh * nqt + t, 0]), float(tm_c[bh * nqt + t, 1])
            assert abs(got_mn - mn) <= 1e-5 * mn + 1e-30 and abs(got_md - md) <= 1e-5 * md + 1e-30, \
                (bh, t, got_mn, mn, got_md, md)


def test_preprocess_requires_o_lo():
    import exact_scaled_dot_gb300 as esd
    w = PADDED[0]
    dev = "cuda:0"
    inp = make_inputs(w)
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = inp.kv_len.tolist()
    O, LSE, O_lo = esd.attn_fwd(Q, K, V, causal=w.causal, kv_len=kv)
    shape = esd.make_shape(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    ws = torch.empty((esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv),), dtype=torch.uint8,
                     device=dev)
    with pytest.raises(esd.AttnError) as ei:
        esd.attn_bwd_preprocess(Q, O, dO, ws, shape=shape, O_lo=None)
    assert ei.value.code == esd.ATTN_ERR_NULL
    with pytest.raises(esd.AttnError) as ei:
        esd.attn_bwd(Q, K, V, O, dO, LSE, O_lo=None, causal=w.causal, kv_len=kv)
    assert ei.value.code == esd.ATTN_ERR_NULL


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
    D, tm, grp, _ctr, _acc, q16, do16 = _views(ws, rows, w.B * w.Hq * nqt, w.B * w.Hkv, w.dh, w.dv)
    q16, do16 = q16.reshape(Tq, w.Hq, w.dh), do16.reshape(Tq, w.Hq, w.dv)

    ref, bound = _row_terms(O, O_lo, dO)                   # [Tq, Hq]
    Dm = D.reshape(w.Hq, Tq).t()                           # D is head-major: [Hq, Tq]
    err = (Dm.double() - ref).abs()
    assert bool((err <= bound).all()), f"D vs fp64 restatement: worst excess {float((err - bound).max()):.3e}"

    tm_c = tm.cpu()
    tiles_of = lambda b: (lens[b] + 127) // 128  # noqa: E731
    keys = [(b, h, t) for b in range(w.B) for h in range(w.Hq) for t in range(tiles_of(b))]
    sl = lambda b, t: slice(int(inp.cu_q[b]) + t * 128, int(inp.cu_q[b]) + min(lens[b], (t + 1) * 128))  # noqa: E731
    tq = {k: _tile_exp(Q[sl(k[0], k[2]), k[1]]) for k in keys}
    to = {k: _tile_exp(dO[sl(k[0], k[2]), k[1]]) for k in keys}
    geq = _group_exps(tq, w.B, w.Hq, w.Hkv, tiles_of)
    geo = _group_exps(to, w.B, w.Hq, w.Hkv, tiles_of)
    grp_c = grp.cpu()
    for b in range(w.B):
        q0 = int(inp.cu_q[b])
        for h in range(w.Hq):
            for t in range(nqt):
                i0, i1 = t * 128, max(t * 128, min(lens[b], (t + 1) * 128))
                mn, md = _tile_bounds(dO[q0 + i0:q0 + i1, h], Dm[q0 + i0:q0 + i1, h])
                got = tm_c[(b * w.Hq + h) * nqt + t]
                assert abs(float(got[0]) - mn) <= 1e-5 * mn + 1e-30, (b, h, t, float(got[0]), mn)
                assert abs(float(got[1]) - md) <= 1e-5 * md + 1e-30, (b, h, t, float(got[1]), md)
                # tiles past the sequence keep the all-zero mark
                te = (tq[(b, h, t)], to[(b, h, t)]) if t < tiles_of(b) else (31, 31)
                assert (int(got[2]), int(got[3])) == te, (b, h, t)
                if t >= tiles_of(b):
                    continue
                eq, eo = geq[(b, h, t)], geo[(b, h, t)]
                gr = grp_c[b * w.Hkv + h // (w.Hq // w.Hkv)]
                assert (int(gr[0]), int(gr[1])) == (eq, eo), (b, h)
                _check_f16_tile(q16[q0 + i0:q0 + i1, h], Q[q0 + i0:q0 + i1, h], eq)
                _check_f16_tile(do16[q0 + i0:q0 + i1, h], dO[q0 + i0:q0 + i1, h], eo)
