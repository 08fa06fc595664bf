"""GPU-vs-oracle parity with strided views for every user tensor.

Attention usually sits between projections, so Q, K and V arrive as slices
of one fused projection output and the gradients leave into one fused
gradient buffer.  The entry points take such views through attn_strides (the
element strides of each tensor's token/row and head index; the innermost
index stays contiguous) and must give the same numbers as on contiguous
copies, without copying:

- packed (token-major) Q, K, V sliced from a fused [T, (Hq + 2 Hkv) d]
  buffer, dQ, dK, dV written into a fused gradient buffer of the same shape,
  O (and O_lo) into a row-padded [T, Hq d + 64] buffer;
- padded (head-major) views with padded rows and padded heads, d_v = 64
  sliced out of a 128-wide buffer, and one batch element of a
  sequence-major [1, n, H, d] tensor.

Each case is compared element by element with the fp64 oracle (the usual
1e-2 + 2e-2 |ref|, LSE 1e-3) and with the same call on contiguous copies:
O, O_lo and LSE bit for bit (the kernels visit the same tiles in the same
order), dQ, dK and dV at 1e-3 (fp32 sums whose order may differ: dQ always,
dK and dV when the backward splits a KV head's query heads).  Outputs
start as NaN, and the padding around every output view holds a sentinel that
must survive: a kernel writing outside its view fails the test.
"""
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, Workload, make_inputs, make_varlen_inputs

from _attn_cases import LSE_ATOL, assert_close, assert_same_sum, f64, problem_of, varlen_reference

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


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


def _status_ok():
    import exact_scaled_dot_gb300 as esd
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0


def _exact(got, want, what):
    assert torch.equal(got, want), f"{what}: strided and contiguous calls differ"


# ---------------------------------------------------------------------------
# packed: fused QKV projection output
# ---------------------------------------------------------------------------
PACKED = {
    "gqa_causal_mixed": VarlenWorkload("strided_gqa_causal_mixed", B=3, Hq=8, Hkv=2, dh=128, dv=128, causal=True,
                                       lens_q=(1, 300, 129), seed=71),
    "mqa_cross": VarlenWorkload("strided_mqa_cross", B=2, Hq=4, Hkv=1, dh=128, dv=128,
                                lens_q=(200, 64), lens_k=(500, 9), seed=72),
    "d64": VarlenWorkload("strided_d64", B=2, Hq=4, Hkv=2, dh=64, dv=64, causal=True, lens_q=(130, 77), seed=73),
}


def _fused(parts, pad=0, fill=SENTINEL):
    """One [T, sum(H d) + pad] buffer holding the [T, H, d] parts side by
    side, and the views of each part inside it."""
    T = parts[0].shape[0]
    widths = [p.shape[1] * p.shape[2] for p in parts]
    buf = torch.full((T, sum(widths) + pad), fill, dtype=torch.bfloat16, device=parts[0].device)
    views, c = [], 0
    for p, wd in zip(parts, widths):
        v = buf[:, c:c + wd].view(T, p.shape[1], p.shape[2])
        v.copy_(p)
        views.append(v)
        c += wd
    return buf, views


def _nan_views(shapes, pad=0):
    """A fused buffer of sentinels whose part views are set to NaN."""
    dev = "cuda:0"
    parts = [torch.empty(s, dtype=torch.bfloat16, device=dev) for s in shapes]
    buf, views = _fused(parts, pad=pad)
    for v in views:
        v.fill_(float("nan"))
    return buf, views


def _outside(buf, views):
    """Entries of buf outside every view."""
    mask = torch.ones(buf.shape, dtype=torch.bool, device=buf.device)
    c = 0
    for v in views:
        wd = v.shape[1] * v.shape[2]
        mask[:, c:c + wd] = False
        c += wd
    return buf[mask]


@pytest.mark.parametrize("name", list(PACKED))
def test_fused_qkv_packed_views(orc, name):
    import exact_scaled_dot_gb300 as esd
    w = PACKED[name]
    inp = make_varlen_inputs(w)
    dev = "cuda:0"
    Qc, Kc, Vc, Gc = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    Tq, Tk = Qc.shape[0], Kc.shape[0]
    assert Tq == Tk or not w.causal
    # Q from a fused Q|K|V buffer when T_q == T_k (self-attention); otherwise
    # Q from a fused Q|pad buffer and K, V from a fused K|V buffer.
    if Tq == Tk:
        _qkv, (Q, K, V) = _fused([Qc, Kc, Vc])
    else:
        _qb, (Q,) = _fused([Qc], pad=64)
        _kvb, (K, V) = _fused([Kc, Vc])
    assert not Q.is_contiguous() and not K.is_contiguous() and not V.is_contiguous()
    obuf, (O,) = _nan_views([(Tq, w.Hq, w.dv)], pad=64)
    olbuf, (O_lo,) = _nan_views([(Tq, w.Hq, w.dv)], pad=64)
    LSE = torch.full((w.Hq, Tq), float("nan"), dtype=torch.float32, device=dev)
    esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=w.causal, O=O, LSE=LSE, O_lo=O_lo)
    _gb, (G,) = _fused([Gc], pad=32)
    if Tq == Tk:
        gbuf, (dQ, dK, dV) = _nan_views([Qc.shape, Kc.shape, Vc.shape])
        outs = [(gbuf, [dQ, dK, dV])]
    else:
        qgbuf, (dQ,) = _nan_views([Qc.shape], pad=64)
        kvgbuf, (dK, dV) = _nan_views([Kc.shape, Vc.shape])
        outs = [(qgbuf, [dQ]), (kvgbuf, [dK, dV])]
    esd.attn_bwd_varlen(Q, K, V, O, G, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=w.causal, dQ=dQ, dK=dK, dV=dV)
    _status_ok()
    # the padding around every output view is untouched
    for buf, views in [(obuf, [O]), (olbuf, [O_lo])] + outs:
        rest = _outside(buf, views)
        assert bool((rest == SENTINEL).all()), "a kernel wrote outside its output view"
    # against the oracle
    rO, rL, rdQ, rdK, rdV = varlen_reference(w, inp, orc)
    assert_close(f64(O), rO, "O")
    assert_close(f64(LSE), rL, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(dQ), rdQ, "dQ")
    assert_close(f64(dK), rdK, "dK")
    assert_close(f64(dV), rdV, "dV")
    # against the same call on contiguous copies
    O2, L2, Olo2 = esd.attn_fwd_varlen(Qc, Kc, Vc, inp.cu_q, inp.cu_k, causal=w.causal)
    dQ2, dK2, dV2 = esd.attn_bwd_varlen(Qc, Kc, Vc, O2, Gc, L2, inp.cu_q, inp.cu_k, O_lo=Olo2, causal=w.causal)
    _status_ok()
    _exact(O, O2, "O")
    _exact(O_lo, Olo2, "O_lo")
    _exact(LSE, L2, "LSE")
    assert_same_sum(dK, dK2, "dK")
    assert_same_sum(dV, dV2, "dV")
    assert_close(f64(dQ), f64(dQ2), "dQ vs contiguous", atol=1e-3, rtol=1e-3)


# ---------------------------------------------------------------------------
# padded: head-major views
# ---------------------------------------------------------------------------
GQA = Workload("strided_padded_gqa", B=2, Hq=4, Hkv=2, nq=300, nk=300, dh=128, dv=128, causal=True,
               kv_len_range=(150, 300), seed=74)
CROSS64 = Workload("strided_padded_cross_dv64", B=2, Hq=2, Hkv=1, nq=200, nk=333, dh=128, dv=64,
                   kv_len_range=(100, 333), seed=75)


def _padded_view(x, row_pad, d_full, fill):
    """x [B, H, n, d] copied into a [B, H, n + row_pad, d_full] buffer: a view
    with padded rows (row stride d_full) and padded heads."""
    B, H, n, d = x.shape
    buf = torch.full((B, H, n + row_pad, d_full), fill, dtype=x.dtype, device=x.device)
    v = buf[:, :, :n, :d]
    v.copy_(x)
    return buf, v


def _check_pad(buf, v, what):
    mask = torch.ones(buf.shape, dtype=torch.bool, device=buf.device)
    mask[:, :, :v.shape[2], :v.shape[3]] = False
    assert bool((buf[mask] == SENTINEL).all()), f"{what}: a kernel wrote outside its view"


def _run_padded(w, Q, K, V, dO, O, O_lo, dQ, dK, dV, kv):
    import exact_scaled_dot_gb300 as esd
    off = w.causal_offset if w.causal else None
    LSE = torch.full((w.B, w.Hq, w.nq), float("nan"), dtype=torch.float32, device=Q.device)
    esd.attn_fwd(Q, K, V, causal=w.causal, causal_offset=off, kv_len=kv, O=O, LSE=LSE, O_lo=O_lo)
    esd.attn_bwd(Q, K, V, O, dO, LSE, O_lo=O_lo, causal=w.causal, causal_offset=off, kv_len=kv, dQ=dQ, dK=dK,
                 dV=dV)
    _status_ok()
    return LSE


@pytest.mark.parametrize("w", [GQA, CROSS64], ids=lambda w: w.name)
def test_padded_strided_views(orc, w):
    import exact_scaled_dot_gb300 as esd
    inp = make_inputs(w)
    dev = "cuda:0"
    Qc, Kc, Vc, Gc = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    nan = float("nan")
    _bq, Q = _padded_view(Qc, 8, 192, SENTINEL)
    _bk, K = _padded_view(Kc, 24, 256, SENTINEL)
    _bv, V = _padded_view(Vc, 0, 128 if w.dv == 64 else 160, SENTINEL)
    _bg, G = _padded_view(Gc, 16, w.dv + 64, SENTINEL)
    bo, O = _padded_view(torch.full((w.B, w.Hq, w.nq, w.dv), nan, dtype=torch.bfloat16, device=dev), 8,
                         w.dv + 64, SENTINEL)
    bol = torch.full_like(bo, SENTINEL)
    O_lo = bol[:, :, :w.nq, :w.dv]
    O_lo.fill_(nan)
    bdq, dQ = _padded_view(torch.full_like(Qc, nan), 8, 136, SENTINEL)
    bdk, dK = _padded_view(torch.full_like(Kc, nan), 0, 144, SENTINEL)
    bdv, dV = _padded_view(torch.full_like(Vc, nan), 40, 128 if w.dv == 64 else 136, SENTINEL)
    for t in (Q, K, V, G, O, O_lo, dQ, dK, dV):
        assert not t.is_contiguous()
    LSE = _run_padded(w, Q, K, V, G, O, O_lo, dQ, dK, dV, kv)
    for buf, v, what in ((bo, O, "O"), (bol, O_lo, "O_lo"), (bdq, dQ, "dQ"), (bdk, dK, "dK"), (bdv, dV, "dV")):
        _check_pad(buf, v, what)
    p = problem_of(w, inp)
    Qd, Kd, Vd, Gd = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    rO, rL = orc.forward(p, Qd, Kd, Vd)
    rdQ, rdK, rdV, _D, _C = orc.backward(p, Qd, Kd, Vd, Gd)
    assert_close(f64(O), rO, "O")
    assert_close(f64(LSE), rL, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(dQ), rdQ, "dQ")
    assert_close(f64(dK), rdK, "dK")
    assert_close(f64(dV), rdV, "dV")
    off = w.causal_offset if w.causal else None
    O2, L2, Olo2 = esd.attn_fwd(Qc, Kc, Vc, causal=w.causal, causal_offset=off, kv_len=kv)
    dQ2, dK2, dV2 = esd.attn_bwd(Qc, Kc, Vc, O2, Gc, L2, O_lo=Olo2, causal=w.causal, causal_offset=off, kv_len=kv)
    _status_ok()
    _exact(O, O2, "O")
    _exact(O_lo, Olo2, "O_lo")
    _exact(LSE, L2, "LSE")
    assert_same_sum(dK, dK2, "dK")
    assert_same_sum(dV, dV2, "dV")
    assert_close(f64(dQ), f64(dQ2), "dQ vs contiguous", atol=1e-3, rtol=1e-3)


def test_sequence_major_batch_element(orc):
    """One batch element of a sequence-major [1, n, H, d] tensor, seen as
    [1, H, n, d]: the head stride (d) is smaller than the row stride (H d)."""
    import exact_scaled_dot_gb300 as esd
    w = Workload("strided_seq_major", B=1, Hq=4, Hkv=2, nq=257, nk=257, dh=128, dv=128, causal=True, seed=76)
    inp = make_inputs(w)
    dev = "cuda:0"
    seq = lambda x: x.to(dev).transpose(1, 2).contiguous().transpose(1, 2)  # noqa: E731
    Q, K, V, G = (seq(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    assert Q.stride(1) == 128 and Q.stride(2) == 4 * 128
    nan = float("nan")
    O = seq(torch.full((1, 4, 257, 128), nan, dtype=torch.bfloat16))
    O_lo = torch.empty_strided(O.shape, O.stride(), dtype=O.dtype, device=dev).fill_(nan)
    dQ, dK, dV = (seq(torch.full(x.shape, nan, dtype=torch.bfloat16)) for x in (inp.Q, inp.K, inp.V))
    LSE = _run_padded(w, Q, K, V, G, O, O_lo, dQ, dK, dV, None)
    p = problem_of(w, inp)
    Qd, Kd, Vd, Gd = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    rO, rL = orc.forward(p, Qd, Kd, Vd)
    rdQ, rdK, rdV, _D, _C = orc.backward(p, Qd, Kd, Vd, Gd)
    assert_close(f64(O), rO, "O")
    assert_close(f64(LSE), rL, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(dQ), rdQ, "dQ")
    assert_close(f64(dK), rdK, "dK")
    assert_close(f64(dV), rdV, "dV")
    # the stage entry points take the same views
    shape = esd.make_shape(1, 4, 2, 257, 257, 128, 128)
    ws = torch.empty((esd.attn_bwd_workspace_bytes(1, 4, 2, 257, 257, 128, 128),), dtype=torch.uint8, device=dev)
    dQ3, dK3, dV3 = (torch.full_like(x, nan) for x in (dQ, dK, dV))
    esd.attn_bwd_preprocess(Q, O, G, ws, shape=shape, O_lo=O_lo)
    esd.attn_bwd_main(K, V, LSE, ws, dK3, dV3, shape=shape, causal=True)
    esd.attn_bwd_finalize(ws, dQ3, shape=shape)
    _status_ok()
    assert_same_sum(dK3, dK, "staged dK")
    assert_same_sum(dV3, dV, "staged dV")
    assert_close(f64(dQ3), f64(dQ), "staged dQ", atol=1e-3, rtol=1e-3)


def test_o_lo_must_share_o_strides():
    import exact_scaled_dot_gb300 as esd
    w = GQA
    inp = make_inputs(w)
    dev = "cuda:0"
    Q, K, V = (x.to(dev) for x in (inp.Q, inp.K, inp.V))
    _b, O = _padded_view(torch.zeros((w.B, w.Hq, w.nq, w.dv), dtype=torch.bfloat16, device=dev), 0, 192, 0.0)
    O_lo = torch.empty((w.B, w.Hq, w.nq, w.dv), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        esd.attn_fwd(Q, K, V, causal=True, O=O, O_lo=O_lo)
