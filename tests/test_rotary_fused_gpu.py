"""GPU-vs-oracle parity of attention with the rotary embedding fused into
the entry points (attn_rotary).

"Chapter 15 -- matrix formulas", section 15.6: the scores are those of the
rotated rows q~_i = R_i q_i, k~_j = R_j k_j; "Chapter 31 -- attention
backprop", section 5: the gradients of q and k are those of q~ and k~ turned
back by the opposite angles.  The reference: oracle/rope.py rotates Q and K
with exact angles in fp64 and rounds the rotated rows to bf16 (the entry
points define the rotated rows as bf16 tensors, those of attn_rope; without
this rounding the scores would move by about 2^-9 |q||k| scale, which shifts
LSE by a few 1e-3), the attention oracle runs forward and backward on them
in fp64, and oracle/rope.py turns dQ~ and dK~ back (inverse=True).  O, LSE,
dQ, dK and dV are compared element by element at the usual tolerance
(1e-2 + 2e-2 |ref|, LSE 1e-3).

Also checked: the fused forward equals, bit for bit, attn_rope on Q and K
followed by the forward without a rotary; the staged backward with a rotary
equals the composite call; the backward's gradients agree with the separate
composition (rotate, attention backward, rotate dQ~ and dK~ back) to the
one extra bf16 rounding that composition makes.  Positions: per-row
offsets plus large values (up to 2^20), and packed sequences that restart at
0 or continue a history.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, Workload, make_inputs, make_varlen_inputs

from _attn_cases import LSE_ATOL, assert_close, assert_same_sum, f64, problem_of

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


PADDED = {
    "gqa_causal": Workload("rot_gqa_causal", B=2, Hq=4, Hkv=2, nq=300, nk=300, dh=128, dv=128, causal=True,
                           kv_len_range=(150, 300), seed=81),
    "cross_dv64": Workload("rot_cross_dv64", B=2, Hq=2, Hkv=1, nq=200, nk=333, dh=128, dv=64,
                           kv_len_range=(100, 333), seed=82),
    "mha_d64": Workload("rot_mha_d64", B=1, Hq=3, Hkv=3, nq=257, nk=257, dh=64, dv=64, causal=True, seed=83),
}
BASES = {"gqa_causal": 10000.0, "cross_dv64": 500000.0, "mha_d64": 10000.0}


def _positions(B, n, seed, big=False):
    """[B, n] int32: a per-batch start plus the row index, or (big) large
    scattered positions up to 2^20."""
    g = torch.Generator().manual_seed(seed)
    if big:
        return torch.randint(0, 1 << 20, (B, n), generator=g, dtype=torch.int32)
    start = torch.randint(0, 5000, (B, 1), generator=g, dtype=torch.int32)
    return start + torch.arange(n, dtype=torch.int32)[None, :]


def _rope64(X, pos, base, inverse=False):
    """fp64 rotation of a padded [B, H, n, d] array by positions [B, n]."""
    from oracle.rope import rope
    out = np.empty_like(X)
    for b in range(X.shape[0]):
        out[b] = rope(X[b].transpose(1, 0, 2), pos[b], base=base, inverse=inverse).transpose(1, 0, 2)
    return out


def _bf16(x):
    """fp64 values rounded to bf16 (to nearest even) and back."""
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def _oracle_rotary(orc, w, inp, pq, pk, base):
    p = problem_of(w, inp)
    Q, K, V, G = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    Qr, Kr = _bf16(_rope64(Q, pq, base)), _bf16(_rope64(K, pk, base))
    O, LSE = orc.forward(p, Qr, Kr, V)
    dQr, dKr, dV, _D, _C = orc.backward(p, Qr, Kr, V, G)
    return dict(O=O, LSE=LSE, dQ=_rope64(dQr, pq, base, inverse=True), dK=_rope64(dKr, pk, base, inverse=True),
                dV=dV)


def _run_fused(w, inp, rot, dev="cuda:0"):
    import exact_scaled_dot_gb300 as esd
    Q, K, V, G = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    off = w.causal_offset if w.causal else None
    nan = float("nan")
    O = torch.full((w.B, w.Hq, w.nq, w.dv), nan, dtype=torch.bfloat16, device=dev)
    O_lo = torch.full_like(O, nan)
    LSE = torch.full((w.B, w.Hq, w.nq), nan, dtype=torch.float32, device=dev)
    esd.attn_fwd(Q, K, V, causal=w.causal, causal_offset=off, kv_len=kv, O=O, LSE=LSE, O_lo=O_lo, rotary=rot)
    dQ, dK, dV = (torch.full_like(x, nan) for x in (Q, K, V))
    esd.attn_bwd(Q, K, V, O, G, LSE, O_lo=O_lo, causal=w.causal, causal_offset=off, kv_len=kv, dQ=dQ, dK=dK, dV=dV,
                 rotary=rot)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    return dict(O=O, O_lo=O_lo, LSE=LSE, dQ=dQ, dK=dK, dV=dV)


def _rope_padded_gpu(X, pos, base, inverse=False):
    """attn_rope on a padded [B, H, n, d] tensor: its rows as tokens of one
    head, each with its batch element's position."""
    import exact_scaled_dot_gb300 as esd
    B, H, n, d = X.shape
    rows = pos.to(X.device)[:, None, :].expand(B, H, n).reshape(-1).contiguous()
    return esd.attn_rope(X.reshape(B * H * n, 1, d), rows, base=base, inverse=inverse).reshape(B, H, n, d)


@pytest.mark.parametrize("big", [False, True], ids=["offsets", "large"])
@pytest.mark.parametrize("name", list(PADDED))
def test_fused_rotary_matches_oracle(orc, name, big):
    import exact_scaled_dot_gb300 as esd
    w = PADDED[name]
    base = BASES[name]
    inp = make_inputs(w)
    pq = _positions(w.B, w.nq, w.seed, big)
    pk = _positions(w.B, w.nk, w.seed + 1, big) if w.nq != w.nk else pq.clone()
    rot = esd.Rotary(pq.cuda(), pk.cuda(), base=base)
    res = _run_fused(w, inp, rot)
    ref = _oracle_rotary(orc, w, inp, pq.numpy(), pk.numpy(), base)
    for k in ("O", "dQ", "dK", "dV"):
        assert_close(f64(res[k]), ref[k], k)
    assert_close(f64(res["LSE"]), ref["LSE"], "LSE", atol=LSE_ATOL, rtol=0.0)


@pytest.mark.parametrize("name", list(PADDED))
def test_fused_forward_equals_separate_rotation(name):
    """attn_fwd with a rotary == attn_rope on Q and K, then attn_fwd, bit for
    bit (the same angles, products and bf16 rounding of the rotated rows)."""
    import exact_scaled_dot_gb300 as esd
    w = PADDED[name]
    base = BASES[name]
    inp = make_inputs(w)
    pq = _positions(w.B, w.nq, w.seed + 7, big=True)
    pk = _positions(w.B, w.nk, w.seed + 8, big=True)
    rot = esd.Rotary(pq.cuda(), pk.cuda(), base=base)
    Q, K, V = (x.cuda() for x in (inp.Q, inp.K, inp.V))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    O1, L1, Olo1 = esd.attn_fwd(Q, K, V, causal=w.causal, kv_len=kv, rotary=rot)
    Qr, Kr = _rope_padded_gpu(Q, pq, base), _rope_padded_gpu(K, pk, base)
    O2, L2, Olo2 = esd.attn_fwd(Qr, Kr, V, causal=w.causal, kv_len=kv)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    assert torch.equal(O1, O2) and torch.equal(L1, L2) and torch.equal(Olo1, Olo2)


def test_fused_backward_agrees_with_separate_composition():
    """The separate composition rounds dQ~, dK~ to bf16 before turning them
    back; the fused backward turns them in fp32 and rounds once.  dV is the
    same product of the same operands (up to the order of its fp32 sums);
    dQ, dK agree within the
    usual tolerance (the composition's extra rounding is 2^-9 of dQ~'s
    components, which can exceed the small element two components cancel to,
    so the bound is the absolute 1e-2, not one relative to dQ)."""
    import exact_scaled_dot_gb300 as esd
    w = PADDED["gqa_causal"]
    base = BASES["gqa_causal"]
    inp = make_inputs(w)
    pq = _positions(w.B, w.nq, 5)
    rot = esd.Rotary(pq.cuda(), pq.cuda(), base=base)
    res = _run_fused(w, inp, rot)
    Q, K, V, G = (x.cuda() for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = inp.kv_len.tolist()
    Qr, Kr = _rope_padded_gpu(Q, pq, base), _rope_padded_gpu(K, pq, base)
    O, L, Olo = esd.attn_fwd(Qr, Kr, V, causal=True, kv_len=kv)
    dQr, dKr, dV = esd.attn_bwd(Qr, Kr, V, O, G, L, O_lo=Olo, causal=True, kv_len=kv)
    dQ, dK = _rope_padded_gpu(dQr, pq, base, inverse=True), _rope_padded_gpu(dKr, pq, base, inverse=True)
    torch.cuda.synchronize()
    assert_same_sum(res["dV"], dV, "dV")
    assert_close(f64(res["dQ"]), f64(dQ), "dQ vs separate")
    assert_close(f64(res["dK"]), f64(dK), "dK vs separate")


def test_staged_and_noalloc_backward_with_rotary():
    """The three stage calls with the same rotary, and attn_bwd_noalloc, equal
    the composite attn_bwd (up to the order of their fp32 sums)."""
    import exact_scaled_dot_gb300 as esd
    w = PADDED["mha_d64"]
    inp = make_inputs(w)
    pq = _positions(w.B, w.nq, 9, big=True)
    rot = esd.Rotary(pq.cuda(), pq.cuda(), base=10000.0)
    res = _run_fused(w, inp, rot)
    Q, K, V, G = (x.cuda() for x in (inp.Q, inp.K, inp.V, inp.dO))
    shape = esd.make_shape(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    ws = torch.empty((esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, rotary=rot),),
                     dtype=torch.uint8, device="cuda:0")
    dQ, dK, dV = (torch.full_like(x, float("nan")) for x in (Q, K, V))
    esd.attn_bwd_preprocess(Q, res["O"], G, ws, shape=shape, O_lo=res["O_lo"], rotary=rot)
    esd.attn_bwd_main(K, V, res["LSE"], ws, dK, dV, shape=shape, causal=True, rotary=rot)
    esd.attn_bwd_finalize(ws, dQ, shape=shape, rotary=rot)
    nQ, nK, nV = esd.attn_bwd_noalloc(Q, K, V, res["O"], G, res["LSE"], O_lo=res["O_lo"], causal=True, rotary=rot)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    for got in ((dQ, dK, dV), (nQ, nK, nV)):
        assert_same_sum(got[1], res["dK"], "dK")
        assert_same_sum(got[2], res["dV"], "dV")
        assert_close(f64(got[0]), f64(res["dQ"]), "dQ", atol=1e-3, rtol=1e-3)


# ---------------------------------------------------------------------------
# packed sequences
# ---------------------------------------------------------------------------
def _varlen_oracle_rotary(orc, w, inp, pq, pk, base):
    import oracle
    from oracle.rope import rope
    Q, K, V, G = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    Qr, Kr = _bf16(rope(Q, pq, base=base)), _bf16(rope(K, pk, base=base))
    Tq, Tk = Q.shape[0], K.shape[0]
    O = np.zeros((Tq, w.Hq, w.dv))
    LSE = np.zeros((w.Hq, Tq))
    dQr = np.zeros((Tq, w.Hq, w.dh))
    dKr = np.zeros((Tk, w.Hkv, w.dh))
    dV = np.zeros((Tk, w.Hkv, w.dv))
    to_bhnd = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2)[None])  # noqa: E731
    for b in range(len(inp.lens_q)):
        lq, lk = inp.lens_q[b], inp.lens_k[b]
        q0, q1, k0, k1 = inp.cu_q[b], inp.cu_q[b + 1], inp.cu_k[b], inp.cu_k[b + 1]
        if lq == 0:
            continue
        p = oracle.Problem(1, w.Hq, w.Hkv, lq, lk, w.dh, w.dv, causal=w.causal, offset=None, kv_len=None)
        Qb, Kb, Vb, Gb = to_bhnd(Qr[q0:q1]), to_bhnd(Kr[k0:k1]), to_bhnd(V[k0:k1]), to_bhnd(G[q0:q1])
        Ob, Lb = orc.forward(p, Qb, Kb, Vb)
        a, c, e, _D, _C = orc.backward(p, Qb, Kb, Vb, Gb)
        O[q0:q1] = Ob[0].transpose(1, 0, 2)
        LSE[:, q0:q1] = Lb[0]
        dQr[q0:q1] = a[0].transpose(1, 0, 2)
        dKr[k0:k1] = c[0].transpose(1, 0, 2)
        dV[k0:k1] = e[0].transpose(1, 0, 2)
    return dict(O=O, LSE=LSE, dQ=rope(dQr, pq, base=base, inverse=True), dK=rope(dKr, pk, base=base, inverse=True),
                dV=dV)


VARLEN = {
    "causal_gqa_restart": VarlenWorkload("rot_varlen_gqa", B=3, Hq=8, Hkv=2, dh=128, dv=128, causal=True,
                                         lens_q=(1, 300, 129), seed=84),
    "chunks_over_history": VarlenWorkload("rot_varlen_chunks", B=2, Hq=4, Hkv=1, dh=128, dv=128, causal=True,
                                          lens_q=(100, 16), lens_k=(600, 200), seed=85),
}


@pytest.mark.parametrize("name", list(VARLEN))
def test_fused_rotary_packed_matches_oracle(orc, name):
    """Packed sequences: positions restart at 0 in every sequence, and a chunk
    of new queries over a history sits at the history's end (query i of a
    sequence at len_k - len_q + i, key j at j)."""
    import exact_scaled_dot_gb300 as esd
    w = VARLEN[name]
    inp = make_varlen_inputs(w)
    pq = np.concatenate([np.arange(lk - lq, lk) for lq, lk in zip(inp.lens_q, inp.lens_k)]).astype(np.int32)
    pk = np.concatenate([np.arange(lk) for lk in inp.lens_k]).astype(np.int32)
    rot = esd.Rotary(torch.from_numpy(pq).cuda(), torch.from_numpy(pk).cuda(), base=10000.0)
    Q, K, V, G = (x.cuda() for x in (inp.Q, inp.K, inp.V, inp.dO))
    O, LSE, O_lo = esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=w.causal, rotary=rot)
    dQ, dK, dV = esd.attn_bwd_varlen(Q, K, V, O, G, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=w.causal,
                                     rotary=rot)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    ref = _varlen_oracle_rotary(orc, w, inp, pq, pk, 10000.0)
    assert_close(f64(O), ref["O"], "O")
    assert_close(f64(LSE), ref["LSE"], "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(dQ), ref["dQ"], "dQ")
    assert_close(f64(dK), ref["dK"], "dK")
    assert_close(f64(dV), ref["dV"], "dV")
    # the fused packed forward equals the separate rotation, bit for bit
    Qr = esd.attn_rope(Q, rot.pos_q, base=10000.0)
    Kr = esd.attn_rope(K, rot.pos_k, base=10000.0)
    O2, L2, Olo2 = esd.attn_fwd_varlen(Qr, Kr, V, inp.cu_q, inp.cu_k, causal=w.causal)
    torch.cuda.synchronize()
    assert torch.equal(O, O2) and torch.equal(LSE, L2) and torch.equal(O_lo, Olo2)


def test_rotary_with_strided_fused_qkv():
    """Rotary and strides together: Q, K, V sliced from one fused projection
    output, rotated inside the packed calls, equal the same calls on
    contiguous copies."""
    import exact_scaled_dot_gb300 as esd
    w = VARLEN["causal_gqa_restart"]
    inp = make_varlen_inputs(w)
    T = inp.Q.shape[0]
    pos = np.concatenate([np.arange(lq) for lq in inp.lens_q]).astype(np.int32)
    rot = esd.Rotary(torch.from_numpy(pos).cuda(), torch.from_numpy(pos).cuda(), base=10000.0)
    Qc, Kc, Vc, G = (x.cuda() for x in (inp.Q, inp.K, inp.V, inp.dO))
    qkv = torch.cat([Qc.reshape(T, -1), Kc.reshape(T, -1), Vc.reshape(T, -1)], dim=1)
    a, b = w.Hq * w.dh, (w.Hq + w.Hkv) * w.dh
    Q = qkv[:, :a].view(T, w.Hq, w.dh)
    K = qkv[:, a:b].view(T, w.Hkv, w.dh)
    V = qkv[:, b:].view(T, w.Hkv, w.dv)
    outs = []
    for q, k, v in ((Q, K, V), (Qc, Kc, Vc)):
        O, L, Olo = esd.attn_fwd_varlen(q, k, v, inp.cu_q, inp.cu_k, causal=True, rotary=rot)
        outs.append((O, L) + esd.attn_bwd_varlen(q, k, v, O, G, L, inp.cu_q, inp.cu_k, O_lo=Olo, causal=True,
                                                 rotary=rot))
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    for i, name in enumerate(("O", "LSE", "dQ", "dK", "dV")):
        if name in ("dQ", "dK", "dV"):
            assert_same_sum(outs[0][i], outs[1][i], name)
        else:
            assert torch.equal(outs[0][i], outs[1][i]), name


@pytest.mark.parametrize("name", ["gqa_causal", "cross_dv64"])
def test_rotated_row_residuals(orc, name):
    """With q_rot, k_rot the forward leaves its rotated rows there (equal, bit
    for bit, to attn_rope's) and a backward given them reads them instead of
    rotating again: its gradients equal those of the backward that rotates
    by itself (up to the order of their fp32 sums), and
    match the oracle."""
    import exact_scaled_dot_gb300 as esd
    w = PADDED[name]
    base = BASES[name]
    inp = make_inputs(w)
    pq = _positions(w.B, w.nq, w.seed + 3, big=True)
    pk = _positions(w.B, w.nk, w.seed + 4, big=True)
    Q, K, V, G = (x.cuda() for x in (inp.Q, inp.K, inp.V, inp.dO))
    q_rot, k_rot = torch.full_like(Q, float("nan")), torch.full_like(K, float("nan"))
    kept = esd.Rotary(pq.cuda(), pk.cuda(), base=base, q_rot=q_rot, k_rot=k_rot)
    plain = esd.Rotary(pq.cuda(), pk.cuda(), base=base)
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    O, L, Olo = esd.attn_fwd(Q, K, V, causal=w.causal, kv_len=kv, rotary=kept)
    torch.cuda.synchronize()
    assert torch.equal(q_rot, _rope_padded_gpu(Q, pq, base)) and torch.equal(k_rot, _rope_padded_gpu(K, pk, base))
    g1 = esd.attn_bwd(Q, K, V, O, G, L, O_lo=Olo, causal=w.causal, kv_len=kv, rotary=kept)
    g2 = esd.attn_bwd(Q, K, V, O, G, L, O_lo=Olo, causal=w.causal, kv_len=kv, rotary=plain)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    assert_same_sum(g1[1], g2[1], "dK")
    assert_same_sum(g1[2], g2[2], "dV")
    assert_close(f64(g1[0]), f64(g2[0]), "dQ", atol=1e-3, rtol=1e-3)
    ref = _oracle_rotary(orc, w, inp, pq.numpy(), pk.numpy(), base)
    for k, got in zip(("dQ", "dK", "dV"), g1):
        assert_close(f64(got), ref[k], k)
