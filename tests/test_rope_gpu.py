"""GPU-vs-oracle parity of the rotary embedding (attn_rope) and of attention
over rotated queries and keys: the rotation within 1e-2 + 2e-2 |ref| of the
fp64 rotation with exact angles (positions up to 2^24 - 1, the largest the
kernel takes; a frequency rounded to fp32 alone would be off by 0.06 rad at
10^6), the inverse undoing
it, and packed causal attention over GPU-rotated Q, K matching the oracle's
rotation (rounded to bf16, the precision of the rotated tensors) followed by
the oracle's attention."""
import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import VarlenWorkload, make_varlen_inputs

from _attn_cases import LSE_ATOL, assert_close, f64

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


@pytest.mark.parametrize("T,H,d,base,maxpos", [(1000, 4, 128, 10000.0, 65535), (333, 2, 64, 500000.0, 4096),
                                                (64, 1, 8, 10.0, 100000), (777, 2, 128, 10000.0, 1_000_000),
                                                (512, 3, 64, 10000.0, (1 << 24) - 1)])
def test_rope_matches_oracle(T, H, d, base, maxpos):
    from oracle.rope import rope
    import exact_scaled_dot_gb300 as esd
    g = torch.Generator().manual_seed(T + d)
    X = torch.randn((T, H, d), generator=g).to(torch.bfloat16)
    pos = torch.randint(0, maxpos + 1, (T,), generator=g, dtype=torch.int32)
    Xd, Pd = X.cuda(), pos.cuda()
    Y = esd.attn_rope(Xd, Pd, base=base)
    Z = esd.attn_rope(Y, Pd, base=base, inverse=True)
    torch.cuda.synchronize()
    ref = rope(f64(X), pos.numpy(), base=base)
    assert_close(f64(Y), ref, "rotated")
    assert_close(f64(Z), f64(X), "rotated back")
    W = Xd.clone()
    esd.attn_rope(W, Pd, base=base, Y=W)   # in place
    torch.cuda.synchronize()
    assert torch.equal(W, Y)


def test_attention_over_rotated_queries_and_keys(orc):
    import oracle
    from oracle.rope import rope
    import exact_scaled_dot_gb300 as esd
    w = VarlenWorkload("rope", B=2, Hq=4, Hkv=2, dh=128, dv=128, causal=True, lens_q=(300, 129), seed=71)
    inp = make_varlen_inputs(w)
    # positions restart at 0 in every sequence
    pos = np.concatenate([np.arange(n) for n in inp.lens_q]).astype(np.int32)
    d = "cuda:0"
    P = torch.from_numpy(pos).to(d)
    Qr = esd.attn_rope(inp.Q.to(d), P)
    Kr = esd.attn_rope(inp.K.to(d), P)
    O, LSE, _ = esd.attn_fwd_varlen(Qr, Kr, inp.V.to(d), inp.cu_q, inp.cu_k, causal=True)
    torch.cuda.synchronize()
    # The rotated rows are stored in bf16 (the precision of the tensors the
    # attention reads), so the reference rounds its exact rotation the same way.
    bf16 = lambda x: torch.from_numpy(x).to(torch.bfloat16).double().numpy()  # noqa: E731
    Qn, Kn = bf16(rope(f64(inp.Q), pos)), bf16(rope(f64(inp.K), pos))
    Vn = f64(inp.V)
    for b in range(2):
        q0, q1 = inp.cu_q[b], inp.cu_q[b + 1]
        n = q1 - q0
        p = oracle.Problem(1, 4, 2, n, n, 128, 128, causal=True)
        tr = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2)[None])  # noqa: E731
        Oref, Lref = orc.forward(p, tr(Qn[q0:q1]), tr(Kn[q0:q1]), tr(Vn[q0:q1]))
        assert_close(f64(O[q0:q1]), Oref[0].transpose(1, 0, 2), f"O[{b}]")
        assert_close(f64(LSE[:, q0:q1]), Lref[0], f"LSE[{b}]", atol=LSE_ATOL, rtol=0.0)


@pytest.mark.parametrize("T,Hq,Hk,d,inverse", [(1000, 32, 8, 128, False), (333, 5, 3, 64, True),
                                               (64, 1, 9, 8, False)])
def test_rope_qk_equals_two_calls(T, Hq, Hk, d, inverse):
    """One launch for queries and keys gives the two single-tensor results bit
    for bit (the kernel is the same; only the work items are concatenated),
    head counts that are not multiples of the kernel's 8-head groups
    included, and in place as well."""
    import exact_scaled_dot_gb300 as esd
    g = torch.Generator().manual_seed(T + Hq + Hk)
    Q = torch.randn((T, Hq, d), generator=g).to(torch.bfloat16).cuda()
    K = torch.randn((T, Hk, d), generator=g).to(torch.bfloat16).cuda()
    pos = torch.randint(0, 70000, (T,), generator=g, dtype=torch.int32).cuda()
    Yq, Yk = esd.attn_rope_qk(Q, K, pos, base=10000.0, inverse=inverse)
    Rq = esd.attn_rope(Q, pos, base=10000.0, inverse=inverse)
    Rk = esd.attn_rope(K, pos, base=10000.0, inverse=inverse)
    Q2, K2 = Q.clone(), K.clone()
    esd.attn_rope_qk(Q2, K2, pos, base=10000.0, inverse=inverse, Yq=Q2, Yk=K2)
    torch.cuda.synchronize()
    assert torch.equal(Yq.view(torch.int16), Rq.view(torch.int16))
    assert torch.equal(Yk.view(torch.int16), Rk.view(torch.int16))
    assert torch.equal(Q2.view(torch.int16), Rq.view(torch.int16))
    assert torch.equal(K2.view(torch.int16), Rk.view(torch.int16))
