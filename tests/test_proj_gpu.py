"""GPU-vs-oracle parity of the projection products (attn_proj_fwd,
attn_proj_bwd_weight, attn_proj_bwd_input; "Appendix A.10", eqs.
A.10.10-A.10.11): each output element within 1e-2 + 2e-2 |ref| of the fp64
product of the same bf16 inputs.  Shapes leave ragged edges on every side of
the 128 x 256 x 64 tiles (and a width that is not a multiple of 64), the input
gradient sums one, two and three branches, and a full-size case is checked on
sampled rows and entries.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import make_proj_inputs

from _attn_cases import assert_close, f64

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


SHAPES = [
    (300, 200, (136,)),
    (1000, 512, (1024, 256, 256)),
    (129, 64, (8, 72)),
    (2048, 384, (640, 128)),
]


def _dev(inp):
    d = "cuda:0"
    return inp.X.to(d), [w.to(d) for w in inp.Ws], [g.to(d) for g in inp.Gs]


@pytest.mark.parametrize("T,D,Ns", SHAPES)
def test_projection_forward(T, D, Ns):
    from oracle.projections import proj_forward
    import exact_scaled_dot_gb300 as esd
    inp = make_proj_inputs(T, D, Ns, seed=T + D)
    X, Ws, _Gs = _dev(inp)
    for k, W in enumerate(Ws):
        Y = esd.attn_proj_fwd(X, W)
        torch.cuda.synchronize()
        assert_close(f64(Y), proj_forward(f64(inp.X), f64(inp.Ws[k])), f"Y[{k}]")


@pytest.mark.parametrize("T,D,Ns", SHAPES)
def test_projection_weight_gradient(T, D, Ns):
    from oracle.projections import proj_grad_weight
    import exact_scaled_dot_gb300 as esd
    inp = make_proj_inputs(T, D, Ns, seed=T + D + 1)
    X, _Ws, Gs = _dev(inp)
    for k, G in enumerate(Gs):
        dW = esd.attn_proj_bwd_weight(X, G)
        torch.cuda.synchronize()
        assert_close(f64(dW), proj_grad_weight(f64(inp.X), f64(inp.Gs[k])), f"dW[{k}]")


@pytest.mark.parametrize("T,D,Ns", SHAPES)
def test_projection_input_gradient_sums_branches(T, D, Ns):
    from oracle.projections import proj_grad_input
    import exact_scaled_dot_gb300 as esd
    inp = make_proj_inputs(T, D, Ns, seed=T + D + 2)
    _X, Ws, Gs = _dev(inp)
    dX = esd.attn_proj_bwd_input(Gs, Ws)
    torch.cuda.synchronize()
    ref = proj_grad_input([(f64(g), f64(w)) for g, w in zip(inp.Gs, inp.Ws)])
    assert_close(f64(dX), ref, "dX")
    if len(Ns) > 1:
        # one branch alone is a different number: the sum is really taken
        only = esd.attn_proj_bwd_input(Gs[:1], Ws[:1])
        torch.cuda.synchronize()
        assert not np.allclose(f64(only), ref, atol=1e-2)


def test_full_size_sampled():
    """The benchmark's shapes (8192 tokens of width 4096 into 4096 + 1024 +
    1024 columns): sampled output rows of Y and dX, sampled entries of dW."""
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300.inputs import PROJ_WORKLOADS
    cfg = PROJ_WORKLOADS["proj_qkv_gqa"]
    inp = make_proj_inputs(cfg["T"], cfg["D"], cfg["Ns"], cfg["seed"])
    X, Ws, Gs = _dev(inp)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 127, 128, cfg["T"] - 1], rng.integers(0, cfg["T"], 24)]))
    Xn = f64(inp.X)
    for k in range(3):
        Y = esd.attn_proj_fwd(X, Ws[k])
        dW = esd.attn_proj_bwd_weight(X, Gs[k])
        torch.cuda.synchronize()
        Wn, Gn = f64(inp.Ws[k]), f64(inp.Gs[k])
        assert_close(f64(Y)[rows], Xn[rows] @ Wn, f"Y[{k}] rows")
        dr = rng.integers(0, cfg["D"], 48)
        dc = rng.integers(0, Wn.shape[1], 48)
        ref = np.einsum("td,tn->dn", Xn[:, dr], Gn[:, dc])[np.arange(48), np.arange(48)]
        assert_close(f64(dW)[dr, dc], ref, f"dW[{k}] entries")
    dX = esd.attn_proj_bwd_input(Gs, Ws)
    torch.cuda.synchronize()
    ref = sum(f64(inp.Gs[k])[rows] @ f64(inp.Ws[k]).T for k in range(3))
    assert_close(f64(dX)[rows], ref, "dX rows")
