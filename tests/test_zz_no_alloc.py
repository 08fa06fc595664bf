"""The backward entry point that allocates nothing (attn_bwd_noalloc).

Some callers cannot allocate device memory where they run the backward pass
(memory owned by a fixed arena or another runtime; loops that cannot afford
an allocation's device-wide synchronisation).  attn_bwd_noalloc serves them
from a static buffer inside the library.  This test calls it through the C
ABI twice in a row and compares each result with the ordinary attn_bwd on
the same inputs, and with the fp64 oracle, within the parity tolerance the
other GPU tests use.  The file is named so that pytest collects it last; it
also runs on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from exact_scaled_dot_gb300.inputs import Workload, make_inputs

from _attn_cases import assert_close, f64, problem_of

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 2e-2


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from exact_scaled_dot_gb300 import build as b
    b.build()
    import exact_scaled_dot_gb300 as esd
    esd.load()
    esd.attn_clear_status()
    yield


def _close(got, ref, what):
    g, r = got.double(), ref.double()
    bad = ~((g - r).abs() <= ATOL + RTOL * r.abs())
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements outside tolerance"


def test_noalloc_backward_matches_workspace_backward_twice(orc):
    import exact_scaled_dot_gb300 as esd
    w = Workload("noalloc", B=2, Hq=4, Hkv=2, nq=200, nk=256, dh=128, dv=128, causal=True,
                 kv_len_range=(120, 256), seed=41)
    inp = make_inputs(w)
    dev = torch.device("cuda", 0)
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = inp.kv_len.tolist()
    need = esd.attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
    assert 0 < need <= esd.attn_bwd_noalloc_max_scratch_bytes()

    O, LSE, O_lo = esd.attn_fwd(Q, K, V, causal=True, kv_len=kv)
    ref = esd.attn_bwd(Q, K, V, O, dO, LSE, O_lo=O_lo, causal=True, kv_len=kv)
    rdQ, rdK, rdV, _D, _C = orc.backward(problem_of(w, inp), *(f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO)))
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in ref]
        esd.attn_bwd_noalloc(Q, K, V, O, dO, LSE, O_lo=O_lo, causal=True, kv_len=kv,
                             dQ=outs[0], dK=outs[1], dV=outs[2])
        torch.cuda.synchronize()
        assert esd.attn_get_status() == esd.ATTN_OK
        for name, got, want, orc_ref in zip(("dQ", "dK", "dV"), outs, ref, (rdQ, rdK, rdV)):
            _close(got, want, f"call {call}: {name}")
            assert_close(f64(got), orc_ref, f"call {call}: {name} vs oracle")


def test_noalloc_refuses_problems_beyond_its_buffer():
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300 import _binding as bnd
    lib = esd.load()
    shape = bnd.make_shape(4, 16, 16, 2048, 2048, 128, 128)   # about 135 MB of scratch
    assert esd.attn_bwd_workspace_bytes(4, 16, 16, 2048, 2048, 128, 128) > esd.attn_bwd_noalloc_max_scratch_bytes()
    mask = bnd.AttnMask(1, 0, bnd.ATTN_OFFSET_DEFAULT, ctypes.POINTER(ctypes.c_int32)())
    p = ctypes.c_void_p(256)
    rc = lib.attn_bwd_noalloc(ctypes.byref(shape), ctypes.byref(mask), None, None, ctypes.c_float(0.088), p, p, p, p,
                              None,
                              p, p, p, p, p, None)
    assert rc == esd.ATTN_ERR_WORKSPACE
