"""Failure detection on the GPU without a fault: a kernel waits on a barrier
that nothing completes, gives up after its time limit, records
ATTN_ERR_TIMEOUT in the device status word and returns.  The context stays
usable: while the status is set the attention kernels skip their work, and
after attn_clear_status() they run normally again."""
import pytest
import torch

from exact_scaled_dot_gb300.inputs import Workload, make_inputs

from _attn_cases import compare_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from exact_scaled_dot_gb300 import build as b
    b.build()
    import exact_scaled_dot_gb300 as esd
    esd.load()
    esd.attn_clear_status()
    yield
    esd.attn_clear_status()


def test_bounded_wait_reports_timeout_and_context_survives(orc):
    import exact_scaled_dot_gb300 as esd
    assert esd.attn_get_status() == esd.ATTN_OK
    esd.attn_selftest_wait_timeout(50_000_000)          # 50 ms limit
    torch.cuda.synchronize()
    assert esd.attn_get_status() == esd.ATTN_ERR_TIMEOUT

    # While the status is set, kernels return at once and leave outputs alone.
    w = Workload("after_timeout", B=1, Hq=2, Hkv=1, nq=130, nk=130, dh=64, dv=64, causal=True, seed=31)
    inp = make_inputs(w)
    res = run_gpu(w, inp, poison=True)
    assert res.status == esd.ATTN_ERR_TIMEOUT
    assert bool(torch.isnan(res.O.float()).all())

    # Cleared, the same call computes the right answer.
    esd.attn_clear_status()
    assert esd.attn_get_status() == esd.ATTN_OK
    compare_full(w, inp, run_gpu(w, inp), orc)
