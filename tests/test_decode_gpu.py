"""GPU-vs-oracle parity of the short-query forward (attn_fwd_decode): query
heads packed per tile, key range split across CTAs and merged by log-sum-exp.

Every case is compared element by element with the fp64 oracle (O within
1e-2 + 2e-2 |ref|, LSE within 1e-3), and with the regular forward on the
same inputs.  The shapes cover single-query decode (MQA, GQA), small chunks
of new queries over a history (the causal offset n_k - n_q), a chunk that
spans two row tiles, full tiles, no split, d = 64 and d_v = 64, key padding
with NaN in the padded rows, a peaked softmax, and full 128-row tiles over
key ranges of one, two, three and five tiles.
"""
import numpy as np
import pytest
import torch

from exact_scaled_dot_gb300.inputs import Workload, make_inputs

from _attn_cases import LSE_ATOL, assert_close, f64, problem_of

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


CASES = {
    "mqa_single_query": Workload("mqa_single_query", B=2, Hq=16, Hkv=1, nq=1, nk=1500, dh=128, dv=128, causal=True,
                                 kv_len_range=(800, 1500), seed=41),
    "gqa_chunk_of_4": Workload("gqa_chunk_of_4", B=2, Hq=8, Hkv=2, nq=4, nk=2000, dh=128, dv=128, causal=True,
                               kv_len_range=(1000, 2000), seed=42),
    "full_tile_no_mask": Workload("full_tile_no_mask", B=1, Hq=16, Hkv=2, nq=16, nk=700, dh=128, dv=128, seed=43),
    "two_row_tiles": Workload("two_row_tiles", B=1, Hq=32, Hkv=1, nq=5, nk=900, dh=128, dv=128, causal=True,
                              seed=44),
    "d64": Workload("d64", B=2, Hq=4, Hkv=2, nq=3, nk=600, dh=64, dv=64, causal=True, kv_len_range=(200, 600),
                    seed=45),
    "dv64_peaked": Workload("dv64_peaked", B=2, Hq=4, Hkv=1, nq=8, nk=1100, dh=128, dv=64,
                            kv_len_range=(500, 1100), sigma_qk=3.0, seed=46),
    "no_split_many_tiles": Workload("no_split_many_tiles", B=8, Hq=40, Hkv=40, nq=2, nk=200, dh=128, dv=128,
                                    causal=True, seed=47),
    "max_rows_128": Workload("max_rows_128", B=1, Hq=2, Hkv=2, nq=128, nk=1000, dh=128, dv=128, causal=True,
                             seed=48),
    "explicit_offset": Workload("explicit_offset", B=1, Hq=8, Hkv=1, nq=3, nk=1200, dh=128, dv=128, causal=True,
                                offset=700, seed=49),
    # Full 128-row tiles over key ranges of one, two, three and (split) five
    # tiles: the scores run one tile ahead of the softmax, so the first and
    # last tiles of a range and the wait for the last PV product are edge
    # cases, with four softmax warps in play.
    "rows128_one_tile": Workload("rows128_one_tile", B=2, Hq=16, Hkv=2, nq=16, nk=100, dh=128, dv=128, causal=True,
                                 seed=50),
    "rows128_two_tiles": Workload("rows128_two_tiles", B=2, Hq=16, Hkv=2, nq=16, nk=250, dh=128, dv=128, seed=51),
    "rows128_three_tiles": Workload("rows128_three_tiles", B=2, Hq=16, Hkv=2, nq=16, nk=300, dh=128, dv=64,
                                    causal=True, kv_len_range=(260, 300), seed=52),
    "rows128_five_tiles_split": Workload("rows128_five_tiles_split", B=1, Hq=16, Hkv=2, nq=16, nk=600, dh=128,
                                         dv=128, causal=True, seed=53),
}


def _run(w: Workload, inp, poison_padding=False):
    import exact_scaled_dot_gb300 as esd
    dev = "cuda:0"
    Q, K, V = (x.to(dev) for x in (inp.Q, inp.K, inp.V))
    if poison_padding and inp.kv_len is not None:
        for b, L in enumerate(inp.kv_len.tolist()):
            K[b, :, L:, :] = float("nan")
            V[b, :, L:, :] = float("nan")
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    mask = dict(causal=w.causal, causal_offset=w.causal_offset if w.causal else None, kv_len=kv)
    O = torch.full((w.B, w.Hq, w.nq, w.dv), float("nan"), dtype=torch.bfloat16, device=dev)
    LSE = torch.full((w.B, w.Hq, w.nq), float("nan"), dtype=torch.float32, device=dev)
    esd.attn_fwd_decode(Q, K, V, O=O, LSE=LSE, **mask)
    torch.cuda.synchronize()
    assert esd.attn_get_status() == 0
    return O, LSE, Q, K, V, mask


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(orc, name):
    w = CASES[name]
    inp = make_inputs(w)
    O, LSE, Q, K, V, mask = _run(w, inp)
    p = problem_of(w, inp)
    Oref, Lref = orc.forward(p, f64(inp.Q), f64(inp.K), f64(inp.V))
    assert_close(f64(O), Oref, "O")
    assert_close(f64(LSE), Lref, "LSE", atol=LSE_ATOL, rtol=0.0)


@pytest.mark.parametrize("name", ["mqa_single_query", "gqa_chunk_of_4", "dv64_peaked"])
def test_decode_agrees_with_regular_forward(name):
    """Same inputs through attn_fwd: both paths compute the same function."""
    import exact_scaled_dot_gb300 as esd
    w = CASES[name]
    inp = make_inputs(w)
    O, LSE, Q, K, V, mask = _run(w, inp)
    O2, LSE2, _ = esd.attn_fwd(Q, K, V, **mask)
    torch.cuda.synchronize()
    assert_close(f64(O), f64(O2), "O vs attn_fwd", atol=1e-2, rtol=2e-2)
    np.testing.assert_allclose(f64(LSE), f64(LSE2), atol=1e-3, rtol=0)


def test_decode_ignores_nan_in_key_padding(orc):
    w = CASES["gqa_chunk_of_4"]
    inp = make_inputs(w)
    O, LSE, *_ = _run(w, inp, poison_padding=True)
    clean = make_inputs(w)
    for b, L in enumerate(clean.kv_len.tolist()):
        clean.K[b, :, L:, :] = 0
        clean.V[b, :, L:, :] = 0
    p = problem_of(w, clean)
    Oref, Lref = orc.forward(p, f64(clean.Q), f64(clean.K), f64(clean.V))
    assert_close(f64(O), Oref, "O")
    assert_close(f64(LSE), Lref, "LSE", atol=LSE_ATOL, rtol=0.0)


def test_decode_split_and_workspace_sizes():
    """Few row tiles split the key range (the merge runs); many do not."""
    import exact_scaled_dot_gb300 as esd
    few = CASES["mqa_single_query"]
    assert esd.attn_fwd_decode_workspace_bytes(few.B, few.Hq, few.Hkv, few.nq, few.nk, few.dh, few.dv,
                                               causal=True, kv_len=[1500, 1500]) > 0
    many = CASES["no_split_many_tiles"]
    assert esd.attn_fwd_decode_workspace_bytes(many.B, many.Hq, many.Hkv, many.nq, many.nk, many.dh, many.dv,
                                               causal=True) == 0
