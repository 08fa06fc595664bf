"""Host-side tests of the C ABI: the library builds, loads and exports every
symbol include/attn.h declares, and argument checks reject bad calls before
any CUDA call (so they run without a GPU)."""
import ctypes
import math
import re
from pathlib import Path

import pytest
import torch

import exact_scaled_dot_gb300 as esd
from exact_scaled_dot_gb300 import _binding as bnd
from exact_scaled_dot_gb300.build import build

HEADER = Path(__file__).resolve().parent.parent / "include" / "attn.h"


@pytest.fixture(scope="module")
def lib():
    build()
    return esd.load()


def _declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_exactly_the_bound_symbols():
    assert sorted(bnd.EXPORTS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert esd.attn_abi_version() == 12


def test_strerror_covers_every_code(lib):
    codes = [getattr(bnd, n) for n in dir(bnd) if n.startswith("ATTN_ERR_") or n == "ATTN_OK"]
    for c in codes:
        assert lib.attn_strerror(c).decode() not in ("", "unknown status")
    assert lib.attn_strerror(999).decode() == "unknown status"


def _call_fwd(lib, shape, mask, scale=None, ptr=256, ws=256, ws_bytes=1 << 40, strides=None, rotary=None):
    p = ctypes.c_void_p(ptr)
    scale = 1.0 / math.sqrt(max(shape.d_h, 1)) if scale is None else scale
    return lib.attn_fwd(ctypes.byref(shape), ctypes.byref(mask) if mask is not None else None, strides, rotary,
                        ctypes.c_float(scale), p, p, p, p, p, None, ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes),
                        None)


def _mask(causal=0, offset=bnd.ATTN_OFFSET_DEFAULT, kv=None, reserved=0):
    keep = None
    ptr = ctypes.POINTER(ctypes.c_int32)()
    if kv is not None:
        keep = (ctypes.c_int32 * len(kv))(*kv)
        ptr = ctypes.cast(keep, ctypes.POINTER(ctypes.c_int32))
    m = bnd.AttnMask(causal, reserved, offset, ptr)
    m._keep = keep
    return m


GOOD = dict(B=2, Hq=4, Hkv=2, n_q=100, n_k=100, d_h=128, d_v=128)


def _shape(**kw):
    d = dict(GOOD)
    d.update(kw)
    return bnd.make_shape(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), bnd.ATTN_ERR_SHAPE),
    (dict(n_q=-1), bnd.ATTN_ERR_SHAPE),
    (dict(Hq=3), bnd.ATTN_ERR_SHAPE),
    (dict(B=bnd.ATTN_MAX_BATCH + 1), bnd.ATTN_ERR_SHAPE),
    (dict(d_h=96, d_v=96), bnd.ATTN_ERR_UNSUPPORTED),
    (dict(d_h=64, d_v=128), bnd.ATTN_ERR_UNSUPPORTED),
])
def test_bad_shapes_rejected(lib, kw, code):
    assert _call_fwd(lib, _shape(**kw), _mask()) == code


def test_empty_rows_rejected_in_closed_form(lib):
    # causal with a negative offset: row 0 sees nothing ("Chapter 31", section 3).
    assert _call_fwd(lib, _shape(), _mask(causal=1, offset=-1)) == bnd.ATTN_ERR_EMPTY_ROW
    # default bottom-right alignment with more queries than keys: first rows empty.
    assert _call_fwd(lib, _shape(n_q=200, n_k=100), _mask(causal=1)) == bnd.ATTN_ERR_EMPTY_ROW
    # a batch element with no keys.
    assert _call_fwd(lib, _shape(), _mask(kv=[100, 0])) == bnd.ATTN_ERR_EMPTY_ROW


def test_bad_masks_rejected(lib):
    assert _call_fwd(lib, _shape(), _mask(kv=[100, 101])) == bnd.ATTN_ERR_SHAPE
    assert _call_fwd(lib, _shape(), _mask(kv=[-3, 10])) == bnd.ATTN_ERR_SHAPE
    assert _call_fwd(lib, _shape(), _mask(reserved=1)) == bnd.ATTN_ERR_SHAPE
    assert _call_fwd(lib, _shape(), _mask(causal=2)) == bnd.ATTN_ERR_SHAPE
    assert _call_fwd(lib, _shape(), None) == bnd.ATTN_ERR_NULL


def test_bad_scale_and_pointers_rejected(lib):
    assert _call_fwd(lib, _shape(), _mask(), scale=0.0) == bnd.ATTN_ERR_SCALE
    assert _call_fwd(lib, _shape(), _mask(), scale=float("nan")) == bnd.ATTN_ERR_SCALE
    assert _call_fwd(lib, _shape(), _mask(), scale=-1.0) == bnd.ATTN_ERR_SCALE
    assert _call_fwd(lib, _shape(), _mask(), ptr=0) == bnd.ATTN_ERR_NULL
    assert _call_fwd(lib, _shape(), _mask(), ptr=0x1008) == bnd.ATTN_ERR_ALIGN


def test_fwd_workspace_checks(lib):
    """The forward's workspace (fp16 V tiles and their exponents) must be
    present, 256-byte aligned and large enough; checked before any CUDA call."""
    s = _shape(n_k=300, d_v=64, d_h=128)
    need = lib.attn_fwd_workspace_bytes(ctypes.byref(s), None)
    r256 = lambda x: ((x + 255) // 256) * 256  # noqa: E731
    tiles = 2 * 2 * 3     # B * Hkv * ceil(300 / 128)
    assert need == r256(tiles * 128 * 64 * 2) + r256(tiles * 4)
    assert _call_fwd(lib, s, _mask(), ws=0, ws_bytes=need) == bnd.ATTN_ERR_WORKSPACE
    assert _call_fwd(lib, s, _mask(), ws=512 + 16, ws_bytes=need) == bnd.ATTN_ERR_WORKSPACE
    assert _call_fwd(lib, s, _mask(), ws=512, ws_bytes=need - 1) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_fwd_workspace_bytes(ctypes.byref(_shape(B=0)), None) == 0


def test_bwd_workspace_checks(lib):
    s = _shape()
    need = lib.attn_bwd_workspace_bytes(ctypes.byref(s), None)
    rows = 2 * 4 * 100
    r256 = lambda x: ((x + 255) // 256) * 256  # noqa: E731
    # D | tile bounds and exponents | group exponents | work counter | fp32 dQ accumulator | fp16 copies of Q
    # and dO | fp32 sums of dK, dV (a launch of 4 work items with two query heads per KV head may split them)
    assert need == (r256(rows * 4) + r256(2 * 4 * 1 * 16) + r256(2 * 2 * 8) + 256 + r256(rows * 128 * 4)
                    + r256(rows * 128 * 2) + r256(rows * s.d_v * 2) + r256(2 * 100 * 2 * (128 + 128) * 4))
    # one query head per KV head: never split, no sums
    mha = _shape(Hq=2, Hkv=2)
    rows2 = 2 * 2 * 100
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(mha), None) == (
        r256(rows2 * 4) + r256(2 * 2 * 1 * 16) + r256(2 * 2 * 8) + 256 + r256(rows2 * 128 * 4) + r256(rows2 * 128 * 2)
        + r256(rows2 * 128 * 2))
    p = ctypes.c_void_p(256)
    m = _mask()
    args = [ctypes.byref(s), ctypes.byref(m), None, None, ctypes.c_float(0.1)] + [p] * 10
    assert lib.attn_bwd(*args, None, ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd(*args, ctypes.c_void_p(512), ctypes.c_size_t(need - 1), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd(*args, ctypes.c_void_p(512 + 16), ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(_shape(B=0)), None) == 0


def test_bwd_requires_the_output_residual(lib):
    """The backward's row terms come from O + O_lo: without O_lo the peaked
    cross-attention gradients miss the tolerance, so every backward entry
    point refuses a NULL O_lo with ATTN_ERR_NULL before any CUDA call."""
    s = _shape()
    need = lib.attn_bwd_workspace_bytes(ctypes.byref(s), None)
    p = ctypes.c_void_p(256)
    m = _mask()
    head = [ctypes.byref(s), ctypes.byref(m), None, None, ctypes.c_float(0.1)]
    # Q, K, V, O, O_lo = NULL, dO, LSE, dQ, dK, dV
    assert lib.attn_bwd(*head, p, p, p, p, None, p, p, p, p, p, p, ctypes.c_size_t(need),
                        None) == bnd.ATTN_ERR_NULL
    assert lib.attn_bwd_preprocess(ctypes.byref(s), None, None, p, p, None, p, p, ctypes.c_size_t(need),
                                   None) == bnd.ATTN_ERR_NULL
    assert lib.attn_bwd_noalloc(*head, p, p, p, p, None, p, p, p, p, p, None) == bnd.ATTN_ERR_NULL
    v = _varlen([0, 100], [0, 100])
    vneed = lib.attn_bwd_varlen_workspace_bytes(ctypes.byref(v), None)
    assert lib.attn_bwd_varlen(ctypes.byref(v), None, None, ctypes.c_float(0.1), p, p, p, p, None, p, p, p, p, p, p,
                               ctypes.c_size_t(vneed), None) == bnd.ATTN_ERR_NULL


def test_visible_pairs_closed_form(lib, orc):
    """The library's closed form equals the oracle's pair-by-pair count."""
    import oracle
    cases = [
        dict(B=2, Hq=2, Hkv=1, n_q=37, n_k=37, causal=True, offset=None, kv=[37, 20]),
        dict(B=1, Hq=3, Hkv=3, n_q=10, n_k=50, causal=True, offset=None, kv=None),
        dict(B=3, Hq=1, Hkv=1, n_q=20, n_k=30, causal=True, offset=4, kv=[30, 1, 9]),
        dict(B=2, Hq=2, Hkv=2, n_q=7, n_k=40, causal=False, offset=None, kv=[40, 13]),
        dict(B=1, Hq=1, Hkv=1, n_q=5, n_k=8, causal=True, offset=100, kv=None),
    ]
    for c in cases:
        got = esd.attn_visible_pairs(c["B"], c["Hq"], c["Hkv"], c["n_q"], c["n_k"], 64, 64, causal=c["causal"],
                                     causal_offset=c["offset"], kv_len=c["kv"])
        p = oracle.Problem(c["B"], c["Hq"], c["Hkv"], c["n_q"], c["n_k"], 64, 64, causal=c["causal"],
                           offset=c["offset"], kv_len=c["kv"])
        assert got == orc.visible_pairs(p), c


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        bnd.load(tmp_path / "nope.so")


def test_decode_entry_point_checks(lib):
    """attn_fwd_decode: n_q > 128 is unsupported (use attn_fwd); a needed
    workspace must be present and 256-byte aligned; all before any CUDA call."""
    m = _mask(causal=1)
    p = ctypes.c_void_p(256)
    big = _shape(n_q=129, n_k=1000)
    assert lib.attn_fwd_decode(ctypes.byref(big), ctypes.byref(m), ctypes.c_float(0.1), p, p, p, p, p, None,
                               None, ctypes.c_size_t(0), None) == bnd.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_decode_workspace_bytes(ctypes.byref(big), ctypes.byref(m)) == 0
    small = _shape(B=1, Hq=8, Hkv=1, n_q=1, n_k=4096)
    need = lib.attn_fwd_decode_workspace_bytes(ctypes.byref(small), ctypes.byref(m))
    # one row tile of 8 heads x 1 query: the key range is split, partials need a workspace
    assert need > 0 and need % 256 == 0
    args = [ctypes.byref(small), ctypes.byref(m), ctypes.c_float(0.1), p, p, p, p, p, None]
    assert lib.attn_fwd_decode(*args, None, ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_fwd_decode(*args, ctypes.c_void_p(512 + 16), ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_fwd_decode(*args, ctypes.c_void_p(512), ctypes.c_size_t(need - 1), None) == bnd.ATTN_ERR_WORKSPACE


def _varlen(cq, ck, causal=0, Hq=4, Hkv=2, d_h=128, d_v=128, B=None):
    B = len(cq) - 1 if B is None else B
    aq = (ctypes.c_int32 * len(cq))(*cq)
    ak = (ctypes.c_int32 * len(ck))(*ck)
    v = bnd.AttnVarlen(B, Hq, Hkv, d_h, d_v, causal, ctypes.cast(aq, ctypes.POINTER(ctypes.c_int32)),
                       ctypes.cast(ak, ctypes.POINTER(ctypes.c_int32)))
    v._keep = (aq, ak)
    return v


def test_varlen_checks(lib):
    """Packed sequences: offsets must start at 0 and not decrease; a sequence
    with queries needs keys, and under the causal (bottom-right) mask at least
    as many keys as queries; zero-query sequences are allowed.  All checked
    before any CUDA call."""
    p = ctypes.c_void_p(256)
    big = ctypes.c_size_t(1 << 40)
    fwd = lambda v: lib.attn_fwd_varlen(ctypes.byref(v), None, None, ctypes.c_float(0.1), p, p, p, p, p, None,  # noqa: E731
                                        p, big, None)
    assert fwd(_varlen([1, 3], [0, 3])) == bnd.ATTN_ERR_SHAPE          # cu[0] != 0
    assert fwd(_varlen([0, 5, 3], [0, 5, 6])) == bnd.ATTN_ERR_SHAPE    # decreasing
    assert fwd(_varlen([0, 3], [0, 0])) == bnd.ATTN_ERR_EMPTY_ROW      # queries, no keys
    assert fwd(_varlen([0, 4], [0, 3], causal=1)) == bnd.ATTN_ERR_EMPTY_ROW
    assert fwd(_varlen([0, 3], [0, 3], causal=2)) == bnd.ATTN_ERR_SHAPE
    assert fwd(_varlen([0, 3], [0, 3], Hq=3)) == bnd.ATTN_ERR_SHAPE
    assert fwd(_varlen([0, 3], [0, 3], d_h=96, d_v=96)) == bnd.ATTN_ERR_UNSUPPORTED
    assert fwd(_varlen([0, 3], [0, 3], B=0)) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_fwd_varlen(None, None, None, ctypes.c_float(0.1), p, p, p, p, p, None, p, big, None) == bnd.ATTN_ERR_NULL
    assert lib.attn_fwd_varlen(ctypes.byref(_varlen([0, 3], [0, 3])), None, None, ctypes.c_float(0.0), p, p, p, p, p, None,
                               p, big, None) == bnd.ATTN_ERR_SCALE
    assert lib.attn_fwd_varlen(ctypes.byref(_varlen([0, 3], [0, 3])), None, None, ctypes.c_float(0.1), p, p, p,
                               ctypes.c_void_p(0x1008), p, None, p, big, None) == bnd.ATTN_ERR_ALIGN
    # the forward workspace: present, aligned, large enough
    v3 = _varlen([0, 3, 200], [0, 3, 300])
    need = lib.attn_fwd_varlen_workspace_bytes(ctypes.byref(v3), None)
    r256 = lambda x: ((x + 255) // 256) * 256  # noqa: E731
    assert need == r256(2 * 2 * 3 * 128 * 128 * 2) + r256(2 * 2 * 3 * 4)   # B Hkv ceil(297/128) tiles
    assert lib.attn_fwd_varlen(ctypes.byref(v3), None, None, ctypes.c_float(0.1), p, p, p, p, p, None, None,
                               ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_fwd_varlen(ctypes.byref(v3), None, None, ctypes.c_float(0.1), p, p, p, p, p, None, p,
                               ctypes.c_size_t(need - 1), None) == bnd.ATTN_ERR_WORKSPACE
    # no query rows at all: nothing to compute, OK without touching the GPU
    assert fwd(_varlen([0, 0, 0], [0, 4, 9])) == bnd.ATTN_OK


def test_varlen_workspace_and_pairs(lib):
    cq, ck = [0, 100, 100, 357], [0, 150, 170, 600]
    v = _varlen(cq, ck, causal=1, Hq=4, Hkv=2, d_h=128, d_v=64)
    need = lib.attn_bwd_varlen_workspace_bytes(ctypes.byref(v), None)
    rows = cq[-1] * 4
    nqt = (257 + 127) // 128
    r256 = lambda x: ((x + 255) // 256) * 256  # noqa: E731
    assert need == (r256(rows * 4) + r256(3 * 4 * nqt * 16) + r256(3 * 2 * 8) + 256 + r256(rows * 128 * 4)
                    + r256(rows * 128 * 2) + r256(rows * 64 * 2) + r256(ck[-1] * 2 * (128 + 64) * 4))
    p = ctypes.c_void_p(512)
    args = [ctypes.byref(v), None, None, ctypes.c_float(0.1)] + [p] * 10
    assert lib.attn_bwd_varlen(*args, None, ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_varlen(*args, ctypes.c_void_p(512 + 16), ctypes.c_size_t(need), None) == bnd.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_varlen(*args, p, ctypes.c_size_t(need - 1), None) == bnd.ATTN_ERR_WORKSPACE
    # visible pairs against a brute-force count of the per-sequence masks
    brute = 0
    for b in range(3):
        lq, lk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        for i in range(lq):
            brute += sum(1 for j in range(lk) if j <= i + lk - lq)
    assert lib.attn_varlen_visible_pairs(ctypes.byref(v)) == brute * 4
    v2 = _varlen(cq, ck, causal=0)
    assert lib.attn_varlen_visible_pairs(ctypes.byref(v2)) == sum(
        (cq[b + 1] - cq[b]) * (ck[b + 1] - ck[b]) for b in range(3)) * 4


def test_proj_checks(lib):
    """Projection entry points: widths must be multiples of 8 (16-byte rows),
    1..3 sources for the input gradient; all checked before any CUDA call."""
    p = ctypes.c_void_p(256)
    assert lib.attn_proj_fwd(100, 60, 64, p, p, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_proj_fwd(100, 64, 60, p, p, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_proj_fwd(0, 64, 64, p, p, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_proj_fwd(100, 64, 64, None, p, p, None) == bnd.ATTN_ERR_NULL
    assert lib.attn_proj_fwd(100, 64, 64, p, ctypes.c_void_p(0x1008), p, None) == bnd.ATTN_ERR_ALIGN
    assert lib.attn_proj_bwd_weight(100, 64, 12, p, p, p, None) == bnd.ATTN_ERR_SHAPE
    n = (ctypes.c_int32 * 4)(64, 64, 64, 64)
    ptrs = (ctypes.c_void_p * 4)(256, 256, 256, 256)
    assert lib.attn_proj_bwd_input(100, 64, 4, n, ptrs, ptrs, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_proj_bwd_input(100, 64, 0, n, ptrs, ptrs, p, None) == bnd.ATTN_ERR_SHAPE
    n2 = (ctypes.c_int32 * 2)(64, 20)
    assert lib.attn_proj_bwd_input(100, 64, 2, n2, ptrs, ptrs, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_proj_bwd_input(100, 64, 2, None, ptrs, ptrs, p, None) == bnd.ATTN_ERR_NULL


def test_rope_checks(lib):
    p = ctypes.c_void_p(256)
    f = ctypes.c_float
    assert lib.attn_rope(10, 2, 12, f(10000.0), p, 0, p, p, None) == bnd.ATTN_ERR_SHAPE    # d % 8
    assert lib.attn_rope(10, 2, 256, f(10000.0), p, 0, p, p, None) == bnd.ATTN_ERR_SHAPE   # d > 128
    assert lib.attn_rope(10, 2, 64, f(10000.0), p, 2, p, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_rope(0, 2, 64, f(10000.0), p, 0, p, p, None) == bnd.ATTN_ERR_SHAPE
    assert lib.attn_rope(10, 2, 64, f(1.0), p, 0, p, p, None) == bnd.ATTN_ERR_SCALE
    assert lib.attn_rope(10, 2, 64, f(float("nan")), p, 0, p, p, None) == bnd.ATTN_ERR_SCALE
    assert lib.attn_rope(10, 2, 64, f(10000.0), None, 0, p, p, None) == bnd.ATTN_ERR_NULL
    assert lib.attn_rope(10, 2, 64, f(10000.0), p, 0, ctypes.c_void_p(0x1008), p, None) == bnd.ATTN_ERR_ALIGN


def test_rope_qk_checks(lib):
    p = ctypes.c_void_p(256)
    f = ctypes.c_float
    ok = dict(tokens=10, hq=4, hk=2, d=64, base=f(10000.0), pos=p, inv=0, xq=p, yq=p, xk=p, yk=p)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.attn_rope_qk(a["tokens"], a["hq"], a["hk"], a["d"], a["base"], a["pos"], a["inv"],
                                a["xq"], a["yq"], a["xk"], a["yk"], None)

    assert call(hk=0) == bnd.ATTN_ERR_SHAPE
    assert call(hq=-1) == bnd.ATTN_ERR_SHAPE
    assert call(d=12) == bnd.ATTN_ERR_SHAPE
    assert call(d=256) == bnd.ATTN_ERR_SHAPE
    assert call(tokens=0) == bnd.ATTN_ERR_SHAPE
    assert call(inv=2) == bnd.ATTN_ERR_SHAPE
    assert call(base=f(0.5)) == bnd.ATTN_ERR_SCALE
    assert call(pos=None) == bnd.ATTN_ERR_NULL
    assert call(yk=None) == bnd.ATTN_ERR_NULL
    assert call(xk=ctypes.c_void_p(0x1008)) == bnd.ATTN_ERR_ALIGN


def _strides(**kw):
    st = bnd.AttnStrides()
    for name, (row, head) in kw.items():
        setattr(st, name, bnd.AttnTensorStrides(row, head))
    return st


def test_strides_validated(lib):
    """attn_strides: element strides that are multiples of 8 (16-byte rows for
    the tensor-memory copies) and at least d; {0, 0} is the contiguous
    default.  Checked before any CUDA call."""
    s = _shape()
    bad_align = _strides(q=(136, 100 * 136 + 4))
    assert _call_fwd(lib, s, _mask(), strides=ctypes.byref(bad_align)) == bnd.ATTN_ERR_ALIGN
    assert _call_fwd(lib, s, _mask(), strides=ctypes.byref(_strides(k=(12, 1200)))) == bnd.ATTN_ERR_ALIGN
    assert _call_fwd(lib, s, _mask(), strides=ctypes.byref(_strides(v=(64, 64 * 100)))) == bnd.ATTN_ERR_SHAPE
    assert _call_fwd(lib, s, _mask(), strides=ctypes.byref(_strides(o=(128, 64)))) == bnd.ATTN_ERR_SHAPE
    assert _call_fwd(lib, s, _mask(), strides=ctypes.byref(_strides(q=(128, 1 << 40)))) == bnd.ATTN_ERR_SHAPE
    # a bad stride of a tensor the forward does not take is still a bad argument
    assert _call_fwd(lib, s, _mask(), strides=ctypes.byref(_strides(dk=(8, 8)))) == bnd.ATTN_ERR_SHAPE
    v = _varlen([0, 100], [0, 100])
    p = ctypes.c_void_p(256)
    rc = lib.attn_fwd_varlen(ctypes.byref(v), ctypes.byref(_strides(q=(3 * 128 + 4, 128))), None,
                             ctypes.c_float(0.1), p, p, p, p, p, None, p, ctypes.c_size_t(1 << 40), None)
    assert rc == bnd.ATTN_ERR_ALIGN


def test_binding_reads_view_strides():
    """The binding passes a view's element strides: Q, K, V sliced out of one
    fused [T, (Hq + 2 Hkv) d] projection output (packed), and head-major
    views with a padded row (padded); contiguous tensors give NULL."""
    T, Hq, Hkv, d = 10, 4, 2, 128
    qkv = torch.empty((T, (Hq + 2 * Hkv) * d), dtype=torch.bfloat16)
    Q = qkv[:, :Hq * d].view(T, Hq, d)
    K = qkv[:, Hq * d:(Hq + Hkv) * d].view(T, Hkv, d)
    V = qkv[:, (Hq + Hkv) * d:].view(T, Hkv, d)
    ref = bnd._strides_arg(True, q=Q, k=K, v=V).contents
    for t in (ref.q, ref.k, ref.v):
        assert (t.row, t.head) == ((Hq + 2 * Hkv) * d, d)
    assert (ref.o.row, ref.o.head) == (0, 0)
    assert bnd._strides_arg(True, q=Q.contiguous()) is None
    B, H, n = 2, 3, 50
    big = torch.empty((B, H, n, 192), dtype=torch.bfloat16)
    X = big[..., :128]
    pst = bnd._strides_arg(False, dO=X).contents
    assert (pst.dO.row, pst.dO.head) == (192, n * 192)
    # sequence-major [B, n, H, d] seen as [B, H, n, d]: head-major batch stride fails
    seq = torch.empty((B, n, H, 128), dtype=torch.bfloat16).transpose(1, 2)
    with pytest.raises(ValueError):
        bnd._strides_arg(False, q=seq)
    # ... but one batch element of it is a valid padded view
    one = torch.empty((1, n, H, 128), dtype=torch.bfloat16).transpose(1, 2)
    pst = bnd._strides_arg(False, q=one).contents
    assert (pst.q.row, pst.q.head) == (H * 128, 128)


def test_rotary_checks_and_workspace_sizes(lib):
    """attn_rotary: base finite and > 1, both position arrays present and
    4-byte aligned, the optional rotated-row buffers 16-byte aligned, all
    checked before any CUDA call; a workspace holds the rotated rows that
    have no caller buffer (the forward's queries and keys, the backward's
    keys)."""
    s = _shape(n_q=100, n_k=300)
    r256 = lambda x: ((x + 255) // 256) * 256  # noqa: E731
    rot = bnd.AttnRotary(10000.0, 256, 512)
    f0 = lib.attn_fwd_workspace_bytes(ctypes.byref(s), None)
    f1 = lib.attn_fwd_workspace_bytes(ctypes.byref(s), ctypes.byref(rot))
    assert f1 == f0 + r256(2 * 100 * 4 * 128 * 2) + r256(2 * 300 * 2 * 128 * 2)
    kept = bnd.AttnRotary(10000.0, 256, 512, 4096, 8192)
    assert lib.attn_fwd_workspace_bytes(ctypes.byref(s), ctypes.byref(kept)) == f0
    b0 = lib.attn_bwd_workspace_bytes(ctypes.byref(s), None)
    b1 = lib.attn_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(rot))
    assert b1 == b0 + r256(2 * 300 * 2 * 128 * 2)
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(kept)) == b0
    v = _varlen([0, 3, 200], [0, 3, 300])
    vf0 = lib.attn_fwd_varlen_workspace_bytes(ctypes.byref(v), None)
    vf1 = lib.attn_fwd_varlen_workspace_bytes(ctypes.byref(v), ctypes.byref(rot))
    assert vf1 == vf0 + r256(200 * 4 * 128 * 2) + r256(300 * 2 * 128 * 2)
    bad = [(bnd.AttnRotary(1.0, 256, 512), bnd.ATTN_ERR_SCALE), (bnd.AttnRotary(float("nan"), 256, 512),
                                                                   bnd.ATTN_ERR_SCALE),
           (bnd.AttnRotary(10000.0, None, 512), bnd.ATTN_ERR_NULL), (bnd.AttnRotary(10000.0, 256, None),
                                                                      bnd.ATTN_ERR_NULL),
           (bnd.AttnRotary(10000.0, 258, 512), bnd.ATTN_ERR_ALIGN),
           (bnd.AttnRotary(10000.0, 256, 512, 0x1008, None), bnd.ATTN_ERR_ALIGN)]
    p = ctypes.c_void_p(256)
    for r, code in bad:
        assert _call_fwd(lib, s, _mask(), rotary=ctypes.byref(r)) == code
        assert lib.attn_fwd_workspace_bytes(ctypes.byref(s), ctypes.byref(r)) == 0
        assert lib.attn_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(r)) == 0
        m = _mask()
        assert lib.attn_bwd(ctypes.byref(s), ctypes.byref(m), None, ctypes.byref(r), ctypes.c_float(0.1),
                            *([p] * 10), p, ctypes.c_size_t(1 << 40), None) == code
    # a workspace sized without the rotary is too small for a call with one
    m = _mask()
    assert lib.attn_bwd(ctypes.byref(s), ctypes.byref(m), None, ctypes.byref(rot), ctypes.c_float(0.1),
                        *([p] * 10), ctypes.c_void_p(512), ctypes.c_size_t(b0), None) == bnd.ATTN_ERR_WORKSPACE
    assert _call_fwd(lib, s, _mask(), ws=512, ws_bytes=f0, rotary=ctypes.byref(rot)) == bnd.ATTN_ERR_WORKSPACE
