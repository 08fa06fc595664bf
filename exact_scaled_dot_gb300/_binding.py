"""ctypes binding of the C ABI in include/attn.h.

Argument marshalling only: shapes, masks, pointers and the current torch
stream go in; every step of the computation runs in the CUDA library.  There
is no fallback: if the compiled library is missing, every call raises.

The prefill forward, the backward and its stages take strided views for Q,
K, V, O (with O_lo), dO and the gradients: any tensor whose innermost index
is contiguous, e.g. Q, K, V sliced out of one fused projection output, with
their element strides passed through attn_strides.  Padded [B, H, n, d]
views additionally need a batch stride of H times their head stride.  The
decode forward takes contiguous tensors only.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path
from typing import Optional, Sequence, Tuple, Union

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libesd_attn.so"

ATTN_OK = 0
ATTN_ERR_NULL = 1
ATTN_ERR_SHAPE = 2
ATTN_ERR_UNSUPPORTED = 3
ATTN_ERR_ALIGN = 4
ATTN_ERR_EMPTY_ROW = 5
ATTN_ERR_SCALE = 6
ATTN_ERR_WORKSPACE = 7
ATTN_ERR_CUDA = 8
ATTN_ERR_TIMEOUT = 9
ATTN_ERR_DEVICE = 10
ATTN_ERR_RANGE = 11
ATTN_MAX_BATCH = 512
ATTN_OFFSET_DEFAULT = -(2 ** 63)

# Every symbol include/attn.h declares.
EXPORTS = ("attn_fwd", "attn_fwd_workspace_bytes", "attn_fwd_varlen_workspace_bytes", "attn_fwd_decode", "attn_fwd_decode_workspace_bytes", "attn_bwd_workspace_bytes", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_main",
           "attn_bwd_finalize", "attn_visible_pairs", "attn_get_status", "attn_clear_status",
           "attn_selftest_wait_timeout", "attn_strerror", "attn_abi_version", "attn_bwd_noalloc",
           "attn_bwd_noalloc_max_scratch_bytes", "attn_varlen_visible_pairs", "attn_fwd_varlen",
           "attn_bwd_varlen_workspace_bytes", "attn_bwd_varlen", "attn_proj_fwd", "attn_proj_bwd_weight",
           "attn_proj_bwd_input", "attn_rope", "attn_rope_qk", "attn_bwd_head_split", "attn_bwd_persistent")


class AttnError(RuntimeError):
    """A non-zero status from the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {strerror(code)} (status {code})")


class AttnShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "Hq", "Hkv", "n_q", "n_k", "d_h", "d_v")]


class AttnMask(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("causal_offset", ctypes.c_int64), ("kv_len", ctypes.POINTER(ctypes.c_int32))]


class AttnTensorStrides(ctypes.Structure):
    _fields_ = [("row", ctypes.c_int64), ("head", ctypes.c_int64)]


class AttnStrides(ctypes.Structure):
    _fields_ = [(n, AttnTensorStrides) for n in ("q", "k", "v", "o", "dO", "dq", "dk", "dv")]


class AttnRotary(ctypes.Structure):
    _fields_ = [("base", ctypes.c_float), ("pos_q", ctypes.c_void_p), ("pos_k", ctypes.c_void_p),
                ("q_rot", ctypes.c_void_p), ("k_rot", ctypes.c_void_p)]


class AttnVarlen(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d_h", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)), ("cu_seqlens_k", ctypes.POINTER(ctypes.c_int32))]


_lib: Optional[ctypes.CDLL] = None
_vp = ctypes.c_void_p


def load(path: Optional[Path] = None) -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"CUDA library {p} not found; build it with exact_scaled_dot_gb300.build.build()")
    lib = ctypes.CDLL(str(p))
    S, M = ctypes.POINTER(AttnShape), ctypes.POINTER(AttnMask)
    ST = ctypes.POINTER(AttnStrides)
    RT = ctypes.POINTER(AttnRotary)
    f = ctypes.c_float
    lib.attn_fwd.argtypes = [S, M, ST, RT, f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_fwd_workspace_bytes.argtypes = [S, RT]
    lib.attn_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_decode.argtypes = [S, M, f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_fwd_decode_workspace_bytes.argtypes = [S, M]
    lib.attn_fwd_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd_workspace_bytes.argtypes = [S, RT]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd.argtypes = [S, M, ST, RT, f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                             _vp]
    lib.attn_bwd_preprocess.argtypes = [S, ST, RT, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_bwd_main.argtypes = [S, M, ST, RT, f, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp]
    lib.attn_bwd_finalize.argtypes = [S, ST, RT, f, _vp, ctypes.c_size_t, _vp, _vp]
    lib.attn_visible_pairs.argtypes = [S, M]
    lib.attn_bwd_head_split.argtypes = [S, M]
    lib.attn_bwd_head_split.restype = ctypes.c_int
    lib.attn_bwd_persistent.argtypes = [S, M, RT]
    lib.attn_bwd_persistent.restype = ctypes.c_int
    lib.attn_visible_pairs.restype = ctypes.c_int64
    lib.attn_get_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.attn_clear_status.argtypes = []
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp]
    lib.attn_strerror.argtypes = [ctypes.c_int]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_abi_version.restype = ctypes.c_int
    lib.attn_bwd_noalloc.argtypes = [S, M, ST, RT, f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.attn_bwd_noalloc.restype = ctypes.c_int
    lib.attn_bwd_noalloc_max_scratch_bytes.argtypes = []
    lib.attn_bwd_noalloc_max_scratch_bytes.restype = ctypes.c_size_t
    VL = ctypes.POINTER(AttnVarlen)
    lib.attn_varlen_visible_pairs.argtypes = [VL]
    lib.attn_varlen_visible_pairs.restype = ctypes.c_int64
    lib.attn_fwd_varlen.argtypes = [VL, ST, RT, f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_fwd_varlen_workspace_bytes.argtypes = [VL, RT]
    lib.attn_fwd_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd_varlen_workspace_bytes.argtypes = [VL, RT]
    lib.attn_bwd_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd_varlen.argtypes = [VL, ST, RT, f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                    _vp]
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    lib.attn_proj_fwd.argtypes = [i64, i32, i32, _vp, _vp, _vp, _vp]
    lib.attn_proj_bwd_weight.argtypes = [i64, i32, i32, _vp, _vp, _vp, _vp]
    lib.attn_proj_bwd_input.argtypes = [i64, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(_vp),
                                        ctypes.POINTER(_vp), _vp, _vp]
    lib.attn_rope.argtypes = [i64, i32, i32, f, _vp, i32, _vp, _vp, _vp]
    lib.attn_rope_qk.argtypes = [i64, i32, i32, i32, f, _vp, i32, _vp, _vp, _vp, _vp, _vp]
    for name in ("attn_fwd", "attn_fwd_decode", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_main", "attn_bwd_finalize",
                 "attn_get_status", "attn_clear_status", "attn_selftest_wait_timeout", "attn_fwd_varlen",
                 "attn_bwd_varlen", "attn_proj_fwd", "attn_proj_bwd_weight", "attn_proj_bwd_input",
                 "attn_rope", "attn_rope_qk"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().attn_strerror(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(rc: int, where: str) -> None:
    if rc != ATTN_OK:
        raise AttnError(rc, where)


# ---------------------------------------------------------------------------
# Marshalling helpers
# ---------------------------------------------------------------------------
def make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v) -> AttnShape:
    return AttnShape(int(B), int(Hq), int(Hkv), int(n_q), int(n_k), int(d_h), int(d_v))


class _MaskArg:
    """Holds an AttnMask and keeps its host kv_len array alive."""

    def __init__(self, causal: bool, causal_offset: Optional[int], kv_len):
        self._keep = None
        kv = ctypes.POINTER(ctypes.c_int32)()
        if kv_len is not None:
            if isinstance(kv_len, torch.Tensor):
                vals = [int(x) for x in kv_len.detach().cpu().reshape(-1).tolist()]
            else:
                vals = [int(x) for x in kv_len]
            arr = (ctypes.c_int32 * max(1, len(vals)))(*vals)
            self._keep = arr
            kv = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        off = ATTN_OFFSET_DEFAULT if causal_offset is None else int(causal_offset)
        self.mask = AttnMask(1 if causal else 0, 0, off, kv)


class Rotary:
    """Rotary position embedding fused into the attention calls (attn_rotary):
    pos_q, pos_k are int32 device tensors with the position of every query /
    key row ([B, n_q] and [B, n_k] for the padded calls, [T_q] and [T_k] for
    the packed ones); base sets the frequencies base^(-2k/d_h).

    q_rot, k_rot (optional): bf16 tensors shaped like contiguous Q and K
    that the forward fills with the rotated rows and the backward then reads
    instead of rotating again (keep them between the two calls)."""

    def __init__(self, pos_q: torch.Tensor, pos_k: torch.Tensor, base: float = 10000.0,
                 q_rot: Optional[torch.Tensor] = None, k_rot: Optional[torch.Tensor] = None):
        self.pos_q, self.pos_k, self.base = pos_q, pos_k, float(base)
        self.q_rot, self.k_rot = q_rot, k_rot

    def check(self, q_shape, k_shape, device, Q=None, K=None):
        for t, name, shp in ((self.pos_q, "pos_q", q_shape), (self.pos_k, "pos_k", k_shape)):
            _check_tensor(t, name, torch.int32, shp, device)
        for t, name, ref in ((self.q_rot, "q_rot", Q), (self.k_rot, "k_rot", K)):
            if t is not None and ref is not None:
                _check_tensor(t, name, torch.bfloat16, tuple(ref.shape), device)

    def arg(self):
        r = AttnRotary(self.base, self.pos_q.data_ptr(), self.pos_k.data_ptr(),
                       None if self.q_rot is None else self.q_rot.data_ptr(),
                       None if self.k_rot is None else self.k_rot.data_ptr())
        return ctypes.pointer(r)


# Stands in for a Rotary without caller buffers where only its presence
# matters (workspace sizes).
_SIZE_ONLY_ROTARY = AttnRotary(10000.0, 4, 4, None, None)


def _rot_size_arg(rotary):
    if isinstance(rotary, Rotary):
        return rotary.arg()
    return ctypes.pointer(_SIZE_ONLY_ROTARY) if rotary else None


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensor(t: torch.Tensor, name: str, dtype, shape: Tuple[int, ...], device, strided: bool = False):
    """strided: the tensor may be a view whose innermost index is contiguous
    (its other strides go to the library through attn_strides)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or (device is not None and t.device != device):
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if strided:
        if t.shape[-1] > 1 and t.stride(-1) != 1:
            raise ValueError(f"{name} must have a contiguous innermost dimension")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _padded_strides(t: torch.Tensor, name: str) -> Tuple[int, int]:
    """(row, head) element strides of a [B, H, n, d] view; its batch stride
    must be H times its head stride (size-1 dimensions are free)."""
    B, H, n, d = (int(x) for x in t.shape)
    sB, sH, sR = (int(x) for x in t.stride()[:3])
    row = sR if n > 1 else d
    head = sH if H > 1 else (sB if B > 1 else n * row)
    if B > 1 and sB != H * head:
        raise ValueError(f"{name}: the batch stride must be H times the head stride (use the packed entry points "
                         f"for sequence-major tensors)")
    return row, head


def _packed_strides(t: torch.Tensor) -> Tuple[int, int]:
    """(row = token, head) element strides of a [T, H, d] view."""
    T, H, d = (int(x) for x in t.shape)
    return (int(t.stride(0)) if T > 1 else H * d), (int(t.stride(1)) if H > 1 else d)


def _strides_arg(packed: bool, **tensors):
    """attn_strides for the given tensors (q=, k=, ... by ABI field name), or
    None when every one of them is contiguous.  Missing tensors keep the
    contiguous default ({0, 0})."""
    st = AttnStrides()
    any_strided = False
    for field, t in tensors.items():
        if t is None:
            continue
        if t.is_contiguous():
            continue
        row, head = _packed_strides(t) if packed else _padded_strides(t, field)
        setattr(st, field, AttnTensorStrides(row, head))
        any_strided = True
    return ctypes.pointer(st) if any_strided else None


def _check_o_lo(O_lo, O, shape, dev):
    _check_tensor(O_lo, "O_lo", torch.bfloat16, shape, dev, strided=True)
    if O_lo.stride() != O.stride():
        raise ValueError("O_lo must have the same strides as O")


def _like_o(O):
    """A residual tensor with O's strides (O may be a view into a larger buffer)."""
    return torch.empty_strided(O.shape, O.stride(), dtype=O.dtype, device=O.device)


def _qkv_shape(Q, K, V):
    if Q.dim() != 4 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("Q, K, V must be 4-D [B, H, n, d]")
    B, Hq, n_q, d_h = Q.shape
    _, Hkv, n_k, _ = K.shape
    d_v = V.shape[3]
    return int(B), int(Hq), int(Hkv), int(n_q), int(n_k), int(d_h), int(d_v)


def _check_qkv(Q, K, V, strided: bool = True):
    B, Hq, Hkv, n_q, n_k, d_h, d_v = _qkv_shape(Q, K, V)
    dev = Q.device
    _check_tensor(Q, "Q", torch.bfloat16, (B, Hq, n_q, d_h), dev, strided=strided)
    _check_tensor(K, "K", torch.bfloat16, (B, Hkv, n_k, d_h), dev, strided=strided)
    _check_tensor(V, "V", torch.bfloat16, (B, Hkv, n_k, d_v), dev, strided=strided)
    return (B, Hq, Hkv, n_q, n_k, d_h, d_v), dev


# ---------------------------------------------------------------------------
# Public functions (names follow the C ABI)
# ---------------------------------------------------------------------------
def attn_fwd_workspace_bytes(B, Hq, Hkv, n_q, n_k, d_h, d_v, *, rotary=None) -> int:
    """rotary: a Rotary (or True) when the forward will rotate; only its presence matters."""
    shape = make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v)
    return int(load().attn_fwd_workspace_bytes(ctypes.byref(shape), _rot_size_arg(rotary)))


def attn_fwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False,
             causal_offset: Optional[int] = None, kv_len=None, scale: Optional[float] = None,
             O: Optional[torch.Tensor] = None, LSE: Optional[torch.Tensor] = None,
             O_lo: Optional[torch.Tensor] = None, residual: bool = True, rotary: Optional[Rotary] = None,
             workspace=None, stream=None):
    """Forward pass: returns (O [B,Hq,n_q,d_v] bf16, LSE [B,Hq,n_q] fp32, O_lo).

    rotary: a Rotary to rotate Q and K by their positions inside the call.

    O_lo is the bf16 rounding residual of O (O + O_lo ~ the fp32 result), which
    the backward requires for its row term; it is None when ``residual`` is
    False and no O_lo tensor is given.  ``workspace`` (uint8, at least
    attn_fwd_workspace_bytes) is created here by torch when not given."""
    dims, dev = _check_qkv(Q, K, V)
    B, Hq, Hkv, n_q, n_k, d_h, d_v = dims
    scale = 1.0 / math.sqrt(d_h) if scale is None else float(scale)
    if O is None:
        O = torch.empty((B, Hq, n_q, d_v), dtype=torch.bfloat16, device=dev)
    if LSE is None:
        LSE = torch.empty((B, Hq, n_q), dtype=torch.float32, device=dev)
    _check_tensor(O, "O", torch.bfloat16, (B, Hq, n_q, d_v), dev, strided=True)
    if O_lo is None and residual:
        O_lo = _like_o(O)
    _check_tensor(LSE, "LSE", torch.float32, (B, Hq, n_q), dev)
    if O_lo is not None:
        _check_o_lo(O_lo, O, (B, Hq, n_q, d_v), dev)
    shape = make_shape(*dims)
    m = _MaskArg(causal, causal_offset, kv_len)
    if rotary is not None:
        rotary.check((B, n_q), (B, n_k), dev, Q, K)
    if workspace is None:
        need = int(load().attn_fwd_workspace_bytes(ctypes.byref(shape), _rot_size_arg(rotary)))
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    st = _strides_arg(False, q=Q, k=K, v=V, o=O)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_fwd(ctypes.byref(shape), ctypes.byref(m.mask), st, rt, ctypes.c_float(scale), _ptr(Q), _ptr(K),
                         _ptr(V), _ptr(O), _ptr(LSE), _ptr(O_lo), *_ws(workspace), _stream(dev, stream))
    _check(rc, "attn_fwd")
    return O, LSE, O_lo


def attn_fwd_decode_workspace_bytes(B, Hq, Hkv, n_q, n_k, d_h, d_v, *, causal: bool = False,
                                    causal_offset: Optional[int] = None, kv_len=None) -> int:
    shape = make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v)
    m = _MaskArg(causal, causal_offset, kv_len)
    return int(load().attn_fwd_decode_workspace_bytes(ctypes.byref(shape), ctypes.byref(m.mask)))


def attn_fwd_decode(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False,
                    causal_offset: Optional[int] = None, kv_len=None, scale: Optional[float] = None,
                    O: Optional[torch.Tensor] = None, LSE: Optional[torch.Tensor] = None,
                    O_lo: Optional[torch.Tensor] = None, residual: bool = True, workspace=None, stream=None):
    """Forward for short query blocks (n_q <= 128) over a long key cache: the
    same outputs as attn_fwd, with the query heads of a KV head packed into
    one tile and the key range split across CTAs (merged by log-sum-exp)."""
    dims, dev = _check_qkv(Q, K, V, strided=False)
    B, Hq, Hkv, n_q, n_k, d_h, d_v = dims
    scale = 1.0 / math.sqrt(d_h) if scale is None else float(scale)
    if O is None:
        O = torch.empty((B, Hq, n_q, d_v), dtype=torch.bfloat16, device=dev)
    if LSE is None:
        LSE = torch.empty((B, Hq, n_q), dtype=torch.float32, device=dev)
    if O_lo is None and residual:
        O_lo = torch.empty((B, Hq, n_q, d_v), dtype=torch.bfloat16, device=dev)
    _check_tensor(O, "O", torch.bfloat16, (B, Hq, n_q, d_v), dev)
    _check_tensor(LSE, "LSE", torch.float32, (B, Hq, n_q), dev)
    if O_lo is not None:
        _check_tensor(O_lo, "O_lo", torch.bfloat16, (B, Hq, n_q, d_v), dev)
    shape = make_shape(*dims)
    m = _MaskArg(causal, causal_offset, kv_len)
    need = int(load().attn_fwd_decode_workspace_bytes(ctypes.byref(shape), ctypes.byref(m.mask)))
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ws_ptr, ws_bytes = (_ws(workspace) if workspace is not None else (None, ctypes.c_size_t(0)))
    rc = load().attn_fwd_decode(ctypes.byref(shape), ctypes.byref(m.mask), ctypes.c_float(scale), _ptr(Q), _ptr(K),
                                _ptr(V), _ptr(O), _ptr(LSE), _ptr(O_lo), ws_ptr, ws_bytes, _stream(dev, stream))
    _check(rc, "attn_fwd_decode")
    return O, LSE, O_lo


def attn_bwd_workspace_bytes(B, Hq, Hkv, n_q, n_k, d_h, d_v, *, rotary=None) -> int:
    shape = make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v)
    return int(load().attn_bwd_workspace_bytes(ctypes.byref(shape), _rot_size_arg(rotary)))


def attn_bwd(Q, K, V, O, dO, LSE, *, O_lo=None, causal: bool = False, causal_offset: Optional[int] = None,
             kv_len=None, scale: Optional[float] = None, dQ=None, dK=None, dV=None, rotary: Optional[Rotary] = None,
             workspace=None, stream=None):
    """Backward pass: returns (dQ, dK, dV) in bf16; dK, dV summed over each KV head's group.

    O_lo (the forward's residual) is required; without it the library
    returns ATTN_ERR_NULL, raised here as AttnError."""
    dims, dev = _check_qkv(Q, K, V)
    B, Hq, Hkv, n_q, n_k, d_h, d_v = dims
    scale = 1.0 / math.sqrt(d_h) if scale is None else float(scale)
    _check_tensor(O, "O", torch.bfloat16, (B, Hq, n_q, d_v), dev, strided=True)
    _check_tensor(dO, "dO", torch.bfloat16, (B, Hq, n_q, d_v), dev, strided=True)
    _check_tensor(LSE, "LSE", torch.float32, (B, Hq, n_q), dev)
    if O_lo is not None:
        _check_o_lo(O_lo, O, (B, Hq, n_q, d_v), dev)
    if dQ is None:
        dQ = torch.empty_like(Q)
    if dK is None:
        dK = torch.empty_like(K)
    if dV is None:
        dV = torch.empty_like(V)
    _check_tensor(dQ, "dQ", torch.bfloat16, tuple(Q.shape), dev, strided=True)
    _check_tensor(dK, "dK", torch.bfloat16, tuple(K.shape), dev, strided=True)
    _check_tensor(dV, "dV", torch.bfloat16, tuple(V.shape), dev, strided=True)
    if rotary is not None:
        rotary.check((B, n_q), (B, n_k), dev, Q, K)
    need = attn_bwd_workspace_bytes(*dims, rotary=rotary)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must hold at least {need} bytes")
    shape = make_shape(*dims)
    m = _MaskArg(causal, causal_offset, kv_len)
    st = _strides_arg(False, q=Q, k=K, v=V, o=O, dO=dO, dq=dQ, dk=dK, dv=dV)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_bwd(ctypes.byref(shape), ctypes.byref(m.mask), st, rt, ctypes.c_float(scale), _ptr(Q), _ptr(K),
                         _ptr(V), _ptr(O), _ptr(O_lo), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV),
                         _ptr(workspace),
                         ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(dev, stream))
    _check(rc, "attn_bwd")
    return dQ, dK, dV


def _ws(workspace):
    return _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size())


def attn_bwd_preprocess(Q, O, dO, workspace, *, shape: AttnShape, O_lo=None, rotary: Optional[Rotary] = None,
                        stream=None):
    """Stage 1 of the backward (row terms, tile bounds, zeroed dQ accumulator, fp16 copies of Q and dO)."""
    if O_lo is not None and O_lo.stride() != O.stride():
        raise ValueError("O_lo must have the same strides as O")
    st = _strides_arg(False, q=Q, o=O, dO=dO)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_bwd_preprocess(ctypes.byref(shape), st, rt, _ptr(Q), _ptr(O), _ptr(O_lo), _ptr(dO),
                                    *_ws(workspace), _stream(O.device, stream))
    _check(rc, "attn_bwd_preprocess")


def attn_bwd_main(K, V, LSE, workspace, dK, dV, *, shape: AttnShape, causal=False, causal_offset=None,
                  kv_len=None, scale: Optional[float] = None, rotary: Optional[Rotary] = None, stream=None):
    """Stage 2 of the backward (the key-tile-stationary main kernel; Q and dO
    come from the fp16 copies stage 1 left in the workspace)."""
    scale = 1.0 / math.sqrt(shape.d_h) if scale is None else float(scale)
    m = _MaskArg(causal, causal_offset, kv_len)
    st = _strides_arg(False, k=K, v=V, dk=dK, dv=dV)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_bwd_main(ctypes.byref(shape), ctypes.byref(m.mask), st, rt, ctypes.c_float(scale), _ptr(K),
                              _ptr(V), _ptr(LSE), *_ws(workspace), _ptr(dK), _ptr(dV), _stream(K.device, stream))
    _check(rc, "attn_bwd_main")


def attn_bwd_finalize(workspace, dQ, *, shape: AttnShape, scale: Optional[float] = None,
                      rotary: Optional[Rotary] = None, stream=None):
    """Stage 3 of the backward (dQ = scale * accumulator in bf16)."""
    scale = 1.0 / math.sqrt(shape.d_h) if scale is None else float(scale)
    st = _strides_arg(False, dq=dQ)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_bwd_finalize(ctypes.byref(shape), st, rt, ctypes.c_float(scale), *_ws(workspace), _ptr(dQ),
                                  _stream(dQ.device, stream))
    _check(rc, "attn_bwd_finalize")


def attn_visible_pairs(B, Hq, Hkv, n_q, n_k, d_h, d_v, *, causal=False, causal_offset=None, kv_len=None) -> int:
    """Visible (i, j) pairs over batch and query heads (closed form; -1 if invalid)."""
    shape = make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v)
    m = _MaskArg(causal, causal_offset, kv_len)
    return int(load().attn_visible_pairs(ctypes.byref(shape), ctypes.byref(m.mask)))


def attn_bwd_head_split(B, Hq, Hkv, n_q, n_k, d_h, d_v, *, causal=False, causal_offset=None, kv_len=None) -> int:
    """How the backward main kernel splits each KV head's query heads on the current device (1 = not)."""
    shape = make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v)
    m = _MaskArg(causal, causal_offset, kv_len)
    rc = int(load().attn_bwd_head_split(ctypes.byref(shape), ctypes.byref(m.mask)))
    if rc < 0:
        raise AttnError(-rc, "attn_bwd_head_split")
    return rc


def attn_bwd_persistent(B, Hq, Hkv, n_q, n_k, d_h, d_v, *, causal=False, causal_offset=None, kv_len=None,
                        rotary=None) -> bool:
    """Whether the backward main kernel runs its persistent schedule for this problem on the current device."""
    shape = make_shape(B, Hq, Hkv, n_q, n_k, d_h, d_v)
    m = _MaskArg(causal, causal_offset, kv_len)
    rc = int(load().attn_bwd_persistent(ctypes.byref(shape), ctypes.byref(m.mask), _rot_size_arg(rotary)))
    if rc < 0:
        raise AttnError(-rc, "attn_bwd_persistent")
    return rc == 1


def attn_get_status() -> int:
    v = ctypes.c_int(0)
    _check(load().attn_get_status(ctypes.byref(v)), "attn_get_status")
    return int(v.value)


def attn_clear_status() -> None:
    _check(load().attn_clear_status(), "attn_clear_status")


def attn_selftest_wait_timeout(limit_ns: int, stream=None, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(load().attn_selftest_wait_timeout(ctypes.c_uint64(int(limit_ns)), _stream(dev, stream)),
           "attn_selftest_wait_timeout")


def attn_bwd_noalloc(Q, K, V, O, dO, LSE, *, O_lo=None, causal: bool = False,
                     causal_offset: Optional[int] = None, kv_len=None, scale: Optional[float] = None,
                     dQ=None, dK=None, dV=None, rotary: Optional[Rotary] = None, stream=None):
    """Backward pass that allocates no device memory in the library.

    For callers that cannot allocate where they run the backward (memory owned
    by a fixed arena or another runtime, or loops that cannot afford the
    device-wide synchronisation of an allocation): the scratch comes from a
    static buffer inside the library instead of a caller workspace.  Outputs
    passed in (dQ, dK, dV) are filled; missing ones are created here by torch,
    which is the caller's allocation, not the library's.  Problems needing more
    than attn_bwd_noalloc_max_scratch_bytes() of scratch raise AttnError
    (ATTN_ERR_WORKSPACE).  Calls that overlap on the GPU share the buffer and
    race; serialise them."""
    dims, dev = _check_qkv(Q, K, V)
    B, Hq, Hkv, n_q, n_k, d_h, d_v = dims
    scale = 1.0 / math.sqrt(d_h) if scale is None else float(scale)
    _check_tensor(O, "O", torch.bfloat16, (B, Hq, n_q, d_v), dev, strided=True)
    _check_tensor(dO, "dO", torch.bfloat16, (B, Hq, n_q, d_v), dev, strided=True)
    _check_tensor(LSE, "LSE", torch.float32, (B, Hq, n_q), dev)
    if O_lo is not None:
        _check_o_lo(O_lo, O, (B, Hq, n_q, d_v), dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check_tensor(dQ, "dQ", torch.bfloat16, tuple(Q.shape), dev, strided=True)
    _check_tensor(dK, "dK", torch.bfloat16, tuple(K.shape), dev, strided=True)
    _check_tensor(dV, "dV", torch.bfloat16, tuple(V.shape), dev, strided=True)
    shape = make_shape(*dims)
    m = _MaskArg(causal, causal_offset, kv_len)
    st = _strides_arg(False, q=Q, k=K, v=V, o=O, dO=dO, dq=dQ, dk=dK, dv=dV)
    if rotary is not None:
        rotary.check((B, n_q), (B, n_k), dev, Q, K)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_bwd_noalloc(ctypes.byref(shape), ctypes.byref(m.mask), st, rt, ctypes.c_float(scale), _ptr(Q),
                                 _ptr(K), _ptr(V), _ptr(O), _ptr(O_lo), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK),
                                 _ptr(dV), _stream(dev, stream))
    _check(rc, "attn_bwd_noalloc")
    return dQ, dK, dV


def attn_bwd_noalloc_max_scratch_bytes() -> int:
    return int(load().attn_bwd_noalloc_max_scratch_bytes())


def attn_abi_version() -> int:
    return int(load().attn_abi_version())


# ---------------------------------------------------------------------------
# Packed variable-length sequences (token-major tensors, per-sequence lengths)
# ---------------------------------------------------------------------------
class _VarlenArg:
    """ctypes description of packed sequences; keeps the host offset arrays alive."""

    def __init__(self, Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, causal):
        cq = [int(x) for x in (cu_seqlens_q.tolist() if hasattr(cu_seqlens_q, "tolist") else cu_seqlens_q)]
        ck = [int(x) for x in (cu_seqlens_k.tolist() if hasattr(cu_seqlens_k, "tolist") else cu_seqlens_k)]
        if len(cq) != len(ck) or len(cq) < 2:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 >= 2 entries")
        self._q = (ctypes.c_int32 * len(cq))(*cq)
        self._k = (ctypes.c_int32 * len(ck))(*ck)
        self.B = len(cq) - 1
        self.total_q, self.total_k = cq[-1], ck[-1]
        self.v = AttnVarlen(self.B, int(Hq), int(Hkv), int(d_h), int(d_v), 1 if causal else 0,
                            ctypes.cast(self._q, ctypes.POINTER(ctypes.c_int32)),
                            ctypes.cast(self._k, ctypes.POINTER(ctypes.c_int32)))


def _varlen_dims(Q, K, V):
    if Q.dim() != 3 or K.dim() != 3 or V.dim() != 3:
        raise ValueError("packed Q, K, V must be 3-D [tokens, heads, d]")
    Tq, Hq, d_h = (int(x) for x in Q.shape)
    Tk, Hkv, _ = (int(x) for x in K.shape)
    d_v = int(V.shape[2])
    dev = Q.device
    _check_tensor(Q, "Q", torch.bfloat16, (Tq, Hq, d_h), dev, strided=True)
    _check_tensor(K, "K", torch.bfloat16, (Tk, Hkv, d_h), dev, strided=True)
    _check_tensor(V, "V", torch.bfloat16, (Tk, Hkv, d_v), dev, strided=True)
    return (Tq, Tk, Hq, Hkv, d_h, d_v), dev


def attn_varlen_visible_pairs(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, *, causal=False) -> int:
    a = _VarlenArg(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, causal)
    return int(load().attn_varlen_visible_pairs(ctypes.byref(a.v)))


def attn_fwd_varlen_workspace_bytes(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, *, causal=False,
                                    rotary=None) -> int:
    a = _VarlenArg(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, causal)
    return int(load().attn_fwd_varlen_workspace_bytes(ctypes.byref(a.v), _rot_size_arg(rotary)))


def attn_fwd_varlen(Q, K, V, cu_seqlens_q, cu_seqlens_k, *, causal: bool = False, scale: Optional[float] = None,
                    O=None, LSE=None, O_lo=None, residual: bool = True, rotary: Optional[Rotary] = None,
                    workspace=None, stream=None):
    """Forward over packed sequences: Q [T_q, Hq, d_h], K [T_k, Hkv, d_h], V [T_k, Hkv, d_v] (bf16);
    cu_seqlens_* are host offsets [B + 1].  Returns (O [T_q, Hq, d_v], LSE [Hq, T_q] fp32, O_lo)."""
    (Tq, Tk, Hq, Hkv, d_h, d_v), dev = _varlen_dims(Q, K, V)
    a = _VarlenArg(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, causal)
    if a.total_q != Tq or a.total_k != Tk:
        raise ValueError("cu_seqlens_q[-1] / cu_seqlens_k[-1] must equal the token counts of Q / K")
    scale = 1.0 / math.sqrt(d_h) if scale is None else float(scale)
    if O is None:
        O = torch.empty((Tq, Hq, d_v), dtype=torch.bfloat16, device=dev)
    if LSE is None:
        LSE = torch.empty((Hq, Tq), dtype=torch.float32, device=dev)
    _check_tensor(O, "O", torch.bfloat16, (Tq, Hq, d_v), dev, strided=True)
    if O_lo is None and residual:
        O_lo = _like_o(O)
    _check_tensor(LSE, "LSE", torch.float32, (Hq, Tq), dev)
    if O_lo is not None:
        _check_o_lo(O_lo, O, (Tq, Hq, d_v), dev)
    if rotary is not None:
        rotary.check((Tq,), (Tk,), dev, Q, K)
    if workspace is None:
        need = int(load().attn_fwd_varlen_workspace_bytes(ctypes.byref(a.v), _rot_size_arg(rotary)))
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    st = _strides_arg(True, q=Q, k=K, v=V, o=O)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_fwd_varlen(ctypes.byref(a.v), st, rt, ctypes.c_float(scale), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                _ptr(LSE), _ptr(O_lo), *_ws(workspace), _stream(dev, stream))
    _check(rc, "attn_fwd_varlen")
    return O, LSE, O_lo


def attn_bwd_varlen_workspace_bytes(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, *, causal=False,
                                    rotary=None) -> int:
    a = _VarlenArg(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, causal)
    return int(load().attn_bwd_varlen_workspace_bytes(ctypes.byref(a.v), _rot_size_arg(rotary)))


def attn_bwd_varlen(Q, K, V, O, dO, LSE, cu_seqlens_q, cu_seqlens_k, *, O_lo=None, causal: bool = False,
                    scale: Optional[float] = None, dQ=None, dK=None, dV=None, rotary: Optional[Rotary] = None,
                    workspace=None, stream=None):
    """Backward over packed sequences: returns (dQ, dK, dV), laid out like Q, K, V."""
    (Tq, Tk, Hq, Hkv, d_h, d_v), dev = _varlen_dims(Q, K, V)
    a = _VarlenArg(Hq, Hkv, d_h, d_v, cu_seqlens_q, cu_seqlens_k, causal)
    if a.total_q != Tq or a.total_k != Tk:
        raise ValueError("cu_seqlens_q[-1] / cu_seqlens_k[-1] must equal the token counts of Q / K")
    scale = 1.0 / math.sqrt(d_h) if scale is None else float(scale)
    _check_tensor(O, "O", torch.bfloat16, (Tq, Hq, d_v), dev, strided=True)
    _check_tensor(dO, "dO", torch.bfloat16, (Tq, Hq, d_v), dev, strided=True)
    _check_tensor(LSE, "LSE", torch.float32, (Hq, Tq), dev)
    if O_lo is not None:
        _check_o_lo(O_lo, O, (Tq, Hq, d_v), dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check_tensor(dQ, "dQ", torch.bfloat16, tuple(Q.shape), dev, strided=True)
    _check_tensor(dK, "dK", torch.bfloat16, tuple(K.shape), dev, strided=True)
    _check_tensor(dV, "dV", torch.bfloat16, tuple(V.shape), dev, strided=True)
    if rotary is not None:
        rotary.check((Tq,), (Tk,), dev, Q, K)
    need = int(load().attn_bwd_varlen_workspace_bytes(ctypes.byref(a.v), _rot_size_arg(rotary)))
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must hold at least {need} bytes")
    st = _strides_arg(True, q=Q, k=K, v=V, o=O, dO=dO, dq=dQ, dk=dK, dv=dV)
    rt = None if rotary is None else rotary.arg()
    rc = load().attn_bwd_varlen(ctypes.byref(a.v), st, rt, ctypes.c_float(scale), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                _ptr(O_lo), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(workspace),
                                ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(dev, stream))
    _check(rc, "attn_bwd_varlen")
    return dQ, dK, dV


# ---------------------------------------------------------------------------
# Projections on either side of attention (row-major bf16 matrices)
# ---------------------------------------------------------------------------
def _mat(t, name, dtype, shape, dev):
    _check_tensor(t, name, dtype, shape, dev)
    return _ptr(t)


def attn_proj_fwd(X, W, *, Y=None, stream=None):
    """Y [T, N] = X [T, D] W [D, N] (bf16 in and out, fp32 accumulation)."""
    if X.dim() != 2 or W.dim() != 2:
        raise ValueError("X and W must be 2-D")
    T, D = (int(x) for x in X.shape)
    N = int(W.shape[1])
    dev = X.device
    Y = torch.empty((T, N), dtype=torch.bfloat16, device=dev) if Y is None else Y
    rc = load().attn_proj_fwd(T, D, N, _mat(X, "X", torch.bfloat16, (T, D), dev),
                              _mat(W, "W", torch.bfloat16, (D, N), dev), _mat(Y, "Y", torch.bfloat16, (T, N), dev),
                              _stream(dev, stream))
    _check(rc, "attn_proj_fwd")
    return Y


def attn_proj_bwd_weight(X, G, *, dW=None, stream=None):
    """dW [D, N] = X^T G (fp32 out)."""
    T, D = (int(x) for x in X.shape)
    N = int(G.shape[1])
    dev = X.device
    dW = torch.empty((D, N), dtype=torch.float32, device=dev) if dW is None else dW
    rc = load().attn_proj_bwd_weight(T, D, N, _mat(X, "X", torch.bfloat16, (T, D), dev),
                                     _mat(G, "G", torch.bfloat16, (T, N), dev),
                                     _mat(dW, "dW", torch.float32, (D, N), dev), _stream(dev, stream))
    _check(rc, "attn_proj_bwd_weight")
    return dW


def attn_proj_bwd_input(Gs, Ws, *, dX=None, stream=None):
    """dX [T, D] = sum_s G_s [T, N_s] W_s[D, N_s]^T over 1..3 branches that share X (bf16 out)."""
    if not 1 <= len(Gs) == len(Ws) <= 3:
        raise ValueError("1 to 3 (G, W) pairs")
    T = int(Gs[0].shape[0])
    D = int(Ws[0].shape[0])
    dev = Gs[0].device
    Ns = [int(g.shape[1]) for g in Gs]
    for k, (g, w) in enumerate(zip(Gs, Ws)):
        _check_tensor(g, f"G[{k}]", torch.bfloat16, (T, Ns[k]), dev)
        _check_tensor(w, f"W[{k}]", torch.bfloat16, (D, Ns[k]), dev)
    dX = torch.empty((T, D), dtype=torch.bfloat16, device=dev) if dX is None else dX
    _check_tensor(dX, "dX", torch.bfloat16, (T, D), dev)
    n_arr = (ctypes.c_int32 * len(Ns))(*Ns)
    g_arr = (_vp * len(Gs))(*[g.data_ptr() for g in Gs])
    w_arr = (_vp * len(Ws))(*[w.data_ptr() for w in Ws])
    rc = load().attn_proj_bwd_input(T, D, len(Gs), n_arr, g_arr, w_arr, _ptr(dX), _stream(dev, stream))
    _check(rc, "attn_proj_bwd_input")
    return dX


def attn_rope(X, positions, *, base: float = 10000.0, inverse: bool = False, Y=None, stream=None):
    """Rotary position embedding of token-major rows X [tokens, heads, d] (bf16)
    at int32 positions [tokens] (device); inverse=True rotates back (the
    gradient map).  Y may be X (in place)."""
    if X.dim() != 3:
        raise ValueError("X must be [tokens, heads, d]")
    T, H, d = (int(x) for x in X.shape)
    dev = X.device
    _check_tensor(X, "X", torch.bfloat16, (T, H, d), dev)
    _check_tensor(positions, "positions", torch.int32, (T,), dev)
    Y = torch.empty_like(X) if Y is None else Y
    _check_tensor(Y, "Y", torch.bfloat16, (T, H, d), dev)
    rc = load().attn_rope(T, H, d, ctypes.c_float(base), _ptr(positions), 1 if inverse else 0, _ptr(X), _ptr(Y),
                          _stream(dev, stream))
    _check(rc, "attn_rope")
    return Y


def attn_rope_qk(Q, K, positions, *, base: float = 10000.0, inverse: bool = False, Yq=None, Yk=None, stream=None):
    """attn_rope of queries Q [tokens, Hq, d] and keys K [tokens, Hkv, d] at
    the same positions, in one launch; returns (Yq, Yk).  Yq may be Q and Yk
    may be K (in place)."""
    if Q.dim() != 3 or K.dim() != 3:
        raise ValueError("Q and K must be [tokens, heads, d]")
    T, Hq, d = (int(x) for x in Q.shape)
    Hk = int(K.shape[1])
    dev = Q.device
    _check_tensor(Q, "Q", torch.bfloat16, (T, Hq, d), dev)
    _check_tensor(K, "K", torch.bfloat16, (T, Hk, d), dev)
    _check_tensor(positions, "positions", torch.int32, (T,), dev)
    Yq = torch.empty_like(Q) if Yq is None else Yq
    Yk = torch.empty_like(K) if Yk is None else Yk
    _check_tensor(Yq, "Yq", torch.bfloat16, (T, Hq, d), dev)
    _check_tensor(Yk, "Yk", torch.bfloat16, (T, Hk, d), dev)
    rc = load().attn_rope_qk(T, Hq, Hk, d, ctypes.c_float(base), _ptr(positions), 1 if inverse else 0, _ptr(Q),
                             _ptr(Yq), _ptr(K), _ptr(Yk), _stream(dev, stream))
    _check(rc, "attn_rope_qk")
    return Yq, Yk
