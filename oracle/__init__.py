"""fp64 CPU oracle for masked scaled dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``exact_scaled_dot_gb300``) never imports it, and this package never imports
the product library: the two share nothing but the seeded inputs they are
handed.

The arithmetic lives in ``attn_oracle.c`` (plain loops, double precision); this
module compiles it with gcc, loads it with ctypes and exposes numpy functions.
Each function names the equation it follows:

* [A10]  "Appendix A.10 -- Attention matrices and backpropagation",
  eqs. A.10.1-A.10.9, sections A.10.5 (GQA) and A.10.6 (causality).
* [HAND] "Computing attention term by term", worked examples 1 and 2.
* [CH31] "Chapter 31 -- attention backprop", sections 1-4.

Parity is pinned by ``tests/test_oracle_pins.py`` (worked examples, closed
forms, invariants, finite differences and negative controls); the large
configurations have no pin beyond those invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from pathlib import Path
from typing import Optional, Sequence

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "attn_oracle.c"
_BUILD = _HERE / "_build"


def build(mutation: int = 0, out_dir: Optional[Path] = None, force: bool = False) -> Path:
    """Compile the oracle into a shared library and return its path.

    ``mutation`` selects a deliberately broken variant for the negative
    controls of the oracle's own tests (see the header of attn_oracle.c);
    0 is the real oracle.
    """
    out_dir = Path(out_dir) if out_dir is not None else _BUILD
    out_dir.mkdir(parents=True, exist_ok=True)
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    lib = out_dir / name
    if force or not lib.exists() or lib.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = out_dir / (name + f".tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               f"-DORACLE_MUTATION={int(mutation)}", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "Hq", "Hkv", "nq", "nk", "dh", "dv")]


class _Mask(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int32), ("offset", ctypes.c_int64),
                ("kv_len", ctypes.POINTER(ctypes.c_int32))]


_P = ctypes.POINTER(ctypes.c_double)
_PI = ctypes.POINTER(ctypes.c_int64)


@dataclass(frozen=True)
class Problem:
    """Shapes and visible-set description of one attention call.

    ``causal`` restricts row i to keys j <= i + offset; ``offset=None`` means
    bottom-right alignment n_k - n_q (0 for self-attention).  ``kv_len`` is a
    per-batch key length (key padding) or None.
    """
    B: int
    Hq: int
    Hkv: int
    nq: int
    nk: int
    dh: int
    dv: int
    causal: bool = False
    offset: Optional[int] = None
    kv_len: Optional[Sequence[int]] = None

    @property
    def causal_offset(self) -> int:
        return (self.nk - self.nq) if self.offset is None else int(self.offset)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: Optional[Path] = None):
        self.path = Path(lib_path) if lib_path is not None else build()
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_visible_pairs.restype = ctypes.c_int64
        lib.oracle_visible_pairs.argtypes = [ctypes.POINTER(_Shape), ctypes.POINTER(_Mask)]
        lib.oracle_first_empty_row.restype = ctypes.c_int64
        lib.oracle_first_empty_row.argtypes = [ctypes.POINTER(_Shape), ctypes.POINTER(_Mask)]
        lib.oracle_dense_matrices.restype = ctypes.c_int
        lib.oracle_dense_matrices.argtypes = [ctypes.POINTER(_Shape), ctypes.POINTER(_Mask),
                                              ctypes.c_double, _P, _P, _P, _P, _P, _P, _P, _P]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [ctypes.POINTER(_Shape), ctypes.POINTER(_Mask),
                                       ctypes.c_double, _P, _P, _P, _PI, ctypes.c_int64, _P, _P]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [ctypes.POINTER(_Shape), ctypes.POINTER(_Mask),
                                        ctypes.c_double, _P, _P, _P, _P,
                                        _PI, ctypes.c_int64, _PI, ctypes.c_int64,
                                        _P, _P, _P, _P, _P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        self._lib = lib

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _structs(p: Problem):
        shape = _Shape(p.B, p.Hq, p.Hkv, p.nq, p.nk, p.dh, p.dv)
        keep = None
        kv = ctypes.POINTER(ctypes.c_int32)()
        if p.kv_len is not None:
            keep = np.ascontiguousarray(np.asarray(p.kv_len, dtype=np.int32))
            if keep.shape != (p.B,):
                raise ValueError("kv_len must have one entry per batch element")
            kv = keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        mask = _Mask(1 if p.causal else 0, p.causal_offset, kv)
        return shape, mask, keep

    @staticmethod
    def _f64(x, shape) -> np.ndarray:
        a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        if a.shape != tuple(shape):
            raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
        return a

    @staticmethod
    def _ptr(a: Optional[np.ndarray]):
        return a.ctypes.data_as(_P) if a is not None else _P()

    def _inputs(self, p: Problem, Q, K, V, G=None):
        Q = self._f64(Q, (p.B, p.Hq, p.nq, p.dh))
        K = self._f64(K, (p.B, p.Hkv, p.nk, p.dh))
        V = self._f64(V, (p.B, p.Hkv, p.nk, p.dv))
        G = None if G is None else self._f64(G, (p.B, p.Hq, p.nq, p.dv))
        if p.Hq % p.Hkv != 0:
            raise ValueError("Hq must be a multiple of Hkv")
        return Q, K, V, G

    @staticmethod
    def _rows(rows):
        if rows is None:
            return None, _PI(), 0
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        return r, r.ctypes.data_as(_PI), r.size

    # -- public API ------------------------------------------------------
    @property
    def threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def set_threads(self, n: int) -> None:
        self._lib.oracle_set_num_threads(int(n))

    def visible_pairs(self, p: Problem) -> int:
        """Count of visible (i, j) pairs summed over batch and query heads."""
        shape, mask, _keep = self._structs(p)
        return int(self._lib.oracle_visible_pairs(ctypes.byref(shape), ctypes.byref(mask)))

    def first_empty_row(self, p: Problem) -> int:
        """Flattened index of the first query row with an empty visible set, or -1."""
        shape, mask, _keep = self._structs(p)
        return int(self._lib.oracle_first_empty_row(ctypes.byref(shape), ctypes.byref(mask)))

    def dense(self, p: Problem, Q, K, V, G=None, scale: Optional[float] = None):
        """Dense S (NaN off the visible set), A, dA and dS, each [B,Hq,nq,nk]."""
        scale = 1.0 / np.sqrt(p.dh) if scale is None else float(scale)
        Q, K, V, G = self._inputs(p, Q, K, V, G)
        shape, mask, _keep = self._structs(p)
        out = [np.empty((p.B, p.Hq, p.nq, p.nk)) for _ in range(4)]
        rc = self._lib.oracle_dense_matrices(ctypes.byref(shape), ctypes.byref(mask), scale,
                                             self._ptr(Q), self._ptr(K), self._ptr(V), self._ptr(G),
                                             *(self._ptr(o) for o in out))
        if rc != 0:
            raise ValueError("a query row has an empty visible set")
        S, A, dA, dS = out
        return S, A, (dA if G is not None else None), (dS if G is not None else None)

    def forward(self, p: Problem, Q, K, V, scale: Optional[float] = None, rows=None):
        """O [.., dv] and LSE for every query row, or for flattened ``rows``."""
        scale = 1.0 / np.sqrt(p.dh) if scale is None else float(scale)
        Q, K, V, _ = self._inputs(p, Q, K, V)
        shape, mask, _keep = self._structs(p)
        r, rp, nr = self._rows(rows)
        n = nr if r is not None else p.B * p.Hq * p.nq
        O = np.empty((n, p.dv))
        LSE = np.empty((n,))
        rc = self._lib.oracle_forward(ctypes.byref(shape), ctypes.byref(mask), scale,
                                      self._ptr(Q), self._ptr(K), self._ptr(V), rp, nr,
                                      self._ptr(O), self._ptr(LSE))
        if rc != 0:
            raise ValueError("a query row has an empty visible set")
        if r is None:
            return O.reshape(p.B, p.Hq, p.nq, p.dv), LSE.reshape(p.B, p.Hq, p.nq)
        return O, LSE

    def backward(self, p: Problem, Q, K, V, G, scale: Optional[float] = None,
                 q_rows=None, k_rows=None, want_dq=True, want_dkdv=True):
        """dQ, dK, dV, D (= rowsum(G*O)) and C (= c_i of A.10.7).

        With ``q_rows``/``k_rows`` (flattened (b, r, i) / (b, h, j) indices) only
        those rows of dQ, D, C / dK, dV are produced, as 2-D arrays.
        """
        scale = 1.0 / np.sqrt(p.dh) if scale is None else float(scale)
        Q, K, V, G = self._inputs(p, Q, K, V, G)
        shape, mask, _keep = self._structs(p)
        qr, qp, nq_ = self._rows(q_rows)
        kr, kp, nk_ = self._rows(k_rows)
        n_q = nq_ if qr is not None else p.B * p.Hq * p.nq
        n_k = nk_ if kr is not None else p.B * p.Hkv * p.nk
        dQ = np.empty((n_q, p.dh)) if want_dq else None
        D = np.empty((n_q,)) if want_dq else None
        C = np.empty((n_q,)) if want_dq else None
        dK = np.empty((n_k, p.dh)) if want_dkdv else None
        dV = np.empty((n_k, p.dv)) if want_dkdv else None
        rc = self._lib.oracle_backward(ctypes.byref(shape), ctypes.byref(mask), scale,
                                       self._ptr(Q), self._ptr(K), self._ptr(V), self._ptr(G),
                                       qp, nq_, kp, nk_,
                                       self._ptr(dQ), self._ptr(D), self._ptr(C),
                                       self._ptr(dK), self._ptr(dV))
        if rc == -1:
            raise ValueError("a query row has an empty visible set")
        if rc != 0:
            raise MemoryError("oracle could not allocate its row statistics")
        if qr is None and want_dq:
            dQ = dQ.reshape(p.B, p.Hq, p.nq, p.dh)
            D = D.reshape(p.B, p.Hq, p.nq)
            C = C.reshape(p.B, p.Hq, p.nq)
        if kr is None and want_dkdv:
            dK = dK.reshape(p.B, p.Hkv, p.nk, p.dh)
            dV = dV.reshape(p.B, p.Hkv, p.nk, p.dv)
        return dQ, dK, dV, D, C


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    """The real (unmutated) oracle, built on first use."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
