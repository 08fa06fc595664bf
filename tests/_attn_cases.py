"""Shared test plumbing: run the CUDA path and the oracle on the same inputs.

Test-only.  The CUDA side goes through the package (the C ABI); the oracle
side receives the very same bf16 inputs upcast exactly to float64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from exact_scaled_dot_gb300.inputs import Inputs, Workload, make_inputs

ATOL, RTOL = 1e-2, 2e-2          # O, dQ, dK, dV: |gpu - ref| <= ATOL + RTOL |ref|
LSE_ATOL = 1e-3                  # LSE: absolute


def problem_of(w: Workload, inp: Inputs):
    import oracle
    kv = None if inp.kv_len is None else [int(x) for x in inp.kv_len.tolist()]
    return oracle.Problem(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal,
                          offset=w.causal_offset if w.causal else None, kv_len=kv)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


@dataclass
class GpuResult:
    O: torch.Tensor
    LSE: torch.Tensor
    dQ: torch.Tensor
    dK: torch.Tensor
    dV: torch.Tensor
    status: int


def run_gpu(w: Workload, inp: Inputs, scale: Optional[float] = None, poison: bool = True,
            device: str = "cuda:0") -> GpuResult:
    import exact_scaled_dot_gb300 as esd
    Q, K, V, dO = (x.to(device) for x in (inp.Q, inp.K, inp.V, inp.dO))
    kv = None if inp.kv_len is None else inp.kv_len.tolist()
    fill = float("nan") if poison else 0.0
    O = torch.full((w.B, w.Hq, w.nq, w.dv), fill, dtype=torch.bfloat16, device=device)
    LSE = torch.full((w.B, w.Hq, w.nq), fill, dtype=torch.float32, device=device)
    dQ = torch.full_like(Q, fill)
    dK = torch.full_like(K, fill)
    dV = torch.full_like(V, fill)
    off = w.causal_offset if w.causal else None
    O_lo = torch.full_like(O, fill)
    esd.attn_fwd(Q, K, V, causal=w.causal, causal_offset=off, kv_len=kv, scale=scale, O=O, LSE=LSE, O_lo=O_lo)
    esd.attn_bwd(Q, K, V, O, dO, LSE, O_lo=O_lo, causal=w.causal, causal_offset=off, kv_len=kv, scale=scale,
                 dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    status = esd.attn_get_status()
    return GpuResult(O, LSE, dQ, dK, dV, status)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    excess = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    bad = ~(excess <= 0)          # NaN counts as bad
    if bad.any():
        idx = np.unravel_index(np.nanargmax(np.where(bad, np.nan_to_num(excess, nan=np.inf), -np.inf)), got.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.size} elements outside {atol} + {rtol}|ref|; "
            f"worst at {idx}: gpu={got[idx]!r} ref={ref[idx]!r}")


def assert_same_sum(got: torch.Tensor, ref: torch.Tensor, what: str):
    """Two results of the same sums accumulated in a different order: dQ
    always, dK and dV when the backward splits a KV head's query heads over
    several CTAs (their fp32 shares are added in whatever order the CTAs
    finish).  Equal up to the last bits of the fp32 sums, which can move the
    bf16 rounding that follows by one unit (a relative 2^-8 to 2^-7)."""
    assert_close(f64(got), f64(ref), what, atol=1e-3, rtol=8e-3)


def max_err(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))


def compare_full(w: Workload, inp: Inputs, res: GpuResult, orc, scale: Optional[float] = None):
    """Element-by-element comparison of every output against the oracle."""
    p = problem_of(w, inp)
    Q, K, V, G = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    O, LSE = orc.forward(p, Q, K, V, scale=scale)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G, scale=scale)
    assert res.status == 0, f"device status {res.status}"
    assert_close(f64(res.O), O, "O")
    assert_close(f64(res.LSE), LSE, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(res.dQ), dQ, "dQ")
    assert_close(f64(res.dK), dK, "dK")
    assert_close(f64(res.dV), dV, "dV")


def sample_rows(w: Workload, n_rows: int, n_keys: int, seed: int = 0):
    """Flattened (b, r, i) query rows and (b, h, j) key rows to check, always
    including the first and last row of the first and last head (tile and
    tail edges) plus random ones."""
    rng = np.random.default_rng(seed)
    total_q = w.B * w.Hq * w.nq
    total_k = w.B * w.Hkv * w.nk
    fixed_q = [0, w.nq - 1, total_q - w.nq, total_q - 1, min(127, w.nq - 1), min(128, w.nq - 1)]
    fixed_k = [0, w.nk - 1, total_k - w.nk, total_k - 1, min(127, w.nk - 1), min(128, w.nk - 1)]
    q = np.unique(np.concatenate([fixed_q, rng.integers(0, total_q, n_rows)]))
    k = np.unique(np.concatenate([fixed_k, rng.integers(0, total_k, n_keys)]))
    return q.astype(np.int64), k.astype(np.int64)


def compare_sampled(w: Workload, inp: Inputs, res: GpuResult, orc, n_rows=192, n_keys=96, seed=0):
    """Compare sampled output rows with the oracle computed row by row."""
    p = problem_of(w, inp)
    Q, K, V, G = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    qr, kr = sample_rows(w, n_rows, n_keys, seed)
    O, LSE = orc.forward(p, Q, K, V, rows=qr)
    dQ, dK, dV, _D, _C = orc.backward(p, Q, K, V, G, q_rows=qr, k_rows=kr)
    assert res.status == 0, f"device status {res.status}"
    assert_close(f64(res.O).reshape(-1, w.dv)[qr], O, "O")
    assert_close(f64(res.LSE).reshape(-1)[qr], LSE, "LSE", atol=LSE_ATOL, rtol=0.0)
    assert_close(f64(res.dQ).reshape(-1, w.dh)[qr], dQ, "dQ")
    assert_close(f64(res.dK).reshape(-1, w.dh)[kr], dK, "dK")
    assert_close(f64(res.dV).reshape(-1, w.dv)[kr], dV, "dV")
    # Properties that hold at any size: every output finite.
    for name in ("O", "LSE", "dQ", "dK", "dV"):
        t = getattr(res, name)
        assert bool(torch.isfinite(t).all()), f"{name} has non-finite entries"


def varlen_reference(w, inp, orc):
    """Oracle outputs packed token-major: O, LSE [Hq, T_q], dQ, dK, dV."""
    import oracle
    Q, K, V, G = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
    Tq, Tk = Q.shape[0], K.shape[0]
    O = np.zeros((Tq, w.Hq, w.dv))
    LSE = np.zeros((w.Hq, Tq))
    dQ = np.zeros((Tq, w.Hq, w.dh))
    dK = np.zeros((Tk, w.Hkv, w.dh))
    dV = np.zeros((Tk, w.Hkv, w.dv))
    for b in range(len(inp.lens_q)):
        lq, lk = inp.lens_q[b], inp.lens_k[b]
        q0, q1, k0, k1 = inp.cu_q[b], inp.cu_q[b + 1], inp.cu_k[b], inp.cu_k[b + 1]
        if lq == 0:
            continue            # no query sees these keys: dK = dV = 0
        p = oracle.Problem(1, w.Hq, w.Hkv, lq, lk, w.dh, w.dv, causal=w.causal, offset=None, kv_len=None)
        to_bhnd = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2)[None])  # noqa: E731  [n,H,d] -> [1,H,n,d]
        Qb, Kb, Vb, Gb = to_bhnd(Q[q0:q1]), to_bhnd(K[k0:k1]), to_bhnd(V[k0:k1]), to_bhnd(G[q0:q1])
        Ob, Lb = orc.forward(p, Qb, Kb, Vb)
        dQb, dKb, dVb, _D, _C = orc.backward(p, Qb, Kb, Vb, Gb)
        O[q0:q1] = Ob[0].transpose(1, 0, 2)
        LSE[:, q0:q1] = Lb[0]
        dQ[q0:q1] = dQb[0].transpose(1, 0, 2)
        dK[k0:k1] = dKb[0].transpose(1, 0, 2)
        dV[k0:k1] = dVb[0].transpose(1, 0, 2)
    return O, LSE, dQ, dK, dV
