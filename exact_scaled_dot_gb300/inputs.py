"""Seeded synthetic inputs for the attention workloads.

This module only describes shapes and draws random numbers: it holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it without sharing any computation.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws, in this order, fp32 samples N(0, sigma_qk^2) for Q and K and
N(0, sigma_v^2) for V and dO, each rounded to bfloat16 (round to nearest
even); then, for key-padded workloads, per-batch key lengths uniform on the
inclusive range ``kv_len_range``.  The pages fix no dataset: these draws stand
in for real activations, with the shapes, masks and value scales of the five
workloads the method is measured on (the peaked-softmax cross-attention case
scales Q and K by 3, so the logits have standard deviation 9 by the variance
argument of eq. A.10.4 of "Appendix A.10 -- Attention matrices and
backpropagation").
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, List, Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, visible-set description and value scales."""
    name: str
    B: int
    Hq: int
    Hkv: int
    nq: int
    nk: int
    dh: int
    dv: int
    causal: bool = False
    offset: Optional[int] = None          # None: n_k - n_q (bottom-right aligned)
    kv_len_range: Optional[Tuple[int, int]] = None   # inclusive, or None (no padding)
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    seed: int = 0

    @property
    def causal_offset(self) -> int:
        return (self.nk - self.nq) if self.offset is None else int(self.offset)

    def with_seed(self, seed: int) -> "Workload":
        return replace(self, seed=seed)

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (e.g. smaller sizes for quick tests)."""
        return replace(self, **kw)


# The five workloads: a tiny single head, causal MHA, causal GQA with key
# padding, peaked cross-attention with key padding, and MQA chunked prefill
# (new queries over a long history, causal with an offset).  Seeds 1000 + k.
WORKLOADS: Dict[str, Workload] = {
    "single_head_full": Workload("single_head_full", B=1, Hq=1, Hkv=1, nq=128, nk=128,
                                 dh=64, dv=64, seed=1001),
    "mha_causal": Workload("mha_causal", B=4, Hq=16, Hkv=16, nq=2048, nk=2048,
                           dh=128, dv=128, causal=True, seed=1002),
    "gqa_causal_padded": Workload("gqa_causal_padded", B=2, Hq=32, Hkv=8, nq=4096, nk=4096,
                                  dh=128, dv=128, causal=True, kv_len_range=(2048, 4096),
                                  seed=1003),
    "cross_padded_peaked": Workload("cross_padded_peaked", B=8, Hq=16, Hkv=16, nq=512, nk=8192,
                                    dh=128, dv=64, kv_len_range=(4096, 8192), sigma_qk=3.0,
                                    seed=1004),
    "mqa_chunked_prefill": Workload("mqa_chunked_prefill", B=1, Hq=64, Hkv=1, nq=1024, nk=16384,
                                    dh=128, dv=128, causal=True, seed=1005),
    # One causal MQA sequence: 32 key tiles, so the backward's CTAs (one per
    # key tile of the single KV head) would fill a fifth of the GPU without
    # the query-head split.  Not one of the five benchmark configurations.
    "mqa_single_sequence": Workload("mqa_single_sequence", B=1, Hq=32, Hkv=1, nq=4096, nk=4096,
                                    dh=128, dv=128, causal=True, seed=1006),
    # Short query blocks over a long key cache (decode and small chunks of new
    # queries): causal with the bottom-right offset n_k - n_q, ragged cache
    # lengths.  Forward only; HBM-bound (the K/V cache is read once).
    "decode_gqa": Workload("decode_gqa", B=8, Hq=32, Hkv=8, nq=1, nk=32768, dh=128, dv=128, causal=True,
                           kv_len_range=(16384, 32768), seed=1101),
    "decode_mqa_chunk": Workload("decode_mqa_chunk", B=8, Hq=64, Hkv=1, nq=16, nk=65536, dh=128, dv=128,
                                 causal=True, kv_len_range=(32768, 65536), seed=1102),
}

DECODE_WORKLOADS = ["decode_gqa", "decode_mqa_chunk"]

WORKLOAD_ORDER = ["single_head_full", "mha_causal", "gqa_causal_padded",
                  "cross_padded_peaked", "mqa_chunked_prefill"]


@dataclass
class Inputs:
    """bf16 tensors on the CPU (contiguous [B, H, n, d]) and int32 key lengths."""
    Q: torch.Tensor
    K: torch.Tensor
    V: torch.Tensor
    dO: torch.Tensor
    kv_len: Optional[torch.Tensor]


def make_inputs(w: Workload, seed: Optional[int] = None) -> Inputs:
    """Draw the workload's inputs (see the module docstring for the recipe)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed if seed is None else seed))

    def draw(shape, sigma):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        return x.to(torch.bfloat16).contiguous()

    Q = draw((w.B, w.Hq, w.nq, w.dh), w.sigma_qk)
    K = draw((w.B, w.Hkv, w.nk, w.dh), w.sigma_qk)
    V = draw((w.B, w.Hkv, w.nk, w.dv), w.sigma_v)
    dO = draw((w.B, w.Hq, w.nq, w.dv), w.sigma_v)
    kv_len = None
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        kv_len = torch.randint(int(lo), int(hi) + 1, (w.B,), generator=g, dtype=torch.int64)
        kv_len = kv_len.to(torch.int32)
    return Inputs(Q, K, V, dO, kv_len)


# ---------------------------------------------------------------------------
# Packed variable-length sequences (token-major tensors)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class VarlenWorkload:
    """Packed sequences: per-sequence query and key lengths, token-major
    tensors Q [T_q, Hq, d_h], K [T_k, Hkv, d_h], V [T_k, Hkv, d_v],
    dO [T_q, Hq, d_v].  With ``len_range`` set, lengths are drawn uniformly
    on that inclusive range (the same length for queries and keys of a
    sequence: packed self-attention); explicit ``lens_q`` / ``lens_k`` take
    precedence."""
    name: str
    B: int
    Hq: int
    Hkv: int
    dh: int
    dv: int
    causal: bool = False
    len_range: Optional[Tuple[int, int]] = None
    lens_q: Optional[Tuple[int, ...]] = None
    lens_k: Optional[Tuple[int, ...]] = None
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    seed: int = 0


@dataclass
class VarlenInputs:
    Q: torch.Tensor
    K: torch.Tensor
    V: torch.Tensor
    dO: torch.Tensor
    lens_q: List[int]
    lens_k: List[int]
    cu_q: List[int]
    cu_k: List[int]


def make_varlen_inputs(w: VarlenWorkload, seed: Optional[int] = None) -> VarlenInputs:
    """Draw the lengths first (when drawn), then Q, K, V, dO as in make_inputs."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed if seed is None else seed))
    if w.lens_q is not None:
        lq = [int(x) for x in w.lens_q]
        lk = [int(x) for x in (w.lens_k if w.lens_k is not None else w.lens_q)]
    else:
        lo, hi = w.len_range
        lq = torch.randint(int(lo), int(hi) + 1, (w.B,), generator=g, dtype=torch.int64).tolist()
        lk = list(lq)
    cu_q, cu_k = [0], [0]
    for a, b in zip(lq, lk):
        cu_q.append(cu_q[-1] + a)
        cu_k.append(cu_k[-1] + b)

    def draw(shape, sigma):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        return x.to(torch.bfloat16).contiguous()

    Q = draw((cu_q[-1], w.Hq, w.dh), w.sigma_qk)
    K = draw((cu_k[-1], w.Hkv, w.dh), w.sigma_qk)
    V = draw((cu_k[-1], w.Hkv, w.dv), w.sigma_v)
    dO = draw((cu_q[-1], w.Hq, w.dv), w.sigma_v)
    return VarlenInputs(Q, K, V, dO, lq, lk, cu_q, cu_k)


# Packed causal GQA sequences of mixed lengths (a training batch without
# padding): 16 sequences of 256..4096 tokens, 32 query heads over 8 KV heads.
VARLEN_WORKLOADS: Dict[str, VarlenWorkload] = {
    "varlen_gqa_causal": VarlenWorkload("varlen_gqa_causal", B=16, Hq=32, Hkv=8, dh=128, dv=128, causal=True,
                                        len_range=(256, 4096), seed=1201),
}


# ---------------------------------------------------------------------------
# Projections on either side of attention
# ---------------------------------------------------------------------------
@dataclass
class ProjInputs:
    X: torch.Tensor          # [T, D]
    Ws: List[torch.Tensor]   # [D, N_s]
    Gs: List[torch.Tensor]   # [T, N_s] upstream gradients of the projections' outputs


def make_proj_inputs(T: int, D: int, Ns, seed: int) -> ProjInputs:
    """X ~ N(0, 1), W_s ~ N(0, 1/D) (so X W_s has unit variance), G_s ~ N(0, 1),
    drawn in that order from a seeded CPU generator and rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def draw(shape, sigma):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        return x.to(torch.bfloat16).contiguous()

    X = draw((T, D), 1.0)
    Ws = [draw((D, int(n)), 1.0 / float(D) ** 0.5) for n in Ns]
    Gs = [draw((T, int(n)), 1.0) for n in Ns]
    return ProjInputs(X, Ws, Gs)


# The projections of the causal GQA workload: 8192 tokens (2 x 4096) of width
# 4096 into Q (32 heads x 128), K and V (8 heads x 128 each).
PROJ_WORKLOADS = {
    "proj_qkv_gqa": dict(T=8192, D=4096, Ns=(4096, 1024, 1024), seed=1301),
}
