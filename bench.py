#!/usr/bin/env python3
"""Benchmark: masked attention forward + backward on GB300, one JSON line.

A step is one forward and one backward pass (every kernel of the path) over
the causal GQA workload with key padding (B=2, Hq=32, Hkv=8, n=4096,
d_h=d_v=128, per-batch key lengths uniform in [2048, 4096]) -- the n=4096,
d=128 causal configuration the throughput target is stated on.  The value is
TFLOP/s counted on visible (i, j) pairs only: 2(d_h+d_v) FLOPs per pair
forward and 2(2 d_h + 3 d_v) backward, summed over all ranks.

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Under torchrun each rank runs its own full replica (the path needs no
exchange between GPUs); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import signal
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "attention fwd+bwd TFLOP/s (visible pairs) and % of GB300 dense-BF16 peak"
DEFAULT_WORKLOAD = "gqa_causal_padded"
PEAKS_FILE = ROOT / "MEASURED_PEAKS.json"
TRAFFIC_FILE = ROOT / "profiles" / "ncu_traffic.json"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# Helpers shared by both arms
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest per-rank value over all ranks of the initialised process
    group (the value itself when not distributed).  Used for the timed
    region: the job takes as long as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank does one step's work per step (weak
    scaling), so the job does `world` times the per-rank FLOPs in the
    slowest rank's time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def flops_per_pair(dh: int, dv: int):
    return 2 * (dh + dv), 2 * (2 * dh + 3 * dv)


def load_peaks():
    if PEAKS_FILE.exists():
        try:
            d = json.loads(PEAKS_FILE.read_text())
            return d, "measured"
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    for p in sorted((ROOT / "exact_scaled_dot_gb300" / "csrc").glob("*")):
        h.update(p.name.encode())
        h.update(p.read_bytes())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.error = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if exe is None:
            self.error = "nvidia-smi not found"
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                [exe, f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError as e:
            self.error = str(e)

    def stop(self):
        if self.proc is None:
            return {"error": self.error or "not sampled"}
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"error": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def oracle_cpu_sample(w, inp, rows: int):
    """Time the fp64 oracle (forward + backward) on a bounded sub-problem of the
    workload: batch 0, KV head 0 with its query heads, the first `rows` query
    rows and the keys they can see.  Returns (TFLOP/s, description, threads)."""
    import numpy as np
    import oracle

    orc = oracle.default()
    g = w.Hq // w.Hkv
    n_q = min(rows, w.nq)
    L0 = int(inp.kv_len[0]) if inp.kv_len is not None else w.nk
    if w.causal:
        n_k = min(w.nk, L0, n_q + w.causal_offset)
    else:
        n_k = min(w.nk, L0)
    n_k = max(n_k, 1)
    off = w.causal_offset if w.causal else None
    p = oracle.Problem(1, g, 1, n_q, n_k, w.dh, w.dv, causal=w.causal, offset=off, kv_len=None)
    f64 = lambda t: t.to(__import__("torch").float64).numpy()  # noqa: E731
    Q = f64(inp.Q[0:1, 0:g, :n_q])
    K = f64(inp.K[0:1, 0:1, :n_k])
    V = f64(inp.V[0:1, 0:1, :n_k])
    G = f64(inp.dO[0:1, 0:g, :n_q])
    pairs = orc.visible_pairs(p)
    ff, fb = flops_per_pair(w.dh, w.dv)
    t0 = time.perf_counter()
    orc.forward(p, Q, K, V)
    orc.backward(p, Q, K, V, G)
    dt = time.perf_counter() - t0
    desc = (f"batch 0, KV head 0 with its {g} query heads, first {n_q} query rows over {n_k} keys "
            f"({pairs} visible pairs), fp64 forward+backward")
    return pairs * (ff + fb) / dt / 1e12, desc, orc.threads, dt


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from exact_scaled_dot_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    rows = args.reference_rows
    for _ in range(max(0, args.warmup)):
        oracle_cpu_sample(w, inp, min(rows, 64))
    vals, times = [], []
    desc, threads = "", 0
    for _ in range(args.steps):
        v, desc, threads, dt = oracle_cpu_sample(w, inp, rows)
        vals.append(v)
        times.append(dt)
    value = len(vals) / sum(1.0 / v for v in vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) draws rounded to bf16, upcast to fp64)",
        "config": {"workload": w.name, "sample_of": "see cpu_baseline.sample"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# CUDA arm
# ---------------------------------------------------------------------------
KERNEL_STAGES = ["attn_fwd (V pre-pass + forward kernel)", "attn_bwd_preprocess_kernel", "attn_bwd_main_kernel",
                 "attn_bwd_finalize_kernel"]
LAUNCHES_PER_STEP = 6   # attn_v16_kernel, attn_fwd_kernel, preprocess, group exponents, main, finalize


class AttnStep:
    """Device buffers of one workload and its fwd+bwd step through the public
    calls (the forward, then the backward's three stages), with optional
    CUDA events between the calls."""

    def __init__(self, esd, w, inp, dev, rotary=False, keep_rotated=False):
        import torch
        self.esd, self.w = esd, w
        self.kv = None if inp.kv_len is None else inp.kv_len.tolist()
        off = w.causal_offset if w.causal else None
        self.mask = dict(causal=w.causal, causal_offset=off, kv_len=self.kv)
        self.shape = esd.make_shape(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
        self.pairs = esd.attn_visible_pairs(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, **self.mask)
        ff, fb = flops_per_pair(w.dh, w.dv)
        self.flops_fwd, self.flops_bwd = self.pairs * ff, self.pairs * fb
        self.scale = 1.0 / math.sqrt(w.dh)
        self.Q, self.K, self.V, self.dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
        self.O = torch.empty((w.B, w.Hq, w.nq, w.dv), dtype=torch.bfloat16, device=dev)
        self.LSE = torch.empty((w.B, w.Hq, w.nq), dtype=torch.float32, device=dev)
        self.O_lo = torch.empty_like(self.O)
        self.dQ, self.dK, self.dV = torch.empty_like(self.Q), torch.empty_like(self.K), torch.empty_like(self.V)
        dims = (w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv)
        # Rotary: every row at its sequence position (queries at the end of
        # the keys when n_q < n_k), the rotation fused into the calls.
        self.rot = None
        if rotary:
            pk = torch.arange(w.nk, dtype=torch.int32, device=dev).expand(w.B, w.nk).contiguous()
            kept = (torch.empty_like(self.Q), torch.empty_like(self.K)) if keep_rotated else (None, None)
            self.rot = esd.Rotary(pk[:, w.nk - w.nq:].contiguous(), pk, base=10000.0, q_rot=kept[0], k_rot=kept[1])
        self.fws = torch.empty((esd.attn_fwd_workspace_bytes(*dims, rotary=self.rot),), dtype=torch.uint8, device=dev)
        self.ws = torch.empty((esd.attn_bwd_workspace_bytes(*dims, rotary=self.rot),), dtype=torch.uint8, device=dev)
        self.rows = w.B * w.Hq * w.nq

    def tensors(self):
        return (self.Q, self.K, self.V, self.dO, self.O, self.O_lo, self.LSE, self.dQ, self.dK, self.dV, self.ws,
                self.fws)

    def bytes_touched(self):
        return sum(x.numel() * x.element_size() for x in self.tensors())

    def __call__(self, stream, ev=None):
        esd = self.esd
        if ev is not None:
            ev[0].record(stream)
        esd.attn_fwd(self.Q, self.K, self.V, scale=self.scale, O=self.O, LSE=self.LSE, O_lo=self.O_lo,
                     rotary=self.rot, workspace=self.fws, stream=stream, **self.mask)
        if ev is not None:
            ev[1].record(stream)
        esd.attn_bwd_preprocess(self.Q, self.O, self.dO, self.ws, shape=self.shape, O_lo=self.O_lo, rotary=self.rot,
                                stream=stream)
        if ev is not None:
            ev[2].record(stream)
        esd.attn_bwd_main(self.K, self.V, self.LSE, self.ws, self.dK, self.dV, shape=self.shape, scale=self.scale,
                          rotary=self.rot, stream=stream, **self.mask)
        if ev is not None:
            ev[3].record(stream)
        esd.attn_bwd_finalize(self.ws, self.dQ, shape=self.shape, scale=self.scale, rotary=self.rot, stream=stream)
        if ev is not None:
            ev[4].record(stream)

    def composite(self, stream):
        """The same step through the composite backward call (one call for
        the three stages; with a rotary, one preparation launch for both
        tables and the rotated keys instead of one per stage)."""
        esd = self.esd
        esd.attn_fwd(self.Q, self.K, self.V, scale=self.scale, O=self.O, LSE=self.LSE, O_lo=self.O_lo,
                     rotary=self.rot, workspace=self.fws, stream=stream, **self.mask)
        esd.attn_bwd(self.Q, self.K, self.V, self.O, self.dO, self.LSE, O_lo=self.O_lo, scale=self.scale,
                     dQ=self.dQ, dK=self.dK, dV=self.dV, rotary=self.rot, workspace=self.ws, stream=stream,
                     **self.mask)

    def io_bytes(self):
        """Algorithmic bytes of the two memory-bound backward kernels: one read
        of each input, one write of each output."""
        w, rows = self.w, self.rows
        bhq = w.B * w.Hq
        return {
            "attn_bwd_preprocess_kernel": (rows * w.dv * 2 * 3 + rows * w.dh * 2 + rows * 4 + rows * w.dh * 4
                                           + bhq * ((w.nq + 127) // 128) * 16 + rows * w.dh * 2 + rows * w.dv * 2),
            "attn_bwd_finalize_kernel": rows * w.dh * 4 + rows * w.dh * 2,
        }

    def compulsory_bytes(self):
        """One read of Q, K, V, dO and one write of O, LSE, dQ, dK, dV: the HBM
        floor of a whole fwd+bwd step."""
        return sum(x.numel() * x.element_size() for x in (self.Q, self.K, self.V, self.dO, self.O, self.LSE,
                                                          self.dQ, self.dK, self.dV))


def time_steps(step, stream, dev, steps, flush=None):
    """Per-call CUDA-event times (ms, averaged over `steps`) of `step`; when
    `flush` is given it is written between steps, outside the timed events,
    so that every step starts with a cold L2."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush.add_(1)
        step(stream, evs[k])
    torch.cuda.synchronize(dev)
    per = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / steps for i in range(4)]
    total = sum(e[0].elapsed_time(e[4]) for e in evs) / steps
    return per, total


def config_line(esd, name, dev, steps, warmup, peaks, rotary=False):
    """One configuration timed on its own: per-stage times, TFLOP/s, fraction
    of the measured bf16 burst peak (the stages are timed in sub-second
    regions), and for the tiny single-head case the HBM view and a CUDA-graph
    replay of the step."""
    import torch
    from exact_scaled_dot_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    st = AttnStep(esd, w, make_inputs(w), dev, rotary=rotary)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        st(stream)
    torch.cuda.synchronize(dev)
    small = st.bytes_touched() < 2 * 129e6
    flush = torch.empty((64 * 1024 * 1024,), dtype=torch.float32, device=dev) if small else None
    per, total = time_steps(st, stream, dev, steps, flush)
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    value = (st.flops_fwd + st.flops_bwd) / (total * 1e-3) / 1e12
    out = {"workload": name + ("+rotary" if rotary else ""), "steps": steps, "ms_per_step": total, "tflops": value,
           "frac": value / peak,
           "peak_kind": "bf16_tflops burst", "visible_pairs": st.pairs,
           "l2": "flushed between steps" if small else "inputs larger than L2",
           "stages": {}}
    io = st.io_bytes()
    for stage, ms in zip(KERNEL_STAGES, per):
        ent = {"ms": ms}
        if stage.startswith("attn_fwd"):
            ent["tflops"] = st.flops_fwd / (ms * 1e-3) / 1e12
            ent["frac"] = ent["tflops"] / peak
        elif stage == "attn_bwd_main_kernel":
            ent["tflops"] = st.flops_bwd / (ms * 1e-3) / 1e12
            ent["frac"] = ent["tflops"] / peak
        else:
            ent["gbs"] = io[stage] / (ms * 1e-3) / 1e9
            ent["frac_hbm"] = ent["gbs"] / peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        out["stages"][stage] = ent
    if small:
        # Launch-bound: the HBM floor of the step against its time, and the
        # same step replayed from a CUDA graph (no host work between launches).
        cb = st.compulsory_bytes()
        out["hbm"] = {"compulsory_bytes": cb, "ideal_us": cb / (peaks.get("hbm_gbs", 6800.0) * 1e9) * 1e6,
                      "achieved_gbs": cb / (total * 1e-3) / 1e9}
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                st(side)
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g):
                st(torch.cuda.current_stream(dev))
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ms = 0.0
            for _ in range(steps):
                flush.add_(1)
                a.record(stream)
                g.replay()
                b.record(stream)
                torch.cuda.synchronize(dev)
                ms += a.elapsed_time(b)
            ms /= steps
            out["graph_replay"] = {"ms_per_step": ms, "tflops": (st.flops_fwd + st.flops_bwd) / (ms * 1e-3) / 1e12,
                                   "achieved_gbs": cb / (ms * 1e-3) / 1e9}
        except Exception as e:  # noqa: BLE001 - report, do not fail the line
            out["graph_replay"] = {"error": f"{type(e).__name__}: {e}"}
    status = esd.attn_get_status()
    if status != 0:
        raise RuntimeError(f"{name}: device status {status}: {esd.strerror(status)}")
    del st
    torch.cuda.empty_cache()
    return out


def rotary_cost(esd, name, dev, steps, reps=3):
    """The same workload without and with the fused rotary embedding, each a
    forward and the composite backward call, timed alternately (reps rounds
    of `steps` steps, the fastest round kept): the step-time overhead of
    rotating Q and K inside the calls, with the forward's rotated rows kept
    for the backward (q_rot, k_rot) and without them (the backward rotates
    again)."""
    import torch
    from exact_scaled_dot_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    inp = make_inputs(w)
    stream = torch.cuda.current_stream(dev)
    best = {}
    modes = {"plain": dict(rotary=False), "kept": dict(rotary=True, keep_rotated=True),
             "recomputed": dict(rotary=True)}
    for _ in range(reps):
        for rot, kw in modes.items():
            st = AttnStep(esd, w, inp, dev, **kw)
            for _ in range(3):
                st.composite(stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a.record(stream)
            for _ in range(steps):
                st.composite(stream)
            b.record(stream)
            torch.cuda.synchronize(dev)
            ms = a.elapsed_time(b) / steps
            best[rot] = min(best.get(rot, float("inf")), ms)
            del st
            torch.cuda.empty_cache()
    status = esd.attn_get_status()
    if status != 0:
        raise RuntimeError(f"rotary cost: device status {status}: {esd.strerror(status)}")
    return {"workload": name, "calls": "attn_fwd + attn_bwd (composite)", "steps": steps, "rounds": reps,
            "plain_ms_per_step": best["plain"], "rotary_ms_per_step": best["kept"],
            "overhead": best["kept"] / best["plain"] - 1.0,
            "recomputed_ms_per_step": best["recomputed"],
            "overhead_recomputed": best["recomputed"] / best["plain"] - 1.0,
            "launches_per_step": {"plain": LAUNCHES_PER_STEP, "kept": LAUNCHES_PER_STEP,
                                  "recomputed": LAUNCHES_PER_STEP + 1}}


def run_cuda(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from exact_scaled_dot_gb300 import build as lib_build
    if rank == 0 or world == 1:
        lib_build.build()
    if world > 1:
        torch.distributed.barrier()
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[args.workload]
    if args.batch is not None:
        w = w.scaled(B=args.batch)
    inp = make_inputs(w)
    st = AttnStep(esd, w, inp, dev, rotary=args.rotary)
    kv, mask, scale, shape = st.kv, st.mask, st.scale, st.shape
    off = mask["causal_offset"]
    pairs, flops_fwd, flops_bwd = st.pairs, st.flops_fwd, st.flops_bwd
    ff, fb = flops_per_pair(w.dh, w.dv)
    Q, K, V, dO, O, O_lo, LSE, dQ, dK, dV, ws, fws = st.tensors()
    rows = st.rows
    stream = torch.cuda.current_stream(dev)
    esd.attn_clear_status()

    def step(ev=None):
        st(stream, ev)

    launches_per_step = LAUNCHES_PER_STEP + (3 if args.rotary else 0)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- device-timed region: K steps, inputs resident in HBM ----
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_stop.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_stop)
    status = esd.attn_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {esd.strerror(status)}")

    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(flops_fwd + flops_bwd, world, ms_per_step)

    names = KERNEL_STAGES
    per_kernel = {n: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i, n in enumerate(names)}

    # ---- roofline of the dominant kernel ----
    # Every stage is timed inside a region of well under a second, so the
    # measured burst bf16 peak is the denominator (the sustained one is for
    # seconds-long loops under the power cap).
    peaks, peak_src = load_peaks()
    bytes_io = st.io_bytes()
    dominant = max(per_kernel, key=per_kernel.get)
    if dominant in (names[0], "attn_bwd_main_kernel"):
        work = flops_fwd if dominant == names[0] else flops_bwd
        achieved = work / (per_kernel[dominant] * 1e-3) / 1e12
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": f"bf16_tflops burst ({peak_src})"}
    else:
        achieved = bytes_io[dominant] / (per_kernel[dominant] * 1e-3) / 1e9
        peak = peaks.get("hbm_gbs")
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": f"hbm_gbs ({peak_src})"}
    roof["kernel"] = dominant
    roof["traffic"] = None
    if TRAFFIC_FILE.exists():
        try:
            tr = json.loads(TRAFFIC_FILE.read_text())
            ent = tr.get("kernels", {}).get(dominant)
            if ent and tr.get("source_digest") == source_digest() and tr.get("workload") == w.name:
                roof["traffic"] = ent.get("dram_bytes_per_launch")
        except (OSError, ValueError):
            pass
    kernels = {}
    for n in names:
        ms = per_kernel[n]
        ent = {"ms": ms, "share": ms / sum(per_kernel.values())}
        if n == names[0]:
            ent["tflops"] = flops_fwd / (ms * 1e-3) / 1e12
        elif n == "attn_bwd_main_kernel":
            ent["tflops"] = flops_bwd / (ms * 1e-3) / 1e12
        else:
            ent["gbs"] = bytes_io[n] / (ms * 1e-3) / 1e9
        kernels[n] = ent

    # ---- end to end through the public API, host buffers ----
    # Every step copies its own inputs from pinned host memory, runs the
    # forward and backward through the public calls and reads its results
    # back into pinned host memory.  Steps are pipelined the way a serving or
    # training loop would run them: two device buffer sets, one stream each
    # for uploads, compute and downloads, so that step k+1's upload and step
    # k-1's download overlap step k's kernels (events keep a buffer set from
    # being overwritten before its previous step is done with it).
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.pin_memory()  # noqa: E731
        hQ, hK, hV, hdO = (pin(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
        nbuf = 2
        dsets, hsets = [], []
        for _ in range(nbuf):
            dsets.append({"Q": torch.empty_like(Q), "K": torch.empty_like(K), "V": torch.empty_like(V),
                          "dO": torch.empty_like(dO), "O": torch.empty_like(O), "LSE": torch.empty_like(LSE),
                          "O_lo": torch.empty_like(O_lo), "dQ": torch.empty_like(dQ), "dK": torch.empty_like(dK),
                          "dV": torch.empty_like(dV), "ws": torch.empty_like(ws), "fws": torch.empty_like(fws)})
            hsets.append({k: torch.empty(dsets[-1][k].shape, dtype=dsets[-1][k].dtype).pin_memory()
                          for k in ("O", "LSE", "dQ", "dK", "dV")})
        h2d = sum(x.numel() * x.element_size() for x in (hQ, hK, hV, hdO))
        d2h = sum(x.numel() * x.element_size() for x in hsets[0].values())
        s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]

        def e2e_step(k_step):
            k = k_step % nbuf
            d, hres = dsets[k], hsets[k]
            with torch.cuda.stream(s_in):
                if k_step >= nbuf:
                    s_in.wait_event(ev_cmp[k])       # the set's previous step no longer reads its inputs
                d["Q"].copy_(hQ, non_blocking=True)
                d["K"].copy_(hK, non_blocking=True)
                d["V"].copy_(hV, non_blocking=True)
                d["dO"].copy_(hdO, non_blocking=True)
                ev_in[k].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[k])
                if k_step >= nbuf:
                    s_cmp.wait_event(ev_out[k])      # the set's previous results have been read back
                esd.attn_fwd(d["Q"], d["K"], d["V"], scale=scale, O=d["O"], LSE=d["LSE"], O_lo=d["O_lo"],
                             workspace=d["fws"], stream=s_cmp, **mask)
                esd.attn_bwd(d["Q"], d["K"], d["V"], d["O"], d["dO"], d["LSE"], O_lo=d["O_lo"], scale=scale,
                             dQ=d["dQ"], dK=d["dK"], dV=d["dV"], workspace=d["ws"], stream=s_cmp, **mask)
                ev_cmp[k].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[k])
                for name, t in hres.items():
                    t.copy_(d[name], non_blocking=True)
                ev_out[k].record(s_out)

        for k_step in range(max(nbuf, args.warmup)):
            e2e_step(k_step)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        for k_step in range(args.steps):
            e2e_step(k_step)
        b.record(s_out)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, dev)
        # The last step's results against the device-resident run: O exactly
        # (the forward has no atomics), dQ within the parity tolerance (its
        # fp32 accumulation order differs from run to run).
        last = hsets[(args.steps - 1) % nbuf]
        ref_dq = dQ.float().cpu()
        if not torch.equal(last["O"], O.cpu()) or bool(
                ((last["dQ"].float() - ref_dq).abs() > 1e-2 + 2e-2 * ref_dq.abs()).any()):
            raise RuntimeError("end-to-end results differ from the device-resident run")
        e2e = {"value": job_throughput(flops_fwd + flops_bwd, world, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipeline": "uploads, kernels and downloads of consecutive steps on three streams, two buffer sets"}

    bytes_touched = st.bytes_touched()

    # ---- parity spot check (oracle rows, forward and dQ) and CPU baseline ----
    parity = None
    cpu = None
    if rank == 0 and not args.no_oracle:
        import oracle
        orc = oracle.default()
        p = oracle.Problem(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal, offset=off, kv_len=kv)
        rng = np.random.default_rng(0)
        rsel = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, 30)]))
        f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()  # noqa: E731
        Qn, Kn, Vn, Gn = (f64(x) for x in (inp.Q, inp.K, inp.V, inp.dO))
        rO, rL = orc.forward(p, Qn, Kn, Vn, rows=rsel)
        rdQ, _, _, _, _ = orc.backward(p, Qn, Kn, Vn, Gn, q_rows=rsel, want_dkdv=False)
        # outputs of the last device-timed step
        gO = f64(O).reshape(-1, w.dv)[rsel]
        gL = f64(LSE).reshape(-1)[rsel]
        gQ = f64(dQ).reshape(-1, w.dh)[rsel]
        ok = bool(np.all(np.abs(gO - rO) <= 1e-2 + 2e-2 * np.abs(rO)) and np.all(np.abs(gL - rL) <= 1e-3)
                  and np.all(np.abs(gQ - rdQ) <= 1e-2 + 2e-2 * np.abs(rdQ)))
        parity = {"rows_checked": int(rsel.size), "ok": ok,
                  "max_abs_err": {"O": float(np.max(np.abs(gO - rO))), "LSE": float(np.max(np.abs(gL - rL))),
                                  "dQ": float(np.max(np.abs(gQ - rdQ)))}}
        v, desc, threads, _dt = oracle_cpu_sample(w, inp, args.cpu_rows)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}

    # ---- the other configurations, each timed on its own after the headline ----
    configs = None
    if not args.no_configs and args.batch is None:
        from exact_scaled_dot_gb300.inputs import WORKLOAD_ORDER
        del st, Q, K, V, dO, O, LSE, O_lo, dQ, dK, dV, ws, fws
        torch.cuda.empty_cache()
        configs = {}
        for name in WORKLOAD_ORDER:
            if name == w.name:
                continue
            configs[name] = config_line(esd, name, dev, args.config_steps, 3, peaks)
        configs["rotary_cost"] = rotary_cost(esd, w.name, dev, args.config_steps)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) draws rounded to bf16; random key lengths)",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "n_q": w.nq, "n_k": w.nk,
                       "d_h": w.dh, "d_v": w.dv, "causal": w.causal, "kv_len": kv, "seed": w.seed,
                       "rotary": bool(args.rotary),
                       "visible_pairs": pairs, "flops_per_step": flops_fwd + flops_bwd,
                       # The backward's five products cost 2(3 d_h + 2 d_v) per pair; the metric counts
                       # 2(2 d_h + 3 d_v).  Equal for d_h = d_v.
                       "tflops_five_product_count": job_throughput(pairs * (ff + 2 * (3 * w.dh + 2 * w.dv)), world,
                                                                   ms_per_step),
                       "arithmetic": "bf16 inputs and outputs; Q K^T in bf16, P V and every backward product in "
                                     "fp16 (exact re-encoding of the bf16 operands), fp32 accumulation",
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (about %.0f MB touched per step)" % (bytes_touched / 1e6)},
            "peak_fraction": value / world / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
            "roofline": roof,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "parity": parity,
            "configs": configs,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_decode(args):
    """Short query blocks over a long key cache (attn_fwd_decode): forward
    only, HBM-bound, so the metric is the K/V cache streamed per second
    (every visible key row read once, plus Q in and O, O_lo, LSE out) against
    the measured copy bandwidth.  The regular forward is timed on the same
    inputs for comparison, and sampled rows are checked against the oracle."""
    import torch
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300 import build as lib_build
    from exact_scaled_dot_gb300.inputs import WORKLOADS, make_inputs

    lib_build.build()
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    kv = inp.kv_len.tolist() if inp.kv_len is not None else [w.nk] * w.B
    mask = dict(causal=w.causal, causal_offset=w.causal_offset if w.causal else None, kv_len=kv)
    Q, K, V = (x.to(dev) for x in (inp.Q, inp.K, inp.V))
    O = torch.empty((w.B, w.Hq, w.nq, w.dv), dtype=torch.bfloat16, device=dev)
    LSE = torch.empty((w.B, w.Hq, w.nq), dtype=torch.float32, device=dev)
    O_lo = torch.empty_like(O)
    need = esd.attn_fwd_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, **mask)
    ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    esd.attn_clear_status()
    # Visible key rows per (batch, KV head): those below the last query's limit.
    rows_read = sum(min(L, w.nk, (w.nq - 1 + w.causal_offset + 1) if w.causal else w.nk) for L in kv) * w.Hkv
    bytes_step = (rows_read * (w.dh + w.dv) * 2 + Q.numel() * 2 + O.numel() * 2 * 2 + LSE.numel() * 4)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / steps

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    ms = timed(lambda: esd.attn_fwd_decode(Q, K, V, O=O, LSE=LSE, O_lo=O_lo, workspace=ws, **mask), args.steps)
    clocks = sampler.stop()
    status = esd.attn_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {esd.strerror(status)}")
    fws = torch.empty((esd.attn_fwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv),), dtype=torch.uint8,
                      device=dev)
    ms_regular = timed(lambda: esd.attn_fwd(Q, K, V, O=O, LSE=LSE, O_lo=O_lo, workspace=fws, **mask),
                       max(5, args.steps // 4))
    esd.attn_fwd_decode(Q, K, V, O=O, LSE=LSE, O_lo=O_lo, workspace=ws, **mask)
    torch.cuda.synchronize(dev)

    parity = None
    if not args.no_oracle:
        import numpy as np
        import oracle
        orc = oracle.default()
        p = oracle.Problem(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, causal=w.causal,
                           offset=w.causal_offset if w.causal else None, kv_len=kv)
        rng = np.random.default_rng(0)
        rows = np.sort(rng.choice(w.B * w.Hq * w.nq, size=min(16, w.B * w.Hq * w.nq), replace=False))
        Oref, Lref = orc.forward(p, inp.Q.double().numpy(), inp.K.double().numpy(), inp.V.double().numpy(),
                                 rows=rows)
        Og = O.double().cpu().numpy().reshape(-1, w.dv)[rows]
        Lg = LSE.double().cpu().numpy().reshape(-1)[rows]
        okO = bool(np.all(np.abs(Og - Oref) <= 1e-2 + 2e-2 * np.abs(Oref)))
        okL = bool(np.all(np.abs(Lg - Lref) <= 1e-3))
        parity = {"rows_checked": int(len(rows)), "ok": okO and okL,
                  "max_abs_err": {"O": float(np.abs(Og - Oref).max()), "LSE": float(np.abs(Lg - Lref).max())}}

    peaks, peak_src = load_peaks()
    gbs = bytes_step / (ms * 1e-3) / 1e9
    # Work: visible pairs x 2 (d_h + d_v).  A packed tile of many query rows
    # per KV head (a chunk over MQA) does enough arithmetic per cache byte to
    # be bound by the tensor core instead; the roofline takes whichever
    # bound is further away.
    pairs = esd.attn_visible_pairs(w.B, w.Hq, w.Hkv, w.nq, w.nk, w.dh, w.dv, **mask)
    flops = pairs * 2 * (w.dh + w.dv)
    tflops = flops / (ms * 1e-3) / 1e12
    t_hbm = bytes_step / (peaks.get("hbm_gbs") * 1e9)
    t_tensor = flops / (peaks.get("bf16_tflops") * 1e12)
    if t_tensor > t_hbm:
        roofline = {"bound": "tensor", "achieved": tflops, "peak": peaks.get("bf16_tflops"), "unit": "TFLOP/s",
                    "frac": tflops / peaks.get("bf16_tflops"), "peak_kind": f"bf16_tflops burst ({peak_src})"}
    else:
        roofline = {"bound": "hbm", "achieved": gbs, "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                    "frac": gbs / peaks.get("hbm_gbs"), "peak_kind": f"hbm_gbs ({peak_src})"}
    roofline.update({"kernel": "attn_decode_kernel + merge", "traffic": None,
                     "intensity_flop_per_byte": flops / bytes_step})
    line = {
        "metric": "short-query attention forward, K/V cache streamed (GB/s)", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) draws rounded to bf16)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "n_q": w.nq, "n_k": w.nk, "d_h": w.dh,
                   "d_v": w.dv, "causal": w.causal, "kv_len": kv, "bytes_per_step": bytes_step,
                   "l2": "K/V cache larger than L2"},
        "roofline": roofline, "tflops": tflops, "visible_pairs": pairs,
        "regular_forward": {"ms_per_step": ms_regular, "gbs": bytes_step / (ms_regular * 1e-3) / 1e9},
        "clocks": clocks, "parity": parity, "gpu_launches": 2 * args.steps if need > 0 else args.steps,
    }
    print(json.dumps(line))
    return 0


def run_varlen(args):
    """Packed variable-length sequences (attn_fwd_varlen + attn_bwd_varlen):
    one step is the forward and the backward over the whole packed batch;
    the metric counts visible pairs like the padded workloads.  Sampled rows
    of two sequences are checked against the oracle (run per sequence)."""
    import numpy as np
    import torch
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300 import build as lib_build
    from exact_scaled_dot_gb300.inputs import VARLEN_WORKLOADS, make_varlen_inputs

    lib_build.build()
    w = VARLEN_WORKLOADS[args.workload]
    inp = make_varlen_inputs(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    Q, K, V, dO = (x.to(dev) for x in (inp.Q, inp.K, inp.V, inp.dO))
    Tq, Tk = Q.shape[0], K.shape[0]
    O = torch.empty((Tq, w.Hq, w.dv), dtype=torch.bfloat16, device=dev)
    O_lo = torch.empty_like(O)
    LSE = torch.empty((w.Hq, Tq), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    need = esd.attn_bwd_varlen_workspace_bytes(w.Hq, w.Hkv, w.dh, w.dv, inp.cu_q, inp.cu_k, causal=w.causal)
    ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    fneed = esd.attn_fwd_varlen_workspace_bytes(w.Hq, w.Hkv, w.dh, w.dv, inp.cu_q, inp.cu_k, causal=w.causal)
    fws = torch.empty((max(fneed, 256),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    pairs = esd.attn_varlen_visible_pairs(w.Hq, w.Hkv, w.dh, w.dv, inp.cu_q, inp.cu_k, causal=w.causal)
    flops_fwd = pairs * 2 * (w.dh + w.dv)
    flops_bwd = pairs * 2 * (2 * w.dh + 3 * w.dv)
    esd.attn_clear_status()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        esd.attn_fwd_varlen(Q, K, V, inp.cu_q, inp.cu_k, causal=w.causal, O=O, LSE=LSE, O_lo=O_lo, workspace=fws)
        if ev is not None:
            ev[1].record(stream)
        esd.attn_bwd_varlen(Q, K, V, O, dO, LSE, inp.cu_q, inp.cu_k, O_lo=O_lo, causal=w.causal, dQ=dQ, dK=dK,
                            dV=dV, workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for k in range(args.steps):
        step(evs[k])
    b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    status = esd.attn_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {esd.strerror(status)}")
    ms = a.elapsed_time(b) / args.steps
    ms_fwd = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    ms_bwd = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    tflops = (flops_fwd + flops_bwd) / (ms * 1e-3) / 1e12

    parity = None
    if not args.no_oracle:
        import oracle
        orc = oracle.default()
        rng = np.random.default_rng(0)
        order = np.argsort(inp.lens_q)
        checks, ok, errs = 0, True, {"O": 0.0, "LSE": 0.0, "dQ": 0.0}
        for bi in (int(order[0]), int(order[-1])):
            lq, lk = inp.lens_q[bi], inp.lens_k[bi]
            q0, q1, k0, k1 = inp.cu_q[bi], inp.cu_q[bi + 1], inp.cu_k[bi], inp.cu_k[bi + 1]
            p = oracle.Problem(1, w.Hq, w.Hkv, lq, lk, w.dh, w.dv, causal=w.causal)
            f = lambda x: np.ascontiguousarray(x.double().numpy().transpose(1, 0, 2)[None])  # noqa: E731
            Qb, Kb, Vb, Gb = f(inp.Q[q0:q1]), f(inp.K[k0:k1]), f(inp.V[k0:k1]), f(inp.dO[q0:q1])
            rows = np.sort(rng.choice(w.Hq * lq, size=min(8, w.Hq * lq), replace=False))
            Oref, Lref = orc.forward(p, Qb, Kb, Vb, rows=rows)
            dQref, _dK, _dV, _D, _C = orc.backward(p, Qb, Kb, Vb, Gb, q_rows=rows, want_dkdv=False)
            h, i = rows // lq, rows % lq
            Og = O[q0:q1].double().cpu().numpy()[i, h]
            Lg = LSE[:, q0:q1].double().cpu().numpy()[h, i]
            dQg = dQ[q0:q1].double().cpu().numpy()[i, h]
            ok &= bool(np.all(np.abs(Og - Oref) <= 1e-2 + 2e-2 * np.abs(Oref)))
            ok &= bool(np.all(np.abs(Lg - Lref) <= 1e-3))
            ok &= bool(np.all(np.abs(dQg - dQref) <= 1e-2 + 2e-2 * np.abs(dQref)))
            errs = {"O": max(errs["O"], float(np.abs(Og - Oref).max())),
                    "LSE": max(errs["LSE"], float(np.abs(Lg - Lref).max())),
                    "dQ": max(errs["dQ"], float(np.abs(dQg - dQref).max()))}
            checks += len(rows)
        parity = {"rows_checked": checks, "ok": ok, "max_abs_err": errs}

    peaks, peak_src = load_peaks()
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) draws rounded to bf16, drawn sequence lengths)",
        "config": {"workload": w.name, "sequences": len(inp.lens_q), "Hq": w.Hq, "Hkv": w.Hkv, "d_h": w.dh,
                   "d_v": w.dv, "causal": w.causal, "tokens": Tq, "lens": inp.lens_q, "visible_pairs": pairs,
                   "l2": "inputs larger than L2"},
        "kernels": {"forward": {"ms": ms_fwd}, "backward (preprocess + main + finalize)": {"ms": ms_bwd}},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks.get("bf16_tflops"), "unit": "TFLOP/s",
                     "frac": tflops / peaks.get("bf16_tflops"), "peak_kind": f"bf16_tflops burst ({peak_src})",
                     "traffic": None},
        "clocks": clocks, "parity": parity, "gpu_launches": 6 * args.steps,
    }
    print(json.dumps(line))
    return 0


def run_proj(args):
    """The projections on either side of attention (A.10.10-A.10.11) at the
    GQA workload's shapes: one step is the three forward products
    Q, K, V = X W_Q, X W_K, X W_V, the three weight gradients X^T G and the
    input gradient sum_s G_s W_s^T.  Dense products: TFLOP/s against the
    measured bf16 peak."""
    import numpy as np
    import torch
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300 import build as lib_build
    from exact_scaled_dot_gb300.inputs import PROJ_WORKLOADS, make_proj_inputs

    lib_build.build()
    cfg = PROJ_WORKLOADS[args.workload]
    T, D, Ns = cfg["T"], cfg["D"], cfg["Ns"]
    inp = make_proj_inputs(T, D, Ns, cfg["seed"])
    dev = torch.device("cuda", torch.cuda.current_device())
    X = inp.X.to(dev)
    Ws = [w.to(dev) for w in inp.Ws]
    Gs = [g.to(dev) for g in inp.Gs]
    Ys = [torch.empty((T, n), dtype=torch.bfloat16, device=dev) for n in Ns]
    dWs = [torch.empty((D, n), dtype=torch.float32, device=dev) for n in Ns]
    dX = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops_each = 2 * T * D * sum(Ns)
    esd.attn_clear_status()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for W, Y in zip(Ws, Ys):
            esd.attn_proj_fwd(X, W, Y=Y)
        if ev is not None:
            ev[1].record(stream)
        for G, dW in zip(Gs, dWs):
            esd.attn_proj_bwd_weight(X, G, dW=dW)
        if ev is not None:
            ev[2].record(stream)
        esd.attn_proj_bwd_input(Gs, Ws, dX=dX)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for k in range(args.steps):
        step(evs[k])
    b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    status = esd.attn_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {esd.strerror(status)}")
    ms = a.elapsed_time(b) / args.steps
    part = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i in range(3)]
    tflops = 3 * flops_each / (ms * 1e-3) / 1e12
    parity = None
    if not args.no_oracle:
        rng = np.random.default_rng(0)
        rows = rng.integers(0, T, 8)
        Xn = inp.X.double().numpy()
        ok, err = True, 0.0
        for k in range(3):
            ref = Xn[rows] @ inp.Ws[k].double().numpy()
            got = Ys[k].double().cpu().numpy()[rows]
            ok &= bool(np.all(np.abs(got - ref) <= 1e-2 + 2e-2 * np.abs(ref)))
            err = max(err, float(np.abs(got - ref).max()))
        ref = sum(inp.Gs[k].double().numpy()[rows] @ inp.Ws[k].double().numpy().T for k in range(3))
        got = dX.double().cpu().numpy()[rows]
        ok &= bool(np.all(np.abs(got - ref) <= 1e-2 + 2e-2 * np.abs(ref)))
        parity = {"rows_checked": int(len(rows)), "ok": ok,
                  "max_abs_err": max(err, float(np.abs(got - ref).max()))}
    peaks, peak_src = load_peaks()
    line = {
        "metric": "projections on either side of attention, fwd + bwd TFLOP/s", "value": tflops,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) draws, weights N(0,1/D), rounded to bf16)",
        "config": {"workload": args.workload, "T": T, "D": D, "N": list(Ns), "l2": "inputs larger than L2"},
        "kernels": {"X W (3 products)": {"ms": part[0], "tflops": flops_each / (part[0] * 1e-3) / 1e12},
                    "X^T G (3 products)": {"ms": part[1], "tflops": flops_each / (part[1] * 1e-3) / 1e12},
                    "sum G W^T": {"ms": part[2], "tflops": flops_each / (part[2] * 1e-3) / 1e12}},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks.get("bf16_tflops"), "unit": "TFLOP/s",
                     "frac": tflops / peaks.get("bf16_tflops"), "peak_kind": f"bf16_tflops burst ({peak_src})",
                     "kernel": "proj_gemm_kernel", "traffic": None},
        "clocks": clocks, "parity": parity, "gpu_launches": 7 * args.steps,
    }
    print(json.dumps(line))
    return 0


def run_rope(args):
    """Rotary embedding of the GQA workload's queries and keys (8192 tokens,
    32 + 8 heads of 128) in one launch: memory-bound, GB/s of rows read and
    written against the measured copy bandwidth; the inverse (gradient) pass
    is the same kernel."""
    import numpy as np
    import torch
    import exact_scaled_dot_gb300 as esd
    from exact_scaled_dot_gb300 import build as lib_build

    lib_build.build()
    T, Hq, Hkv, d = 8192, 32, 8, 128
    g = torch.Generator().manual_seed(1401)
    dev = torch.device("cuda", torch.cuda.current_device())
    Q = torch.randn((T, Hq, d), generator=g).to(torch.bfloat16).to(dev)
    K = torch.randn((T, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    pos = (torch.arange(T, dtype=torch.int32) % 4096).to(dev)
    Qr, Kr = torch.empty_like(Q), torch.empty_like(K)
    stream = torch.cuda.current_stream(dev)
    esd.attn_clear_status()

    def step():
        esd.attn_rope_qk(Q, K, pos, Yq=Qr, Yk=Kr)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if esd.attn_get_status() != 0:
        raise RuntimeError("device status set")
    ms = a.elapsed_time(b) / args.steps
    nbytes = 2 * (Q.numel() + K.numel()) * 2 + T * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    parity = None
    if not args.no_oracle:
        from oracle.rope import rope
        rows = np.random.default_rng(0).integers(0, T, 16)
        ref = np.concatenate([rope(X[rows].double().cpu().numpy(), pos[rows].cpu().numpy()).reshape(16, -1)
                              for X in (Q, K)], axis=1)
        got = np.concatenate([Y[rows].double().cpu().numpy().reshape(16, -1) for Y in (Qr, Kr)], axis=1)
        parity = {"rows_checked": 16, "ok": bool(np.all(np.abs(got - ref) <= 1e-2 + 2e-2 * np.abs(ref))),
                  "max_abs_err": float(np.abs(got - ref).max())}
    peaks, peak_src = load_peaks()
    line = {
        "metric": "rotary embedding of queries and keys (GB/s)", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) draws rounded to bf16)",
        "config": {"workload": "rope_gqa", "tokens": T, "Hq": Hq, "Hkv": Hkv, "d": d, "bytes_per_step": nbytes},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                     "frac": gbs / peaks.get("hbm_gbs"), "peak_kind": f"hbm_gbs ({peak_src})", "kernel": "rope_kernel",
                     "traffic": None},
        "clocks": clocks, "parity": parity, "gpu_launches": args.steps,
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller cases for profiling)")
    ap.add_argument("--cpu-rows", type=int, default=768, help="query rows in the timed oracle sample")
    ap.add_argument("--reference-rows", type=int, default=384, help="query rows per reference-arm step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-oracle", action="store_true", help="skip the parity spot check and CPU baseline")
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other configurations")
    ap.add_argument("--rotary", action="store_true",
                    help="headline step with the rotary embedding fused into the calls")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps per other configuration")
    args = ap.parse_args(argv)
    if args.warmup < 0 or args.steps < 1:
        ap.error("need --steps >= 1 and --warmup >= 0")
    if args.impl == "reference":
        return run_reference(args)
    from exact_scaled_dot_gb300.inputs import DECODE_WORKLOADS, PROJ_WORKLOADS, VARLEN_WORKLOADS
    if args.workload in DECODE_WORKLOADS:
        return run_decode(args)
    if args.workload in VARLEN_WORKLOADS:
        return run_varlen(args)
    if args.workload in PROJ_WORKLOADS:
        return run_proj(args)
    if args.workload == "rope_gqa":
        return run_rope(args)
    return run_cuda(args)


if __name__ == "__main__":
    sys.exit(main())
