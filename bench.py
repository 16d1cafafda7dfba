#!/usr/bin/env python3
"""Benchmark of the SSD forward pass (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 27b|sweep:B:L:S|long|varlen|varlen_states|tiny|decode[:B]|bwd[:B]|gatenorm]

A step is one ssd_fwd call over one batch of the workload.  The default is
the largest single-GPU configuration, one 65,536-token sequence with 32 heads
(P 64, N 128, bf16, split length 2048, initial and final states); the same
run then measures the other points of the tokens/s-vs-L curve (the 2.7B-like
layer, the 16,384-token sweep at every (batch, L) and split length, the
packed-document case) and reports them under "vs_L" in the same JSON line
(--no-sweep skips them).  Inputs are synthetic (seeded), resident in HBM
before timing; L2 is flushed (a 256 MiB write) before every timed step.  Under torchrun each rank runs its
own copy of the workload (independent batch rows: weak scaling) and rank 0
reports the aggregate over ranks with the slowest rank's time.

--impl reference times the fp64 CPU oracle recurrence on the host cores on a
bounded sample of the same workload (one batch row, at most 16,384 tokens of
it, per step).

--workload decode[:B] times the single-token decode step (ssd_step) of the
same layer shape over a batch of B rows (default 256) from a resident state;
--workload bwd[:B] times the backward pass (ssd_bwd) of the 2.7B-like layer
(batch B, default 8); --workload gatenorm the gated RMS norm of its output.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from mamba_ssd_chunked_scan_gb300 import synth  # noqa: E402

METRIC = "SSD fwd tokens/s and achieved HBM GB/s (% of GB300 roofline) vs L, 1 GPU"
# the headline: the largest single-GPU forward configuration (65,536 tokens of
# one sequence, 32 heads, split length 2048, initial and final states)
DEFAULT_WORKLOAD = "long"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0   # dense bf16, burst


DECODE_METRIC = "SSD decode step tokens/s and achieved HBM GB/s on the resident state, 1 GPU"
GATE_NORM_METRIC = "gated RMS norm of the scan output, tokens/s and achieved HBM GB/s, 1 GPU"
BWD_METRIC = "SSD bwd tokens/s and achieved TFLOP/s against the kernel's peak, 1 GPU"
# fp32 CUDA-core peak: 152 SMs x 128 fp32 lanes x 2 flop (FMA) x 2.07 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def bwd_flops(p, Qb=32) -> float:
    """Algorithmic flops of ssd_bwd (2 per multiply-add): per token and head,
    2PN (chunk-entry states and the adjoint carry) + Qb (N + P) / 2 (C B^T and
    dy x^T, lower triangle) + P (2N + Qb / 2) (dx: Lam B, S_in C, the masked
    sum) + N (2P + Qb) (dB and dC)."""
    P, N = p.headdim, p.dstate
    mac = 2 * P * N + Qb * (N + P) / 2 + P * (2 * N + Qb / 2) + N * (2 * P + Qb)
    return 2.0 * mac * p.batch * p.seqlen * p.nheads


def bwd_uses_tensor_cores(p) -> bool:
    """ssd_bwd runs on the tensor cores for the bf16 Mamba-2 head shape."""
    return p.dtype == "bf16" and p.headdim == 64 and p.dstate == 128


def bwd_tc_flops(p, Q=128) -> float:
    """Algorithmic flops of the tensor-core backward's contractions (2 per
    multiply-add, the causal lower triangles only): per token and head, 6PN
    (the chunk-entry states, B Lam^T, C S_in^T, the two state terms of dB and
    dC, the adjoint update) + Q (3N/2 + P) (C B^T, dy x^T, (L o G)^T dy and the
    masked products of dB and dC)."""
    P, N = p.headdim, p.dstate
    mac = 6 * P * N + Q * (1.5 * N + P)
    return 2.0 * mac * p.batch * p.seqlen * p.nheads


def workload(name: str):
    if name.startswith("decode"):
        parts = name.split(":")
        return synth.config_decode(int(parts[1]) if len(parts) > 1 else 256)
    if name == "bwd_long":
        return synth.config_long()
    if name == "bwd_varlen_states":
        return synth.config_varlen(init_std=0.2)
    if name.startswith("bwd"):
        parts = name.split(":")
        return synth.config_27b(batch=int(parts[1]) if len(parts) > 1 else 8)
    if name in ("27b", "gatenorm"):
        return synth.config_27b()
    if name == "tiny":
        return synth.config_tiny_f32()
    if name == "long":
        return synth.config_long()
    if name == "varlen":
        return synth.config_varlen()
    if name == "varlen_states":
        return synth.config_varlen(init_std=0.2)
    if name.startswith("sweep"):
        _, b, L, s = name.split(":")
        return synth.config_sweep(int(b), int(L), int(s))
    raise ValueError(name)


def compulsory_bytes(p) -> int:
    """x + dt + B + C + y, and with initial states also those and the final
    states (which the bench then asks for): the bytes the operator must move
    at least once."""
    e = 2 if p.dtype == "bf16" else 4
    T = p.batch * p.seqlen
    nb = T * (2 * p.nheads * p.headdim * e + p.nheads * 4 + 2 * p.ngroups * p.dstate * e)
    if p.initial_states is not None:
        nb += 2 * p.nstates * p.nheads * p.headdim * p.dstate * 4
    return nb


def decode_bytes(p) -> int:
    """State read and write, x, y, dt, B and C of one decode step."""
    e = 2 if p.dtype == "bf16" else 4
    bh = p.batch * p.nheads
    return bh * (2 * p.headdim * p.dstate * 4 + 2 * p.headdim * e + 4) + p.batch * p.ngroups * 2 * p.dstate * e


def bf16_peak():
    """Dense bf16 tensor TFLOP/s for a kernel timed alone (the burst figure)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            if "bf16_tflops" in d:
                return float(d["bf16_tflops"]), "measured (cuBLAS bf16 GEMM, burst)"
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def slowest_rank(times, device):
    """Each timing's maximum over the ranks of the process group (the job is as
    fast as its slowest rank); the local values when there is no group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(times), dtype=torch.float64, device=device)
    if dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
    return [float(v) for v in t]


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time per step (weak scaling: each rank runs its own copy)."""
    return world * units_per_rank / (ms / 1e3)


def device_copy_gbps(dev, stream, nbytes=1 << 30, reps=5):
    """Context only: a 1 GiB device-to-device copy (read + write bytes over its
    CUDA-event time, best of `reps`), the copy bandwidth of this GPU now."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    dst.copy_(src)
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src)
        b.record(stream)
        b.synchronize()
        best = max(best, 2 * nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
    del src, dst
    return best


def tail_pieces(p, nsm):
    """Pieces with an incoming state under the leftover-unit plan (one split):
    the last U % S units are cut into m pieces, all but the first of each
    continue a sequence."""
    units = p.batch * p.nheads
    T = units % nsm
    nch = (p.seqlen + p.chunk - 1) // p.chunk
    if units < nsm or T == 0 or nch < 4:
        return 0
    m = min(nsm // T, 8, nch // 2)
    while m >= 2 and T * m * p.headdim * p.dstate * 4 > (4 << 20):
        m -= 1
    if m < 2:
        return 0
    split = (nch + m - 1) // m * p.chunk
    m = (p.seqlen + split - 1) // split
    return T * (m - 1)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# the sources that define each kernel family's device code and launch
FAMILY_SOURCES = {1: ("ssd_tc.cu", "tc_ptx.cuh", "ssd_common.cuh", "segsum.cuh", "ssd_kernels.h"),
                  0: ("ssd_simt.cu", "segsum.cuh", "ssd_common.cuh", "ssd_kernels.h")}


def kernel_sources_sha(family: int) -> str:
    """Fingerprint of the CUDA sources of one kernel family (to tell whether a
    recorded counter still belongs to the kernel being timed)."""
    csrc = os.path.join(ROOT, "mamba_ssd_chunked_scan_gb300", "csrc")
    h = hashlib.sha256()
    for name in FAMILY_SOURCES[family]:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(family: int, workload: str):
    """DRAM bytes per launch of the dominant kernel (the full pass) on this
    workload, from the committed ncu summary, used only while the kernel
    source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        ent = json.load(open(path)).get(f"{family}:{workload}")
        if not ent:
            return None
        return ent["dram_bytes_per_launch"] if kernel_sources_sha(family) == ent["source_sha"] else None
    except Exception:
        return None


def oracle_decode(p, rows):
    import oracle
    return oracle.ssd_step(p.initial_states[:rows], p.x[:rows, 0], p.dt[:rows, 0], p.A, p.B[:rows, 0],
                           p.C[:rows, 0], p.D)


def run_reference(args):
    import oracle
    rank, _, world = dist_env()
    if rank != 0:
        return
    p = workload(args.workload)
    if args.workload == "gatenorm":
        rows, width = 1024, p.nheads * p.headdim
        rng = np.random.default_rng(13)
        y = synth.bf16_to_f32(synth.bf16_bits(rng.standard_normal((rows, width)).astype(np.float32)))
        z = synth.bf16_to_f32(synth.bf16_bits(rng.standard_normal((rows, width)).astype(np.float32)))
        w = rng.uniform(0.5, 1.5, width)
        for _ in range(args.warmup):
            oracle.gate_norm(y, z, w, width, 1e-5)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle.gate_norm(y, z, w, width, 1e-5)
            times.append(time.perf_counter() - t0)
        ms = 1e3 * sum(times) / len(times)
        value = rows / (ms / 1e3)
        print(json.dumps({
            "impl": "reference", "metric": GATE_NORM_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"gate_norm_width{width}", "sample": f"{rows} rows per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"fp64 numpy gate and norm of {rows} rows of {width} channels"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    if args.workload.startswith("bwd"):
        dy_h = np.random.default_rng(11).standard_normal((p.batch, p.seqlen, p.nheads, p.headdim)).astype(np.float32)
        q, dyq = bwd_sample(p, dy_h)
        for _ in range(args.warmup):
            oracle.ssd_backward(q, dyq)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle.ssd_backward(q, dyq)
            times.append(time.perf_counter() - t0)
        ms = 1e3 * sum(times) / len(times)
        value = q.seqlen / (ms / 1e3)
        print(json.dumps({
            "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "bwd_" + p.name, "sample": f"batch row 0, {q.seqlen} tokens per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"fp64 reverse-mode recurrence on batch row 0, {q.seqlen} tokens"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    if p.seqlen == 1:
        rows = min(p.batch, 64)
        for _ in range(args.warmup):
            oracle_decode(p, rows)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle_decode(p, rows)
            times.append(time.perf_counter() - t0)
        ms = 1e3 * sum(times) / len(times)
        value = rows / (ms / 1e3)
        sample = f"fp64 decode step of batch rows 0..{rows - 1} of {p.name} per step"
        print(json.dumps({
            "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": p.name, "sample": f"{rows} of {p.batch} batch rows per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    # bounded sample: one batch row of the workload per step, at most 16,384 tokens of it
    T = p.seqlen if p.cu_seqlens is not None else min(p.seqlen, 16384)
    q = synth.SSDProblem(1, T, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0,
                         p.dtype, p.x[:1, :T].copy(), p.dt[:1, :T].copy(), p.A, p.B[:1, :T].copy(),
                         p.C[:1, :T].copy(), p.D,
                         None if p.initial_states is None else p.initial_states[:1].copy(), p.cu_seqlens,
                         p.name)
    for _ in range(args.warmup):
        oracle.ssd_recurrence(q, want_final=p.initial_states is not None)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ssd_recurrence(q, want_final=p.initial_states is not None)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    tok = q.batch * q.seqlen
    value = tok / (ms / 1e3)
    cores = oracle.max_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": p.name, "sample": f"batch row 0 of {p.batch}, tokens 0..{T - 1}, per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"fp64 sequential recurrence, batch row 0 (tokens 0..{T - 1}) of "
                                       f"{p.name} per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(p):
    """The oracle beside the GPU number: all cores on a bounded sample (batch
    row 0, at most 16,384 tokens), and one thread on its first 2,048 tokens."""
    import oracle
    r = oracle_rate(p, seconds=10.0)
    T = min(p.seqlen, 2048) if p.cu_seqlens is None else p.seqlen
    q = synth.SSDProblem(1, T, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0,
                         p.dtype, p.x[:1, :T].copy(), p.dt[:1, :T].copy(), p.A, p.B[:1, :T].copy(),
                         p.C[:1, :T].copy(), p.D, None, p.cu_seqlens, p.name)
    t0 = time.perf_counter()
    oracle.ssd_recurrence(q, want_final=False, nthreads=1)
    r["single_thread_value"] = T / (time.perf_counter() - t0)
    r["single_thread_sample"] = f"batch row 0, tokens 0..{T - 1}, one thread"
    return r


def run_decode(args, p, dev, rank, local_rank, world):
    """Decode workload: a step is one ssd_step over the whole batch (one new
    token per row), the state resident in HBM and updated in place."""
    import torch
    import torch.distributed as dist
    import mamba_ssd_chunked_scan_gb300 as ssd

    def io(name):
        return torch.from_numpy(p.storage(name)[:, 0].view(np.int16).copy()).to(dev).view(torch.bfloat16)

    x, B, C = io("x"), io("B"), io("C")
    dt = torch.from_numpy(p.dt[:, 0].copy()).to(dev)
    A = torch.from_numpy(p.A).to(dev)
    D = torch.from_numpy(p.D).to(dev)
    state = torch.from_numpy(p.initial_states).to(dev)
    y = torch.empty_like(x)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(xx=x, dd=dt, bb=B, cc=C, yy=y):
        ssd.ssd_step(state, xx, dd, A, bb, cc, D, y=yy, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps

    # end to end: each step's token inputs come from pinned host memory and its
    # y goes back; the state stays resident on the device between steps
    hx, hB, hC, hdt = (t.cpu().pin_memory() for t in (x, B, C, dt))
    hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hx, hB, hC, hdt))
    d2h = hy.numel() * hy.element_size()
    dx, dB, dC, ddt = (torch.empty_like(t) for t in (x, B, C, dt))

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dB.copy_(hB, non_blocking=True)
        dC.copy_(hC, non_blocking=True)
        ddt.copy_(hdt, non_blocking=True)
        step(dx, ddt, dB, dC, y)
        hy.copy_(y, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps

    ms_max, e2e_max = slowest_rank([ms, e2e_ms], dev)
    if rank == 0:
        nbytes = decode_bytes(p)
        peak, peak_kind = peaks()
        achieved = nbytes / (ms / 1e3) / 1e9
        line = {
            "metric": DECODE_METRIC, "value": job_rate(p.batch, world, ms_max), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": p.name, "batch": p.batch, "nheads": p.nheads, "headdim": p.headdim,
                       "dstate": p.dstate, "ngroups": p.ngroups, "storage": p.dtype, "kernel": "ssd_step",
                       "l2": "256 MiB write before every timed step; the state is larger than L2",
                       "bytes_per_step": nbytes, "achieved_GBps": achieved},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind, "traffic": None,
                         "scope": "state read + write, x, y, dt, B, C of one ssd_step launch"},
            "e2e": {"value": job_rate(p.batch, world, e2e_max), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
        }
        if world == 1 and not args.no_cpu_baseline:
            rows = min(p.batch, 64)
            reps, t_all = 0, 0.0
            while t_all < 5.0 and reps < 200:
                t0 = time.perf_counter()
                oracle_decode(p, rows)
                t_all += time.perf_counter() - t0
                reps += 1
            import oracle
            line["cpu_baseline"] = {"value": rows * reps / t_all, "unit": "tokens/s", "cores": oracle.max_threads(),
                                    "kind": "oracle",
                                    "sample": f"fp64 decode step of {rows} batch rows of {p.name}, {reps} passes"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_gate_norm(args, p, dev, rank, local_rank, world):
    """Gate/norm workload: a step is one ssd_gate_norm over the 2.7B-like layer's
    scan output (batch x L tokens, 5120 channels normalised as one group)."""
    import torch
    import mamba_ssd_chunked_scan_gb300 as ssd

    rows, width = p.batch * p.seqlen, p.nheads * p.headdim
    rng = np.random.default_rng(13)

    def io(a):
        return torch.from_numpy(synth.bf16_bits(a).view(np.int16).copy()).to(dev).view(torch.bfloat16)

    y = io(rng.standard_normal((rows, width)).astype(np.float32))
    z = io(rng.standard_normal((rows, width)).astype(np.float32))
    w = torch.from_numpy(rng.uniform(0.5, 1.5, width).astype(np.float32)).to(dev)
    out = torch.empty_like(y)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        ssd.gate_norm(y, z, w, width, out=out, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            ssd.gate_norm(y, z, w, width, out=out, stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    # end to end: y and z from pinned host memory, out back to it
    hy, hz = y.cpu().pin_memory(), z.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dy_, dz_ = torch.empty_like(y), torch.empty_like(z)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        dy_.copy_(hy, non_blocking=True)
        dz_.copy_(hz, non_blocking=True)
        ssd.gate_norm(dy_, dz_, w, width, out=out, stream=stream)
        ho.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    ms_max, e2e_max = slowest_rank([ms, e2e_ms], dev)
    if rank == 0:
        nbytes = 3 * rows * width * 2 + width * 4
        peak, peak_kind = peaks()
        achieved = nbytes / (ms / 1e3) / 1e9
        print(json.dumps({
            "metric": GATE_NORM_METRIC, "value": job_rate(rows, world, ms_max), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"gate_norm_rows{rows}_width{width}_group{width}", "storage": "bf16",
                       "kernel": "ssd_gate_norm_kernel", "l2": "256 MiB write before every timed step",
                       "bytes_per_step": nbytes},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": peak_kind, "traffic": None,
                         "scope": "y and z read, out written, weight read: one ssd_gate_norm launch"},
            "e2e": {"value": job_rate(rows, world, e2e_max), "unit": "tokens/s",
                    "h2d_bytes_per_step": 2 * rows * width * 2, "d2h_bytes_per_step": rows * width * 2},
            "gpu_launches": args.steps, "clocks": clk.summary()}), flush=True)


def run_bwd(args, p, dev, rank, local_rank, world):
    """Backward workload: a step is one ssd_bwd call over the configuration's
    inputs, random dy and dfinal_states (packed documents: every document's
    initial state and final-state gradient, and its dinit)."""
    import torch
    import torch.distributed as dist
    import mamba_ssd_chunked_scan_gb300 as ssd

    def io(a):
        return torch.from_numpy(synth.bf16_bits(a).view(np.int16).copy()).to(dev).view(torch.bfloat16)

    rng = np.random.default_rng(11)
    dy_h = rng.standard_normal((p.batch, p.seqlen, p.nheads, p.headdim)).astype(np.float32)
    x, B, C, dy = io(p.x), io(p.B), io(p.C), io(dy_h)
    dt = torch.from_numpy(p.dt).to(dev)
    A = torch.from_numpy(p.A).to(dev)
    D = torch.from_numpy(p.D).to(dev)
    docs = p.cu_seqlens is not None
    nst = p.nstates if docs else p.batch
    dfin = torch.from_numpy(rng.standard_normal((nst, p.nheads, p.headdim, p.dstate)).astype(np.float32)).to(dev)
    init = torch.from_numpy(p.initial_states).to(dev) if p.initial_states is not None else None
    cu = torch.from_numpy(p.cu_seqlens).to(dev) if docs else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(xx=x, dd=dt, bb=B, cc=C, yy=dy, ii=init, ff=dfin):
        return ssd.ssd_bwd(xx, dd, A, bb, cc, yy, D, ii, ff, cu, want_dinit=docs, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps

    # end to end: inputs from pinned host memory, the gradients back to pinned host memory
    ins = (x, dt, B, C, dy) + ((init, dfin) if docs else ())
    hin = [t.cpu().pin_memory() for t in ins]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    din = [torch.empty_like(t) for t in ins]
    g0 = step()
    hout = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in g0.items() if v is not None}
    d2h = sum(t.numel() * t.element_size() for t in hout.values())

    def e2e_step():
        for dst, src in zip(din, hin):
            dst.copy_(src, non_blocking=True)
        g = step(*din)
        for k, t in hout.items():
            t.copy_(g[k], non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps

    ms_max, e2e_max = slowest_rank([ms, e2e_ms], dev)
    tokens = p.batch * p.seqlen
    if rank == 0:
        tc = bwd_uses_tensor_cores(p)
        fl = bwd_tc_flops(p) if tc else bwd_flops(p)
        achieved = fl / (ms / 1e3) / 1e12
        if tc:
            pk, pk_kind = bf16_peak()
            roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
                    "peak_source": pk_kind, "traffic": None,
                    "scope": "algorithmic bf16 MMA flops of the whole ssd_bwd call (2 launches)"}
            kern = "ssd_bwd_tc (tcgen05, bf16 operands, fp32 accumulation) + ssd_bwd_reduce"
        else:
            roof = {"bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                    "frac": achieved / FP32_PEAK_TFLOPS,
                    "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 x 2.07 GHz", "traffic": None,
                    "scope": "algorithmic fp32 flops of the whole ssd_bwd call (2 launches)"}
            kern = "ssd_bwd_chunk + ssd_bwd_reduce (CUDA cores, fp32)"
        line = {
            "metric": BWD_METRIC, "value": job_rate(tokens, world, ms_max), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if tc else "f32", "data": "synthetic",
            "config": {"workload": "bwd_" + p.name, "batch": p.batch, "seq_len": p.seqlen, "nheads": p.nheads,
                       "headdim": p.headdim, "dstate": p.dstate, "ngroups": p.ngroups, "storage": p.dtype,
                       "kernel": kern,
                       "l2": "256 MiB write before every timed step; inputs larger than L2",
                       "algorithmic_flops": fl},
            "roofline": roof,
            "e2e": {"value": job_rate(tokens, world, e2e_max), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = bwd_cpu_baseline(p, dy_h)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bwd_sample(p, dy_h, tokens=512):
    """One batch row, the first `tokens` tokens: the oracle backward's sample."""
    q = synth.SSDProblem(1, tokens, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0, p.dtype,
                         p.x[:1, :tokens].copy(), p.dt[:1, :tokens].copy(), p.A, p.B[:1, :tokens].copy(),
                         p.C[:1, :tokens].copy(), p.D, None, None, p.name)
    return q, dy_h[:1, :tokens].copy()


def bwd_cpu_baseline(p, dy_h):
    import oracle
    q, dyq = bwd_sample(p, dy_h)
    reps, t_all = 0, 0.0
    while t_all < 10.0 and reps < 8:
        t0 = time.perf_counter()
        oracle.ssd_backward(q, dyq)
        t_all += time.perf_counter() - t0
        reps += 1
    return {"value": q.seqlen * reps / t_all, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"fp64 reverse-mode recurrence, batch row 0, tokens 0..{q.seqlen - 1} of {p.name}, {reps} passes"}


def forward_inputs(p, dev):
    """Device tensors of one forward workload (the bytes the oracle reads)."""
    import torch

    def dev_io(name):
        if p.dtype == "bf16":
            return torch.from_numpy(p.storage(name).view(np.int16).copy()).to(dev).view(torch.bfloat16)
        return torch.from_numpy(getattr(p, name)).to(dev)

    d = dict(x=dev_io("x"), B=dev_io("B"), C=dev_io("C"), dt=torch.from_numpy(p.dt).to(dev),
             A=torch.from_numpy(p.A).to(dev))
    d["D"] = None if p.D is None else torch.from_numpy(p.D).to(dev)
    d["init"] = None if p.initial_states is None else torch.from_numpy(p.initial_states).to(dev)
    d["cu"] = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(dev)
    return d


def time_forward(p, d, dev, stream, flush, warmup, steps, clk_index=None):
    """Device time of one ssd_fwd call (CUDA events on the launching stream, L2
    flushed before every call), and each launch's own duration (ssd_fwd_timed).
    Returns (call object, plan, y, final_states, mean call ms, mean ms per launch, clocks)."""
    import torch
    import mamba_ssd_chunked_scan_gb300 as ssd

    dtype = torch.bfloat16 if p.dtype == "bf16" else torch.float32
    f = ssd.SSDForward(p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, p.split_len,
                       p.ndocs, dtype, dev)
    want_final = d["init"] is not None
    plan = f.plan(want_final, want_final)
    y = torch.empty_like(d["x"])
    fin = torch.empty((f.nstates, p.nheads, p.headdim, p.dstate), dtype=torch.float32, device=dev) \
        if want_final else None

    def step():
        f(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["cu"], y=y, final_states=fin, stream=stream)

    for _ in range(warmup):
        flush.zero_()
        step()
    assert f.check_status() == 0
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clk = ClockSampler(clk_index) if clk_index is not None else None
    if clk:
        clk.__enter__()
    try:
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    finally:
        if clk:
            clk.__exit__()
    st = f.check_status()
    assert st == 0, f"device status {st}"
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    per_launch = []
    for _ in range(steps):
        flush.zero_()
        per_launch.append(f.launch_times(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["cu"],
                                         y=y, final_states=fin, stream=stream))
    launch_ms = [sum(r[k] for r in per_launch) / len(per_launch) for k in range(len(per_launch[0]))]
    return f, plan, y, fin, ms, launch_ms, (clk.summary() if clk else None)


def forward_roofline(p, plan, ms, launch_ms, nsm):
    """The call's compulsory-byte rate and the full-pass launch's roofline: the
    full pass (the call's last launch) reads all of x, dt, B, C, writes all of
    y, and reads the incoming state of every unit that continues a sequence."""
    family, launches, nsplit = plan
    nbytes = compulsory_bytes(p)
    peak, peak_kind = peaks()
    achieved_call = nbytes / (ms / 1e3) / 1e9
    state_bytes = 0
    if launches > 1:
        cont = p.batch * p.nheads * (nsplit - 1) if nsplit > 1 else tail_pieces(p, nsm)
        state_bytes = cont * p.headdim * p.dstate * 4
    kernel_bytes = nbytes + state_bytes
    achieved = kernel_bytes / (launch_ms[-1] / 1e3) / 1e9
    traffic = kernel_traffic(family, p.name)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": peak_kind, "traffic": traffic, "algorithmic_bytes": kernel_bytes,
            "frac_of_8TBps_spec": achieved / 8000.0,
            "scope": ("the full-pass launch of ssd_chunk_tc: compulsory bytes plus incoming states, over its "
                      f"own CUDA-event duration; frac_call is the whole call ({launches} launches)")
            if family == 1 else f"the full-pass launch of ssd_chunk_simt ({launches} launches per call)"}
    return nbytes, achieved_call, achieved_call / peak, roof


def sweep_points():
    """The other forward configurations, each a point of the tokens/s-vs-L
    curve: the 2.7B-like layer, the fixed-16,384-token sweep at every (batch,
    L) and split length, and the packed-document stress case."""
    pts = [("27b", synth.config_27b)]
    for b, L in ((16, 1024), (8, 2048), (4, 4096), (2, 8192), (1, 16384)):
        for sc in (1, 4, 16):
            pts.append((f"sweep:{b}:{L}:{sc}", lambda b=b, L=L, sc=sc: synth.config_sweep(b, L, sc)))
    pts.append(("varlen", synth.config_varlen))
    pts.append(("varlen_states", lambda: synth.config_varlen(init_std=0.2)))
    return pts


def oracle_rate(p, seconds=2.0, max_tokens=16384):
    """The fp64 oracle recurrence on a bounded sample (batch row 0, at most
    max_tokens tokens; packed documents: the whole row), tokens/s on all cores."""
    import oracle
    T = p.seqlen if p.cu_seqlens is not None else min(p.seqlen, max_tokens)
    q = synth.SSDProblem(1, T, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk, 0,
                         p.dtype, p.x[:1, :T].copy(), p.dt[:1, :T].copy(), p.A, p.B[:1, :T].copy(),
                         p.C[:1, :T].copy(), p.D,
                         None if p.initial_states is None else
                         (p.initial_states if p.cu_seqlens is not None else p.initial_states[:1].copy()),
                         p.cu_seqlens, p.name)
    reps, t_all = 0, 0.0
    while t_all < seconds and reps < 16:
        t0 = time.perf_counter()
        oracle.ssd_recurrence(q, want_final=False)
        t_all += time.perf_counter() - t0
        reps += 1
    return {"value": T * reps / t_all, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"fp64 recurrence on batch row 0 (tokens 0..{T - 1}) of {p.name}, {reps} passes, "
                      f"{t_all:.1f} s wall"}


def run_sweep(args, dev, stream, flush, nsm):
    """One line per point of the vs-L curve (device time per call, the
    full-pass roofline, the oracle on the host beside it)."""
    import torch
    out, rates = [], {}
    for name, make in sweep_points():
        p = make()
        d = forward_inputs(p, dev)
        f, plan, y, fin, ms, launch_ms, _ = time_forward(p, d, dev, stream, flush, 3, min(args.steps, 10))
        nbytes, ach_call, frac_call, roof = forward_roofline(p, plan, ms, launch_ms, nsm)
        key = (p.nheads, p.headdim, p.dstate, p.ngroups, p.cu_seqlens is not None, p.initial_states is not None)
        if not args.no_cpu_baseline and key not in rates:
            rates[key] = oracle_rate(p)
        out.append({"workload": p.name, "batch": p.batch, "seq_len": p.seqlen, "nheads": p.nheads,
                    "split_len": p.split_len, "nsplits": plan[2], "launches": plan[1],
                    "ms_per_step": ms, "tokens_per_s": p.batch * p.seqlen / (ms / 1e3),
                    "achieved_GBps_call": ach_call, "frac_call": frac_call, "launch_ms": launch_ms,
                    "roofline": roof, "cpu_baseline": rates.get(key)})
        del d, f, y, fin
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    p = workload(args.workload)
    if p.seqlen == 1:
        return run_decode(args, p, dev, rank, local_rank, world)
    if args.workload.startswith("bwd"):
        return run_bwd(args, p, dev, rank, local_rank, world)
    if args.workload == "gatenorm":
        return run_gate_norm(args, p, dev, rank, local_rank, world)

    d = forward_inputs(p, dev)
    x, B, C, dt, A, D, init, cu = (d[k] for k in ("x", "B", "C", "dt", "A", "D", "init", "cu"))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    f, plan, y, fin, ms, launch_ms, clocks = time_forward(p, d, dev, stream, flush, args.warmup, args.steps,
                                                          clk_index=local_rank)
    family, launches, nsplit = plan
    if world > 1:
        dist.barrier()
    copy_bw = device_copy_gbps(dev, stream)

    # End to end through the public API, as a job that streams batches runs it: every
    # step copies its inputs from pinned host memory to the device and its result back
    # to pinned host memory.  Step i's inputs move host->device while step i-1 computes
    # and step i-2's result moves device->host (the two directions use different copy
    # engines): two device buffer sets, one stream per direction.  The timed region
    # spans all K steps, pipeline fill and drain included.
    hx, hB, hC, hdt = (t.cpu().pin_memory() for t in (x, B, C, dt))
    h2d = sum(t.numel() * t.element_size() for t in (hx, hB, hC, hdt))
    d2h = y.numel() * y.element_size() + (fin.numel() * 4 if fin is not None else 0)
    dbufs = [dict(x=x, B=B, C=C, dt=dt, y=y, fin=fin),
             dict(x=torch.empty_like(x), B=torch.empty_like(B), C=torch.empty_like(C), dt=torch.empty_like(dt),
                  y=torch.empty_like(y), fin=None if fin is None else torch.empty_like(fin))]
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    hfin = [torch.empty(fin.shape, dtype=torch.float32).pin_memory() for _ in range(2)] if fin is not None else None
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i):
        k = i % 2
        b = dbufs[k]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[k])       # step i-2 has read this buffer set's inputs
            b["x"].copy_(hx, non_blocking=True)
            b["B"].copy_(hB, non_blocking=True)
            b["C"].copy_(hC, non_blocking=True)
            b["dt"].copy_(hdt, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if i >= 2:
            stream.wait_event(ev_out[k])          # step i-2's result has left this buffer set
        f(b["x"], b["dt"], A, b["B"], b["C"], D, init, cu, y=b["y"], final_states=b["fin"], stream=stream)
        ev_comp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            hy[k].copy_(b["y"], non_blocking=True)
            if hfin is not None:
                hfin[k].copy_(b["fin"], non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.warmup, args.warmup + args.steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    assert f.check_status() == 0
    e2e_ms = e0.elapsed_time(e1) / args.steps
    del dbufs, hy, hfin

    ms_max, e2e_max = slowest_rank([ms, e2e_ms], dev)
    tokens = p.batch * p.seqlen
    value = job_rate(tokens, world, ms_max)
    e2e_value = job_rate(tokens, world, e2e_max)
    if rank == 0:
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        nbytes, achieved_call, frac_call, roof = forward_roofline(p, plan, ms, launch_ms, nsm)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if family == 1 else "f32", "data": "synthetic",
            "config": {"workload": p.name, "batch": p.batch, "seq_len": p.seqlen, "nheads": p.nheads,
                       "headdim": p.headdim, "dstate": p.dstate, "ngroups": p.ngroups, "chunk": p.chunk,
                       "split_len": p.split_len, "nsplits": nsplit, "storage": p.dtype,
                       "kernel": "tcgen05" if family == 1 else "simt",
                       "l2": "256 MiB write before every timed step; inputs larger than L2",
                       "compulsory_bytes": nbytes, "achieved_GBps_call": achieved_call,
                       "frac_call": frac_call, "pct_of_8TBps_spec_call": 100.0 * achieved_call / 8000.0,
                       "launch_ms": launch_ms, "copy_GBps_here": copy_bw},
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(p)
        if world == 1 and not args.no_sweep and args.workload == DEFAULT_WORKLOAD:
            del d, x, B, C, dt, y, fin, hx, hB, hC, hdt, f
            torch.cuda.empty_cache()
            line["vs_L"] = run_sweep(args, dev, stream, flush, nsm)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the vs-L points of the default run")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
