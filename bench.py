#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch: attn_fwd (O, L), then
attn_bwd = preprocess (D) + fused main kernel (dK, dV, dQ accumulation) + dQ
convert.  The headline metric is backward TFLOP/s: 10*B*H*N^2*d FLOPs
(halved under the causal mask) divided by the device time of attn_bwd.

Timing: W untimed warm-up steps, then exactly K timed steps; before every
step a 512 MiB buffer is written to flush the 129 MB L2; each step is
bracketed by CUDA events on the launching stream; a barrier and a device
synchronisation bracket the timed region; with several ranks the time is the
maximum over ranks.  nvidia-smi samples SM clocks and throttle reasons during
the timed region.

Legs reported on the one JSON line (rank 0):
  value       backward TFLOP/s, inputs resident in HBM
  e2e         the same metric through the public API with pinned HOST
              buffers: every step uploads its inputs, runs forward and
              backward, and downloads its gradients; uploads and downloads
              run on their own streams and overlap neighbouring steps
  roofline    the backward main kernel (tensor-bound) against the measured
              dense bf16 peak
  cpu_baseline the fp64 oracle on the host cores (their count and CPU model),
              on a bounded sample
  other_workloads  the other named workloads (d = 64 causal N = 2048, and
              the two causal d = 128 ones), main-kernel TF/s, sliding-window
              attention (N = 16384, a 4096-key window) and packed documents
              (N = 16384, six documents)

The headline workload is the largest named one, B=4 H=16 N=8192 d=128
without the mask: it is the configuration the metric is quoted on.

--impl reference times the fp64 CPU oracle (the only reference this project
has) on the same workload, metric and unit.

Multi-GPU (torchrun, one rank per GPU): heads are independent, so every rank
runs its own replica of the workload with no collective on the data path
(weak scaling); value = all ranks' FLOPs / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "b4h16n8192d128"
OTHER = ["b2h16n2048d64_causal", "b1h32n4096d128_causal", "b1h16n16384d128_causal"]
METRIC = "attention backward TFLOP/s (bf16, 1xGB300) and fraction of dense bf16 peak"
FLUSH_BYTES = 512 << 20
# The extra workloads' timing: the median of a short run (10 steps after 3
# warm-ups; 200 steps on the d = 64 workloads, whose steps take tens of
# microseconds), so that they run at full clock and compare with the burst
# peak.  The headline's seconds-long loop gives the sustained figure: 50-step
# runs of the larger workloads already settle under the power cap (the
# N = 16384 causal main kernel at 1,362 TFLOP/s against 1,425-1,445).
EXTRA_WARMUP = 3
EXTRA_REPS = 10
SMALL_REPS = 200


def extra_reps(w) -> int:
    return SMALL_REPS if w.d == 64 else EXTRA_REPS
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _strip_comments(src: str) -> str:
    """C/C++ source without comments or blank lines (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':  # string literal, copied whole
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).split("\n")]
    return "\n".join(ln for ln in lines if ln.strip())


# The CUDA sources each profiled kernel is built from (its own code, the
# PTX wrappers and mask helpers it includes, and its launcher).
KERNEL_SOURCES = {
    "attn_bwd_main_kernel": ["attn_bwd_main.cuh", "attn_bwd.cu", "ptx.cuh", "mask.cuh",
                             "f32x2.cuh", "kernels.h"],
    # the same template without dQ (the separate-dQ method's first pass)
    "attn_bwd_main_kernel_dkdv": ["attn_bwd_main.cuh", "attn_bwd.cu", "ptx.cuh", "mask.cuh",
                                  "f32x2.cuh", "kernels.h"],
    "attn_bwd_preprocess_kernel": ["attn_bwd.cu", "attn_bwd_main.cuh", "ptx.cuh", "mask.cuh"],
    "attn_bwd_dq_convert_kernel": ["attn_bwd.cu", "attn_bwd_main.cuh", "ptx.cuh", "mask.cuh"],
    "attn_fwd_kernel": ["attn_fwd.cu", "ptx.cuh", "mask.cuh", "f32x2.cuh", "kernels.h"],
    "attn_fwd_fp8_kernel": ["attn_fwd_fp8.cu", "ptx.cuh", "f32x2.cuh", "kernels.h"],
    "attn_bwd_fp8_kernel": ["attn_bwd_fp8.cu", "ptx.cuh"],
    "attn_bwd_dq_kernel": ["attn_bwd_dq.cu", "ptx.cuh", "mask.cuh", "kernels.h"],
    "ssd_chunk_bwd_kernel": ["ssd.cu", "ptx.cuh"],
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the CUDA sources a kernel is built from (all of them when no
    kernel is named), comments excluded: a stored ncu traffic figure is only
    used if that code has not changed since it was captured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_backward_pass_attn_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) if kernel else None
    if names is None:
        names = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h"))]
    for name in sorted(names):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = _strip_comments(f.read())
        h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def stored_ncu(kernel: str, workload: str):
    """The committed ncu entry of a kernel on a workload (DRAM bytes per
    launch, tensor-pipe activity), if the CUDA sources are still those it was
    captured on; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get("%s@%s" % (kernel, workload))
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent


def stored_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if still valid."""
    ent = stored_ncu(kernel, workload)
    return ent.get("dram_bytes_per_launch") if ent else None


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms: float, local_flops: float, group=None):
    """(max time over ranks, total FLOPs over ranks): the slowest rank sets the
    job time; every rank's work counts."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return local_ms, local_flops
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    f = torch.tensor([local_flops], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(f, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(f.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def workload_of(args):
    """The named workload, or (with --batch B) the same shape with B batch
    elements, renamed after its shape."""
    from attention_backward_pass_attn_gb300.inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.batch > 0 and args.batch != w.B:
        name = "b%dh%dn%dd%d%s" % (args.batch, w.H, w.N, w.d, "_causal" if w.causal else "")
        w = w.with_shape(B=args.batch, name=name)
    return w


def config_dict(w) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    return {
        "workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
        "scale": "1/sqrt(d)", "l2": "flushed before every step (512 MiB write)",
        "timing": "CUDA events per step on the launching stream, around the forward and "
                  "around the whole attn_bwd call (no events between its three kernels, "
                  "which start early by programmatic dependent launch); value = backward "
                  "FLOPs (10*B*H*N^2*d, halved causal) / attn_bwd device time",
        "parallelism": "replicas (independent heads), no collective on the data path",
    }


# ----------------------------------------------------------------------------- our arm
def time_workload(w, steps: int, warmup: int, flush, split=False, dq_method=None):
    """Run fwd + bwd `warmup + steps` times; returns per-step event times (ms).

    Events go before the forward, between forward and backward, and after the
    backward.  With `split`, events also separate the three backward kernels,
    giving each kernel's time -- but an event between two kernels stops the
    next one from starting early (programmatic dependent launch), so the
    backward is timed as a whole without them."""
    import torch

    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import make_doc_map, make_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = ab.alloc_workspace(w.B, w.H, w.N, w.d, dev)
    stream = torch.cuda.current_stream()
    dmap = make_doc_map(w)
    dmap = dmap.to(dev) if dmap is not None else None
    method = ab.ATTN_DQ_AUTO if dq_method is None else dq_method

    def step():
        ab.attn_fwd(q, k, v, w.causal, w.scale, out=o, lse=lse, stream=stream, window=w.window,
                    doc=dmap)
        e[1].record(stream)
        if split and method == ab.ATTN_DQ_SEPARATE:
            ab.attn_bwd_preprocess(o, do, lse, ws, stream=stream)
            e[2].record(stream)
            ab.attn_bwd_main_dkdv(q, k, v, do, dk, dv, w.causal, ws, scale=w.scale,
                                  stream=stream)
            e[3].record(stream)
            ab.attn_bwd_dq(q, k, v, do, dq, w.causal, ws, scale=w.scale, stream=stream)
        elif split:
            ab.attn_bwd_preprocess(o, do, lse, ws, stream=stream)
            e[2].record(stream)
            ab.attn_bwd_main(q, k, v, do, dk, dv, w.causal, ws, scale=w.scale, stream=stream)
            e[3].record(stream)
            ab.attn_bwd_dq_convert(dq, ws, scale=w.scale, stream=stream)
        else:  # the public call
            ab.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, dq=dq, dk=dk, dv=dv,
                        workspace=ws, stream=stream, window=w.window, doc=dmap,
                        dq_method=method)

    rec = []
    for i in range(warmup + steps):
        flush()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        e[0].record(stream)
        step()
        e[4].record(stream)
        if i >= warmup:
            rec.append(e)
    torch.cuda.synchronize()
    st = ab.attn_last_device_error()
    if st != ab.ATTN_OK:
        raise RuntimeError("device error status %d during the benchmark" % st)
    out = {"fwd": [], "prep": [], "main": [], "conv": [], "bwd": [], "step": []}
    for e in rec:
        out["fwd"].append(e[0].elapsed_time(e[1]))
        out["bwd"].append(e[1].elapsed_time(e[4]))
        out["step"].append(e[0].elapsed_time(e[4]))
        if split:
            out["prep"].append(e[1].elapsed_time(e[2]))
            out["main"].append(e[2].elapsed_time(e[3]))
            out["conv"].append(e[3].elapsed_time(e[4]))
    return out


def time_fp8_forward(w, steps: int, warmup: int, flush):
    """attn_fwd_fp8 on the workload's inputs quantised to e4m3 (per-tensor
    descale); per-launch CUDA-event times (ms)."""
    import torch

    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import make_inputs_fp8

    dev = torch.device("cuda", torch.cuda.current_device())
    (q8, qd), (k8, kd), (v8, vd), _ = make_inputs_fp8(w)
    q8, k8, v8 = q8.to(dev), k8.to(dev), v8.to(dev)
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    rec = []
    for i in range(warmup + steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ab.attn_fwd_fp8(q8, k8, v8, (qd, kd, vd), w.causal, w.scale, out=o, lse=lse,
                        stream=stream)
        e1.record(stream)
        if i >= warmup:
            rec.append((e0, e1))
    torch.cuda.synchronize()
    if ab.attn_last_device_error() != ab.ATTN_OK:
        raise RuntimeError("device error during the fp8 forward")
    return [a.elapsed_time(b) for a, b in rec]


def time_ssd(w, steps: int, warmup: int, flush):
    """ssd_fwd and ssd_bwd of one Mamba-2 layer shape: per-call CUDA-event
    times (ms) of each, L2 flushed before every call."""
    import torch

    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import make_ssd_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    x, dt, A, B, C, D, dy = (t.to(dev) for t in make_ssd_inputs(w))
    ws = ab.ssd_workspace(w.Bt, w.T, w.H, w.G, w.N, w.P, dev)
    y = torch.empty(x.shape, dtype=torch.float32, device=dev)
    out = None
    stream = torch.cuda.current_stream()
    fwd, bwd = [], []
    for i in range(warmup + steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush()
        ev[0].record(stream)
        ab.ssd_fwd(x, dt, A, B, C, D, y=y, workspace=ws, stream=stream)
        ev[1].record(stream)
        flush()
        ev[2].record(stream)
        out = ab.ssd_bwd(x, dt, A, B, C, D, dy, workspace=ws, out=out, stream=stream)
        ev[3].record(stream)
        if i >= warmup:
            fwd.append(ev)
    torch.cuda.synchronize()
    if ab.attn_last_device_error() != ab.ATTN_OK:
        raise RuntimeError("device error during the state-space layer")
    return ([e[0].elapsed_time(e[1]) for e in fwd], [e[2].elapsed_time(e[3]) for e in fwd])


def ssd_chunked_flops(w, chunk: int = 64):
    """FLOPs the chunked backward executes (the kernels' own algorithm):
    per chunk of L steps, the chunk states S and R (4 L N P), the scans over
    chunks (4 N P), and the chunk gradients: C B^T and dy x^T (2 L^2 (N+P)),
    the triangular products for dx, dB, dC (L^2 P + 2 L^2 N) and their state
    terms (6 L N P), <dH, H> (2 N P)."""
    L, N, P = chunk, w.N, w.P
    nc = (w.T + L - 1) // L
    per = 4 * L * N * P + 4 * N * P + 2 * L * L * (N + P) + L * L * P + 2 * L * L * N \
        + 6 * L * N * P + 2 * N * P
    return float(per) * w.Bt * w.H * nc


def time_fp8_backward(w, steps: int, warmup: int, flush):
    """attn_bwd_fp8 on the workload's inputs quantised to e4m3 (per-tensor
    descales), O and L from attn_fwd_fp8, dS scaled the way fp8 training
    scales it (a first call reports max |dS|; the timed calls use the largest
    power of two that keeps it within e4m3's range); per-call CUDA-event
    times (ms)."""
    import torch

    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import make_inputs, quantize_e4m3

    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = make_inputs(w)
    (q8, qd), (k8, kd), (v8, vd), (do8, dod) = (quantize_e4m3(t) for t in (q, k, v, do))
    q8, k8, v8, do8 = (t.to(dev) for t in (q8, k8, v8, do8))
    o, lse = ab.attn_fwd_fp8(q8, k8, v8, (qd, kd, vd), w.causal, w.scale)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    ws = ab.alloc_workspace(w.B, w.H, w.N, w.d, dev)
    ab.attn_bwd_fp8(q8, k8, v8, o, do8, lse, (qd, kd, vd, dod), 1.0, w.causal, w.scale,
                    ds_amax=amax, workspace=ws)
    torch.cuda.synchronize()
    ds_scale = 2.0 ** math.floor(math.log2(448.0 / max(float(amax.item()), 1e-30)))
    stream = torch.cuda.current_stream()
    rec = []
    for i in range(warmup + steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ab.attn_bwd_fp8(q8, k8, v8, o, do8, lse, (qd, kd, vd, dod), ds_scale, w.causal, w.scale,
                        ds_amax=amax, workspace=ws, stream=stream)
        e1.record(stream)
        if i >= warmup:
            rec.append((e0, e1))
    torch.cuda.synchronize()
    if ab.attn_last_device_error() != ab.ATTN_OK:
        raise RuntimeError("device error during the fp8 backward")
    return [a.elapsed_time(b) for a, b in rec]


def e2e_workload(w, steps: int, warmup: int, with_forward: bool = False):
    """The backward through the public API with pinned host buffers, pipelined
    as a training loop would run it: each step copies the backward's inputs
    (Q, K, V, O, dO and L) host -> device, runs attn_bwd, and copies dQ, dK,
    dV device -> host; the copies run on their own streams, so step i+1's
    upload and step i-1's download overlap step i's compute (two sets of device
    buffers).  O and L come from one attn_fwd before the loop.  With
    `with_forward`, each step instead uploads Q, K, V, dO and runs attn_fwd
    then attn_bwd (a whole attention training step).
    Returns (ms per step over the timed steps, h2d bytes, d2h bytes, device
    bytes of both buffer sets)."""
    import torch

    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import make_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = make_inputs(w)
    if with_forward:
        host_in = [t.pin_memory() for t in (q, k, v, do)]
    else:
        qd, kd, vd = (t.to(dev) for t in (q, k, v))
        o, lse = ab.attn_fwd(qd, kd, vd, w.causal, w.scale)
        torch.cuda.synchronize()
        host_in = [t.pin_memory() for t in (q, k, v, o.cpu(), do, lse.cpu())]
        del qd, kd, vd, o, lse
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in host_in[:3]]
    sets = []
    for _ in range(2):
        dev_in = [torch.empty_like(t, device=dev) for t in host_in]
        sets.append({
            "in": dev_in,
            "o": torch.empty_like(dev_in[0]) if with_forward else None,
            "lse": (torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
                    if with_forward else None),
            "grads": [torch.empty_like(dev_in[0]) for _ in range(3)],
            "ws": ab.alloc_workspace(w.B, w.H, w.N, w.d, dev),
            "in_ready": torch.cuda.Event(), "done": torch.cuda.Event(),
            "out_free": torch.cuda.Event(), "in_free": torch.cuda.Event(),
        })
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    total = warmup + steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(total):
        b = sets[i % 2]
        if i == warmup:
            t_start.record(s_in)
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(b["in_free"])
            for h, d in zip(host_in, b["in"]):
                d.copy_(h, non_blocking=True)
            b["in_ready"].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(b["in_ready"])
            if i >= 2:
                s_comp.wait_event(b["out_free"])
            if with_forward:
                q_, k_, v_, do_ = b["in"]
                o_, lse_ = b["o"], b["lse"]
                ab.attn_fwd(q_, k_, v_, w.causal, w.scale, out=o_, lse=lse_, stream=s_comp)
            else:
                q_, k_, v_, o_, do_, lse_ = b["in"]
            ab.attn_bwd(q_, k_, v_, o_, do_, lse_, w.causal, w.scale, dq=b["grads"][0],
                        dk=b["grads"][1], dv=b["grads"][2], workspace=b["ws"], stream=s_comp)
            b["in_free"].record(s_comp)
            b["done"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["done"])
            for d, h in zip(b["grads"], host_out):
                h.copy_(d, non_blocking=True)
            b["out_free"].record(s_out)
    t_end.record(s_out)
    torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end) / steps
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    resident = 0
    for b in sets:
        for t in b["in"] + b["grads"] + [b["ws"]] + ([b["o"], b["lse"]] if with_forward else []):
            resident += t.numel() * t.element_size()
    return ms, h2d, d2h, resident


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, else lscpu), or the machine type."""
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def cpu_baseline(w, target_seconds: float = 15.0):
    """The fp64 oracle, as it stands, on the host cores, on a bounded sample of
    the workload: its first k heads (fwd + bwd), k sized from a one-head
    calibration run so that the timed sample takes about `target_seconds`.
    FLOPs are counted pro rata (k / B*H of the workload's backward FLOPs)."""
    import oracle
    from attention_backward_pass_attn_gb300.inputs import make_inputs

    q, k, v, do = make_inputs(w)
    flat = [t.reshape(w.heads, 1, w.N, w.d) for t in (q, k, v, do)]
    lib = oracle.load()
    t0 = time.perf_counter()
    oracle.attention_forward_backward(*(t[:1] for t in flat), w.causal, w.scale, lib=lib)
    t_head = time.perf_counter() - t0
    heads = int(max(1, min(w.heads, target_seconds // max(t_head, 1e-6))))
    sample = [t[:heads] for t in flat]
    t0 = time.perf_counter()
    oracle.attention_forward_backward(*sample, w.causal, w.scale, lib=lib)
    el = time.perf_counter() - t0
    flops = w.bwd_flops() * heads / w.heads
    return {"value": flops / el / 1e12, "unit": "TFLOP/s",
            "cores": oracle.max_threads(lib), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": "the first %d of %d heads of %s, fp64 fwd+bwd in one call, %.1f s; "
                      "backward FLOPs of those heads / time" % (heads, w.heads, w.name, el)}


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS

    ab.load_library()
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak_tf))
    w = workload_of(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    # warm-up outside the sampled window, then the timed region
    time_workload(w, 0, max(args.warmup, 3), flush)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    res = time_workload(w, args.steps, 0, flush)
    torch.cuda.synchronize()
    barrier()
    wall_s = time.perf_counter() - t_wall0
    time.sleep(0.2)
    clocks = sampler.stop()

    bwd_ms_total = sum(res["bwd"])
    step_ms_total = sum(res["step"])
    bwd_max_ms, flops_all = aggregate(bwd_ms_total, w.bwd_flops() * args.steps)
    step_max_ms, _ = aggregate(step_ms_total, 0.0)
    value = flops_all / (bwd_max_ms * 1e-3) / 1e12

    # Per-kernel times from a pass of the same steps with events between the
    # backward kernels (which the timed steps leave out, see time_workload).
    brk_steps = max(20, min(args.steps, 200))
    brk = time_workload(w, brk_steps, 3, flush, split=True)
    main_ms = statistics.mean(brk["main"])
    achieved = w.bwd_flops() / (main_ms * 1e-3) / 1e12

    e2e_steps = max(10, min(args.steps, 200))
    e2e_ms, h2d, d2h, e2e_resident = e2e_workload(w, e2e_steps, 3)
    e2e_max, e2e_flops = aggregate(e2e_ms * e2e_steps, w.bwd_flops() * e2e_steps)
    e2e_value = e2e_flops / (e2e_max * 1e-3) / 1e12
    # the same pipeline around a whole attention training step (attn_fwd then
    # attn_bwd), reported beside it
    ts_ms, ts_h2d, ts_d2h, _ = e2e_workload(w, e2e_steps, 3, with_forward=True)
    ts_max, ts_flops = aggregate(ts_ms * e2e_steps, w.bwd_flops() * e2e_steps)

    extra = None
    if not args.no_extra:
        extra = {}
        for name in OTHER:
            ow = WORKLOADS[name]
            r = time_workload(ow, extra_reps(ow), EXTRA_WARMUP, flush, split=True)
            rw = time_workload(ow, extra_reps(ow), EXTRA_WARMUP, flush)
            mm = statistics.median(r["main"])
            extra[name] = {
                "bwd_main_tflops": round(ow.bwd_flops() / mm / 1e9, 1),
                "bwd_main_frac": round(ow.bwd_flops() / mm / 1e9 / peak_tf, 4),
                "bwd_total_tflops": round(ow.bwd_flops() / statistics.median(rw["bwd"]) / 1e9, 1),
                "fwd_tflops": round(ow.fwd_flops() / statistics.median(r["fwd"]) / 1e9, 1),
                "main_ms_median": round(mm, 4),
                "bwd_ms_median": round(statistics.median(rw["bwd"]), 4),
            }
        # The two ways of forming dQ, timed against each other: the main
        # kernel reducing dQ partials into an fp32 accumulator, or a separate
        # query-stationary pass (two extra contractions, no accumulator).
        from attention_backward_pass_attn_gb300.binding import ATTN_DQ_REDUCE, ATTN_DQ_SEPARATE
        cmp = {}
        for name in [w.name] + OTHER:
            cw = w if name == w.name else WORKLOADS[name]
            n, wu = extra_reps(cw), EXTRA_WARMUP
            red = time_workload(cw, n, wu, flush, dq_method=ATTN_DQ_REDUCE)
            sep = time_workload(cw, n, wu, flush, dq_method=ATTN_DQ_SEPARATE)
            sep_split = time_workload(cw, n, wu, flush, split=True, dq_method=ATTN_DQ_SEPARATE)
            r_ms, s_ms = statistics.median(red["bwd"]), statistics.median(sep["bwd"])
            cmp[name] = {
                "reduce_bwd_ms": round(r_ms, 4), "separate_bwd_ms": round(s_ms, 4),
                "reduce_bwd_tflops": round(cw.bwd_flops() / r_ms / 1e9, 1),
                "separate_bwd_tflops": round(cw.bwd_flops() / s_ms / 1e9, 1),
                "separate_main_dkdv_ms": round(statistics.median(sep_split["main"]), 4),
                "separate_dq_pass_ms": round(statistics.median(sep_split["conv"]), 4),
                "faster": "reduce" if r_ms <= s_ms else "separate",
            }
        extra["dq_methods"] = cmp
        # The e4m3 forward beside the bf16 one, against the dense fp8 peak:
        # the measured bf16 figure times the nominal fp8/bf16 ratio (2).
        f8 = {}
        for name in [n for n in [w.name] + OTHER if WORKLOADS[n].d == 128]:
            fw = WORKLOADS[name]
            ms = statistics.median(time_fp8_forward(fw, EXTRA_REPS, EXTRA_WARMUP, flush))
            bms = statistics.median(time_fp8_backward(fw, EXTRA_REPS, EXTRA_WARMUP, flush))
            bf = time_workload(fw, EXTRA_REPS, EXTRA_WARMUP, flush)
            f8[name] = {"fp8_fwd_ms": round(ms, 4),
                        "fp8_fwd_tflops": round(fw.fwd_flops() / ms / 1e9, 1),
                        "fp8_fwd_frac_of_fp8_peak": round(fw.fwd_flops() / ms / 1e9
                                                          / (2 * peak_tf), 4),
                        "bf16_fwd_tflops": round(fw.fwd_flops() / statistics.median(bf["fwd"])
                                                 / 1e9, 1),
                        "fp8_bwd_ms": round(bms, 4),
                        "fp8_bwd_tflops": round(fw.bwd_flops() / bms / 1e9, 1),
                        "fp8_bwd_frac_of_fp8_peak": round(fw.bwd_flops() / bms / 1e9
                                                          / (2 * peak_tf), 4),
                        "bf16_bwd_tflops": round(fw.bwd_flops() / statistics.median(bf["bwd"])
                                                 / 1e9, 1)}
        extra["fp8"] = {"peak_tflops": 2 * peak_tf,
                                "peak_source": "measured bf16_tflops x 2 (nominal fp8/bf16 "
                                               "dense ratio 4.5/2.25)",
                                "workloads": f8}
        # The Mamba-2 layer of the hybrid model: fp32 arithmetic on the CUDA
        # cores, so its peak is the fp32 FMA rate: 152 SMs x 128 lanes x 2
        # FLOP x the SM clock (2070 MHz maximum).
        from attention_backward_pass_attn_gb300.inputs import SSD_WORKLOADS
        alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12
        ssd_res = {}
        for name, sw in SSD_WORKLOADS.items():
            f_ms, b_ms = time_ssd(sw, EXTRA_REPS, EXTRA_WARMUP, flush)
            fm, bm = statistics.median(f_ms), statistics.median(b_ms)
            ssd_res[name] = {
                "fwd_ms": round(fm, 4), "bwd_ms": round(bm, 4),
                "bwd_tokens_per_s": round(sw.tokens / (bm * 1e-3), 1),
                "bwd_recurrence_tflops": round(sw.recurrence_flops() / bm / 1e9, 2),
                "bwd_chunked_tflops": round(ssd_chunked_flops(sw) / bm / 1e9, 2),
                "bwd_alu_frac": round(ssd_chunked_flops(sw) / bm / 1e9 / alu_peak, 4)}
        extra["ssd"] = {"alu_peak_tflops": round(alu_peak, 1),
                        "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz",
                        "workloads": ssd_res}
        # Mask variants: a sliding window (4096 keys) and packed documents.
        # FLOPs are those of the visible pairs: N*W - W^2/2 per head under the
        # window, the sum of n^2/2 over documents of lengths n.
        for name, sw in EXTRA_WORKLOADS.items():
            rw = time_workload(sw, EXTRA_REPS, EXTRA_WARMUP, flush)
            extra[name] = {
                "window": sw.window,
                "documents": len(sw.doc_lengths),
                "bwd_total_tflops": round(sw.bwd_flops() / statistics.median(rw["bwd"]) / 1e9, 1),
                "bwd_total_frac": round(sw.bwd_flops() / statistics.median(rw["bwd"]) / 1e9
                                        / peak_tf, 4),
                "fwd_tflops": round(sw.fwd_flops() / statistics.median(rw["fwd"]) / 1e9, 1),
                "bwd_ms_median": round(statistics.median(rw["bwd"]), 4),
                "flops": "10*d*(visible pairs) per head (backward), 4*d*(...) (forward)",
            }

    if rank != 0:
        return None
    ncu_main = stored_ncu("attn_bwd_main_kernel", w.name)
    # The denominator: the measured dense bf16 GEMM as a burst for a kernel
    # that ran at full clock, its sustained (power-capped) figure when the
    # timed region itself ran under the power cap, as a seconds-long loop of
    # this size does.
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    peak_used = peak_sus if capped else peak_tf
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_max_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 inputs (no dataset)",
        "config": config_dict(w),
        "fwd_tflops": round(w.fwd_flops() / statistics.mean(res["fwd"]) / 1e9, 2),
        "bwd_ms": round(bwd_ms_total / args.steps, 5),
        "fwd_ms": round(sum(res["fwd"]) / args.steps, 5),
        "bwd_fwd_time_ratio": round(sum(res["bwd"]) / max(sum(res["fwd"]), 1e-9), 3),
        "wall_s_timed_region": round(wall_s, 3),
        "bwd_kernels_ms": {
            "preprocess": round(statistics.mean(brk["prep"]), 5),
            "main": round(main_ms, 5),
            "dq_convert": round(statistics.mean(brk["conv"]), 5),
            "sum_with_events_between": round(statistics.mean(brk["bwd"]), 5),
            "steps": brk_steps,
            "what": "a pass of the same steps after the timed region, with an event between "
                    "each backward kernel (this disables their early start)"},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5), "steps": e2e_steps,
                "what": "the backward through the public API: its inputs (Q, K, V, O, dO, L) "
                        "pinned host -> device, attn_bwd, dQ/dK/dV -> host every step; copies "
                        "on their own streams overlap neighbouring steps' compute (two device "
                        "buffer sets); backward FLOPs / step time",
                "l2": "not flushed: the two alternating device buffer sets hold %.0f MiB, "
                      "more than the 129 MB L2" % (e2e_resident / 2**20),
                "training_step": {
                    "value": round(ts_flops / (ts_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "ms_per_step": round(ts_ms, 5), "h2d_bytes_per_step": ts_h2d,
                    "d2h_bytes_per_step": ts_d2h,
                    "what": "the same pipeline around attn_fwd then attn_bwd (Q, K, V, dO "
                            "uploaded); backward FLOPs / step time, the forward's time "
                            "included"}},
        "roofline": {
            "kernel": "attn_bwd_main_kernel", "bound": "tensor",
            "achieved": round(achieved, 2), "peak": peak_used, "unit": "TFLOP/s",
            "frac": round(achieved / peak_used, 4),
            "traffic": stored_traffic("attn_bwd_main_kernel", w.name),
            "ncu_tensor_pipe_active_pct": (ncu_main or {}).get("tensor_pipe_active_pct"),
            "peak_source": "%s %s" % (
                "of measured" if peak_src == "measured" else "of fallback",
                "bf16_tflops_sustained (the timed region ran under the power cap)" if capped
                else "bf16_tflops (burst: the timed region ran at full clock)"),
            "frac_of_burst": round(achieved / peak_tf, 4),
            "frac_of_sustained": round(achieved / peak_sus, 4),
            "flops_per_launch": w.bwd_flops(),
            "avg_launch_ms": round(main_ms, 5),
            "launch_timing": "CUDA events around each main-kernel launch, %d steps of the same "
                             "workload run right after the timed region" % brk_steps,
        },
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    if extra is not None:
        line["other_workloads"] = extra
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    return line


def run_leg(args):
    """One leg alone (the e4m3 forward, the backward with the separate dQ
    pass, or the Mamba-2 layer) on --workload, W + K calls, for profiler
    captures of those kernels; prints their median CUDA-event times."""
    import torch

    torch.cuda.set_device(0)
    from attention_backward_pass_attn_gb300 import binding as ab
    from attention_backward_pass_attn_gb300.inputs import SSD_WORKLOADS

    ab.load_library()
    dev = torch.device("cuda", 0)
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    steps, warm = max(args.steps, 1), max(args.warmup, 3)
    if args.leg == "ssd":
        w = SSD_WORKLOADS[args.workload]
        f_ms, b_ms = time_ssd(w, steps, warm, flush)
        return {"leg": "ssd", "workload": w.name, "fwd_ms": statistics.median(f_ms),
                "bwd_ms": statistics.median(b_ms)}
    w = workload_of(args)
    if args.leg == "fp8_backward":
        ms = statistics.median(time_fp8_backward(w, steps, warm, flush))
        return {"leg": "fp8_backward", "workload": w.name, "ms": ms,
                "tflops": w.bwd_flops() / ms / 1e9}
    if args.leg == "fp8_forward":
        ms = statistics.median(time_fp8_forward(w, steps, warm, flush))
        return {"leg": "fp8_forward", "workload": w.name, "ms": ms,
                "tflops": w.fwd_flops() / ms / 1e9}
    r = time_workload(w, steps, warm, flush, split=True, dq_method=ab.ATTN_DQ_SEPARATE)
    return {"leg": "dq_separate", "workload": w.name,
            "main_dkdv_ms": statistics.median(r["main"]), "dq_ms": statistics.median(r["conv"])}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 CPU oracle as the reference arm.  Each step evaluates a bounded
    sample of the same workload, sized by a calibration run so that the whole
    warm-up + timed run stays within about three minutes: whole heads when a
    head fits the per-step budget, otherwise evenly spaced query rows of the
    first head (their O, L and dQ)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import numpy as np

    import oracle
    from attention_backward_pass_attn_gb300.inputs import WORKLOADS, make_inputs

    w = workload_of(args)
    q, k, v, do = make_inputs(w)
    flat = [t.reshape(w.B * w.H, 1, w.N, w.d) for t in (q, k, v, do)]
    lib = oracle.load()
    per_step_budget = 180.0 / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    oracle.attention_forward_backward(*(t[:1] for t in flat), w.causal, w.scale, lib=lib)
    t_head = time.perf_counter() - t0
    if t_head <= per_step_budget:
        heads = int(max(1, min(w.heads, per_step_budget // t_head)))
        sample = [t[:heads] for t in flat]
        sample_flops = w.bwd_flops() * heads / w.heads

        def step():
            oracle.attention_forward_backward(*sample, w.causal, w.scale, lib=lib)

        desc = "first %d of %d heads of %s per step (fp64 fwd+bwd)" % (heads, w.heads, w.name)
    else:
        rows = int(max(1, min(w.N, w.N * per_step_budget / t_head)))
        idx = np.unique(np.linspace(0, w.N - 1, rows).astype(np.int64))
        h0 = [t[0, 0] for t in flat]
        sample_flops = w.bwd_flops() / w.heads * len(idx) / w.N

        def step():
            oracle.attention_head_rows(*h0, w.causal, w.scale, idx, [], lib=lib)

        desc = ("%d evenly spaced query rows of head 0 of %s per step (fp64 O, L, dQ); "
                "FLOPs counted pro rata" % (len(idx), w.name))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = sample_flops * args.steps / el / 1e12
    cores = oracle.max_threads(lib)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) bf16 inputs (no dataset)",
        "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE)
    p.add_argument("--batch", type=int, default=0,
                   help="run the workload with this many batch elements instead (a smaller "
                        "case of the same kernels, for profiler captures); 0 = as named")
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--leg", default="attention",
                   choices=["attention", "fp8_forward", "fp8_backward", "dq_separate", "ssd"],
                   help="run one other leg alone on --workload (for profiler captures); "
                        "prints its timing, not the benchmark line")
    args = p.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        p.error("--warmup must be >= 3")
    if args.leg != "attention":
        line = run_leg(args)
    else:
        line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist

        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
