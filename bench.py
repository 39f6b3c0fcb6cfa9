#!/usr/bin/env python
"""Benchmark of the linear-attention library on one GB300 (or N replicas).

Headline (the JSON line's `value`): causal chunked forward, bf16 in / fp32
accumulate, B=4 H=8 N=2048 dk=dv=64, chunk 128, in tokens/s (B*N sequence
positions per second; all heads of a position count once).  One step is one
`la_forward_causal` over one batch.  Steps run from a CUDA graph; 16 input /
output buffer sets are rotated (537 MB > 4x the 129 MB L2) so every step reads
q, k, v from HBM.

Also reported ("paths"): the long causal forward (B=1 H=32 N=65536 d=128),
the non-causal forward (B=8 H=12 N=4096 d=64), the decode step (128 x 32
heads, d=128, fp32 state) and its prefill state, the decayed-state, gated-state
and feature-map variants, the backward pass, and FAVOR+ (features alone, causal,
non-causal and decode), each with its roofline fraction.

`--impl reference` times the float64 CPU oracle (the only reference this
method has) on a bounded sample of the same workload, on the host cores.

Multi-GPU: each rank runs its own replica of the workload (independent (b,h)
sequences: no collective on the data path); `value` is the work of all ranks
divided by the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "causal linear-attn fwd tokens/s & TFLOP/s (%roofline); decode tokens/s (%HBM BW)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


# --------------------------------------------------------------------------- accounting
def causal_flops(BH, N, dk, dv, chunk):
    """Algorithmic flop (2 per MAC): masked half of each intra-chunk tile only,
    BH*N*[(C+1)(dk+dv) + 4*dk*dv]."""
    return float(BH) * N * ((chunk + 1) * (dk + dv) + 4 * dk * dv)


def noncausal_flops(BH, N, dk, dv):
    return float(BH) * N * (4 * dk * dv + 3 * dk + dv)


def decode_flops_per_step(BH, dk, dv):
    return float(BH) * (4 * dk * dv + 6 * dk)


def forward_bytes(BH, N, dk, dv, elem):
    """Read q, k, v once and write o once."""
    return BH * N * (2 * dk + 2 * dv) * elem


def decode_bytes_per_step(BH, dk, dv, elem):
    """Read + write fp32 S and z, read q, k, v, write o."""
    return BH * (8 * dk * dv + 8 * dk + (2 * dk + 2 * dv) * elem)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def roofline(flops, nbytes, seconds, peaks, source, traffic=None, burst=True):
    """Bound = the slower of flops at the bf16 dense peak and bytes at HBM bandwidth."""
    tflops_peak = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
    t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_cmp = flops / (tflops_peak * 1e12)
    if t_mem >= t_cmp:
        achieved = nbytes / seconds / 1e9
        r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = flops / seconds / 1e12
        r = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tflops_peak, "unit": "TFLOP/s",
             "frac": round(achieved / tflops_peak, 4)}
    r["traffic"] = traffic
    r["peak_source"] = "%s (%s)" % (source, "MEASURED_PEAKS.json" if source == "measured" else "recipe fallback")
    r["algorithmic_bytes"] = int(nbytes)
    r["algorithmic_flop"] = flops
    r["tflops"] = round(flops / seconds / 1e12, 3)
    return r


# fp32 CUDA-core peak for the paths that run fp32 FMAs (no tensor cores): 152 SMs x 128
# FP32 lanes x 2 flop per FMA x the 2070 MHz maximum SM clock.
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def roofline_alu(flops, nbytes, seconds, peaks, source, traffic=None):
    """Roofline of an fp32 CUDA-core path: the slower of flops at the fp32 ALU peak
    and bytes at the measured HBM bandwidth."""
    t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_alu = flops / (FP32_ALU_TFLOPS * 1e12)
    if t_mem >= t_alu:
        achieved = nbytes / seconds / 1e9
        r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = flops / seconds / 1e12
        r = {"bound": "alu", "achieved": round(achieved, 2), "peak": round(FP32_ALU_TFLOPS, 1), "unit": "TFLOP/s",
             "frac": round(achieved / FP32_ALU_TFLOPS, 4)}
    r["traffic"] = traffic
    r["peak_source"] = ("derived fp32 ALU peak (152 SMs x 128 lanes x 2 x 2.07 GHz)" if r["bound"] == "alu" else
                        "%s (%s)" % (source, "MEASURED_PEAKS.json" if source == "measured" else "recipe fallback"))
    r["algorithmic_bytes"] = int(nbytes)
    r["algorithmic_flop"] = flops
    r["tflops"] = round(flops / seconds / 1e12, 3)
    return r


def ncu_traffic(kernel_tag):
    """DRAM bytes per launch from a committed ncu summary, if it still matches the
    kernel source (profiles/<tag>.md holds `traffic_bytes_per_launch:`,
    `source_file:` -- one path, or several separated by commas -- and
    `source_sha256:`, the SHA-256 of those files' bytes concatenated in that
    order); None otherwise."""
    import hashlib
    path = os.path.join(ROOT, "profiles", kernel_tag + ".md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_file", "source_sha256")):
            k, v = line.strip().split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    try:
        h = hashlib.sha256()
        for f in fields["source_file"].split(","):
            h.update(open(os.path.join(ROOT, f.strip()), "rb").read())
        sha = h.hexdigest()
        if sha != fields["source_sha256"]:
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def whole_job_throughput(world: int, units_per_rank: float, steps: int, slowest_secs: float) -> float:
    """Units per second of the whole job: every rank processes `units_per_rank`
    per step (weak scaling), and the job takes as long as its slowest rank."""
    return world * units_per_rank * steps / slowest_secs


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU works.

    Each sample carries nvidia-smi's own timestamp; stop(window=(t0, t1)) reports
    the samples taken inside that host-time window (the timed region) as the ones
    under load, and the throttle reasons seen anywhere in the run."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0, period_ms=20):
        self.proc = None
        self.gpu_index = gpu_index
        self.period_ms = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    @staticmethod
    def _epoch(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarise(out, window, self.period_ms)

    @classmethod
    def summarise(cls, text, window, period_ms):
        """Median SM clock of the samples inside `window` (all samples if none is),
        the maximum clock, and every throttle reason seen."""
        rows = [r for r in csv.reader(io.StringIO(text)) if len(r) >= 10]
        sm, smax, reasons, inside = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                s, m = float(r[2]), float(r[3])
            except ValueError:
                continue
            smax = m
            sm.append(s)
            t = cls._epoch(r[0])
            if window is not None and t is not None and window[0] <= t <= window[1]:
                inside.append(s)
            for n, val in zip(names, r[6:10]):
                if val.strip().lower().startswith("active"):
                    reasons.add(n)
        use = inside if inside else sm
        return {"sm_mhz": statistics.median(use) if use else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "samples_in_timed_region": len(inside),
                "sampling_ms": period_ms}


# --------------------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() and self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# --------------------------------------------------------------------------- GPU arm
def _graph_steps(torch, fn, n, stream):
    """Capture n calls of fn(i) into CUDA graphs of at most 256 steps."""
    graphs = []
    i = 0
    while i < n:
        m = min(256, n - i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(i, i + m):
                fn(j)
        graphs.append(g)
        i += m
    return graphs


def time_graph_steps(torch, la, fn, steps, warmup, dist, sampler=None):
    """W warm-up steps, then exactly `steps` timed steps, all replayed from CUDA
    graphs on one side stream; CUDA events on that stream bracket the timed
    steps, with a barrier and device synchronisation on both sides.  Returns
    (seconds, kernel launches inside the timed steps)."""
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        fn(0)  # plain call first: sets kernel attributes outside capture
    torch.cuda.synchronize()
    n0 = la.la_kernel_launches()
    timed = _graph_steps(torch, fn, steps, stream)
    launches = la.la_kernel_launches() - n0
    warm = _graph_steps(torch, fn, warmup, stream) if warmup > 0 else []
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for g in warm:
            g.replay()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        time.sleep(0.25)  # let the sampler take its first reading before the timed region
    t_begin = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for g in timed:
            g.replay()
        stop.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if sampler is not None:
        time.sleep(2.5 * sampler.period_ms / 1e3)  # one more reading after the timed region
    clocks = sampler.stop(window=(t_begin, t_end)) if sampler is not None else None
    dist.barrier()
    secs = start.elapsed_time(stop) / 1e3
    del timed, warm
    return secs, launches, clocks


def dev_copy(torch, x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def n_rotations(bytes_per_set):
    return max(2, math.ceil(4 * L2_BYTES / bytes_per_set))


def bench_causal_headline(torch, la, w, steps, warmup, dist, peaks, src, sampler=None):
    q, k, v = workloads.forward_inputs(w)
    es = 2 if w.dtype == "bf16" else 4
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, es)
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, w.dtype) for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_forward_causal(s[0], s[1], s[2], s[3], chunk=w.chunk, eps=w.eps)

    secs, launches, clocks = time_graph_steps(torch, la, step, steps, warmup, dist, sampler)
    return secs, launches, nbytes, R, clocks


def bench_causal_e2e_pipelined(torch, la, w, steps, warmup, dist, nbuf=2):
    """The public call with host buffers: every step copies its q, k, v from
    pinned host memory to the device, calls la_forward_causal once and copies o
    back to pinned host memory.  The copies overlap across steps the way a
    serving loop would: `nbuf` device buffer sets; step i's inputs are copied in
    on one stream while step i - 1 computes on another and step i - 2's o is
    copied out on a third."""
    q, k, v = workloads.forward_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def pinned(x):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if w.dtype == "bf16" else x)
        t = t.view(tdt) if w.dtype == "bf16" else t
        return t.pin_memory()

    hq, hk, hv = pinned(q), pinned(k), pinned(v)
    ho = torch.empty(hv.shape, dtype=tdt).pin_memory()
    bufs = [[torch.empty(t.shape, dtype=tdt, device="cuda") for t in (hq, hk, hv, hv)] for _ in range(nbuf)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def step(i):
        b = i % nbuf
        dq, dk_, dv_, do = bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_comp[b])  # the compute that read buffer b is done
            dq.copy_(hq, non_blocking=True)
            dk_.copy_(hk, non_blocking=True)
            dv_.copy_(hv, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[b])
            if used[b]:
                s_comp.wait_event(ev_out[b])  # buffer b's previous o has been copied out
            la.la_forward_causal(dq, dk_, dv_, do, chunk=w.chunk, eps=w.eps)
            ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            ho.copy_(do, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(max(warmup, 1)):
        step(i)
    torch.cuda.synchronize()
    dist.barrier()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    stop.record(s_out)
    torch.cuda.synchronize()
    dist.barrier()
    secs = start.elapsed_time(stop) / 1e3
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size()
    return secs, h2d, d2h


def bench_path_causal_long(torch, la, reps, peaks, src):
    w = workloads.CAUSAL_BF16_LONG
    q, k, v = workloads.device_forward_inputs(w)
    o = torch.empty_like(v)

    def step(i):
        la.la_forward_causal(q, k, v, o, chunk=w.chunk, eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2)
    fl = causal_flops(w.BH, w.N, w.dk, w.dv, w.chunk)
    return {"workload": w.name, "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("causal_long")),
            "l2": "inputs 2.1 GB > L2"}


def bench_path_noncausal(torch, la, reps, peaks, src):
    w = workloads.NONCAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2)
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_forward_noncausal(s[0], s[1], s[2], s[3], eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = noncausal_flops(w.BH, w.N, w.dk, w.dv)
    return {"workload": w.name, "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("noncausal")),
            "l2": "%d rotating buffer sets" % R}


def bench_path_decode(torch, la, steps, peaks, src):
    w = workloads.DECODE_BF16
    (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
    S, z = la.la_prefill_state(kp, vp)
    del qp, kp, vp
    o = torch.empty((w.B, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    S0, z0 = S.clone(), z.clone()

    def step(i):
        la.la_decode_step(S, z, qd[i], kd[i], vd[i], o, eps=w.eps)

    n = min(steps, w.steps)
    secs, launches, _ = time_graph_steps(torch, la, step, n, 3, Dist())
    S.copy_(S0)
    z.copy_(z0)
    t = secs / n
    nbytes = decode_bytes_per_step(w.BH, w.dk, w.dv, 2)
    fl = decode_flops_per_step(w.BH, w.dk, w.dv)
    return {"workload": w.name, "value": round(w.B / t, 1), "unit": "tokens/s",
            "head_steps_per_s": round(w.BH / t, 1), "ms_per_step": round(t * 1e3, 5), "steps": n,
            "launches_per_step": launches / n,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("decode")),
            "l2": "state 270 MB > L2"}


def bench_path_prefill(torch, la, reps, peaks, src):
    """la_prefill_state on the decode workload's prefill (k, v 1.07 GB > L2): S, z
    fp32 sums over 512 tokens of 4096 heads at d = 128."""
    w = workloads.DECODE_BF16
    (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
    del qp, qd, kd, vd
    S = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    z = torch.empty((w.B, w.H, w.dk), dtype=torch.float32, device="cuda")

    def step(i):
        la.la_prefill_state(kp, vp, S, z)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    nbytes = w.BH * w.N * (w.dk + w.dv) * 2 + w.BH * w.dk * (w.dv + 1) * 4
    fl = 2.0 * w.BH * w.N * w.dk * (w.dv + 1)
    return {"workload": "prefill_state_bf16_b%d_h%d_n%d_d%d" % (w.B, w.H, w.N, w.dk),
            "value": round(w.B * w.N / t, 1), "unit": "tokens/s", "ms_per_step": round(t * 1e3, 4),
            "launches_per_step": launches / reps,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("prefill_state")),
            "l2": "k, v 1.07 GB > L2"}


def bench_path_causal_decay(torch, la, reps, peaks, src):
    """la_forward_causal_decay on the headline causal shape (B=4 H=8 N=2048 d=64,
    chunk 128, bf16) with per-head decays from 0.9 to 0.999; CUDA cores, fp32."""
    w = workloads.CAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2)
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]
    g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda()

    def step(i):
        s = sets[i % R]
        la.la_forward_causal_decay(s[0], s[1], s[2], g, s[3], chunk=w.chunk, eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = causal_flops(w.BH, w.N, w.dk, w.dv, w.chunk)
    return {"workload": w.name + "_decay", "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("causal_decay")),
            "l2": "%d rotating buffer sets" % R}


def bench_path_causal_gated(torch, la, reps, peaks, src):
    """la_forward_causal_gated on the headline causal shape (B=4 H=8 N=2048 d=64, bf16)
    with one gate per (token, key feature) drawn uniformly in [0.8, 1); the gates are a
    third input stream (fp32, the size of q and k together): bytes read q, k, v, alpha,
    written o.  CUDA cores, fp32, in chunks of 32 tokens."""
    w = workloads.CAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    alpha = np.random.default_rng(w.seed + 7).uniform(0.8, 1.0, size=(w.B, w.H, w.N, w.dk)).astype(np.float32)
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2) + alpha.nbytes
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)] + [torch.from_numpy(alpha).cuda()]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_forward_causal_gated(s[0], s[1], s[2], s[3], s[4], eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = float(w.BH) * w.N * (6 * w.dk * w.dv + 4 * w.dk)  # per token: gate, update, read (2 flop per MAC)
    return {"workload": w.name + "_gated", "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "roofline": roofline_alu(fl, nbytes, t, peaks, src, None),
            "l2": "%d rotating buffer sets" % R}


def bench_path_prefill_decay(torch, la, reps, peaks, src):
    """la_prefill_state_decay on the decode workload's prefill (4096 heads x 512
    tokens, d = 128, per-head decays 0.9 .. 0.999)."""
    w = workloads.DECODE_BF16
    (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
    del qp, qd, kd, vd
    g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda()
    S = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    z = torch.empty((w.B, w.H, w.dk), dtype=torch.float32, device="cuda")

    def step(i):
        la.la_prefill_state_decay(kp, vp, g, S, z)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    nbytes = w.BH * w.N * (w.dk + w.dv) * 2 + w.BH * w.dk * (w.dv + 1) * 4
    fl = 2.0 * w.BH * w.N * w.dk * (w.dv + 1)
    return {"workload": "prefill_state_decay_bf16_b%d_h%d_n%d_d%d" % (w.B, w.H, w.N, w.dk),
            "value": round(w.B * w.N / t, 1), "unit": "tokens/s", "ms_per_step": round(t * 1e3, 4),
            "launches_per_step": launches / reps,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("prefill_state_decay")),
            "l2": "k, v 1.07 GB > L2"}


def bench_path_causal_variant(torch, la, reps, peaks, src, tag, decay, fmap, shift, normalize):
    """la_forward_causal_ex on the headline causal shape (B=4 H=8 N=2048 d=64, chunk
    128, bf16) with a feature map, normaliser choice and optional per-head decay."""
    w = workloads.CAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2)
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]
    g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda() if decay else None

    def step(i):
        s = sets[i % R]
        la.la_forward_causal_ex(s[0], s[1], s[2], s[3], gamma=g, feature_map=fmap, shift=shift,
                                normalize=normalize, chunk=w.chunk, eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = causal_flops(w.BH, w.N, w.dk, w.dv, w.chunk)
    return {"workload": w.name + "_" + tag, "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "variant": {"feature_map": fmap, "shift": shift, "normalize": normalize, "decay": decay},
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("causal_" + tag)),
            "l2": "%d rotating buffer sets" % R}


def bench_path_noncausal_variant(torch, la, reps, peaks, src, tag, fmap, shift, normalize):
    """la_forward_noncausal_ex on the non-causal workload (B=8 H=12 N=4096 d=64, bf16)."""
    w = workloads.NONCAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2)
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_forward_noncausal_ex(s[0], s[1], s[2], s[3], feature_map=fmap, shift=shift, normalize=normalize,
                                   eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = noncausal_flops(w.BH, w.N, w.dk, w.dv)
    return {"workload": w.name + "_" + tag, "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "variant": {"feature_map": fmap, "shift": shift, "normalize": normalize},
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("noncausal_" + tag)),
            "l2": "%d rotating buffer sets" % R}


def bench_path_backward(torch, la, reps, peaks, src):
    """la_backward_causal on the headline causal shape (B=4 H=8 N=2048 d=64, bf16): read
    q, k, v, dO and write dq, dk, dv once; bf16 operands on the tensor cores with fp32
    accumulation.  Algorithmic flop: three times the forward's at chunk 128 (the
    masked half of each intra-chunk tile); the bound is the slower of those flop at
    the bf16 peak and the bytes at HBM bandwidth."""
    w = workloads.CAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    dout = workloads.random_inputs(w.seed + 100, w.B, w.H, w.N, w.dv, w.dv, "bf16")[2]
    nbytes = w.BH * w.N * (4 * w.dk + 3 * w.dv) * 2
    R = n_rotations(nbytes)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v, dout)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[0]), torch.empty_like(base[1]),
                                         torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_backward_causal(s[0], s[1], s[2], s[3], s[4], s[5], s[6], eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = 3.0 * causal_flops(w.BH, w.N, w.dk, w.dv, 128)
    return {"workload": w.name + "_backward", "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("backward")),
            "l2": "%d rotating buffer sets" % R}


FAVOR_SIGMA = 0.5  # inputs of the FAVOR+ paths: N(0, 0.25), about the Performer's d^(-1/4) input scale at d = 64


def favor_flops(rows, d, m):
    """Projection flop of FAVOR+ features for `rows` input rows (2 per MAC)."""
    return 2.0 * rows * d * m


def bench_path_causal_favor(torch, la, reps, peaks, src):
    """la_forward_causal_favor on the headline causal shape (B=4 H=8 N=2048 d=64, chunk 128,
    bf16) with m = 64 orthogonal random features: features of q and k (one launch), then the
    causal forward on them.  Algorithmic bytes: q, k, v, w read and o written once (the
    features' round trip through HBM is this design's, not the method's)."""
    w = workloads.CAUSAL_BF16
    m = 64
    q, k, v = workloads.random_inputs(w.seed, w.B, w.H, w.N, w.dk, w.dv, "bf16", sigma=FAVOR_SIGMA)
    wp = dev_copy(torch, workloads.favor_projection(w.seed + 1, m, w.dk, "bf16"), "bf16")
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2) + m * w.dk * 2
    R = n_rotations(nbytes + 2 * w.BH * w.N * m * 2)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_forward_causal_favor(s[0], s[1], s[2], wp, s[3], chunk=w.chunk, eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = favor_flops(2 * w.BH * w.N, w.dk, m) + causal_flops(w.BH, w.N, m, w.dv, w.chunk)
    return {"workload": w.name + "_favor_m%d" % m, "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps, "m": m,
            "sigma": FAVOR_SIGMA,
            "roofline": roofline(fl, nbytes, t, peaks, src, None),
            "l2": "%d rotating buffer sets" % R}


def bench_path_favor_features(torch, la, reps, peaks, src):
    """la_favor_features alone over the rows of the headline shape's q and k together
    (x [8, 8, 2048, 64] bf16, m = 64): read x and w, write phi once."""
    w = workloads.CAUSAL_BF16
    m = 64
    x = workloads.random_inputs(w.seed, 2 * w.B, w.H, w.N, w.dk, w.dv, "bf16", sigma=FAVOR_SIGMA)[0]
    wp = dev_copy(torch, workloads.favor_projection(w.seed + 1, m, w.dk, "bf16"), "bf16")
    rows = 2 * w.BH * w.N
    nbytes = rows * (w.dk + m) * 2 + m * w.dk * 2
    R = n_rotations(nbytes)
    base = dev_copy(torch, x, "bf16")
    sets = [(base.clone(), torch.empty(base.shape[:-1] + (m,), dtype=base.dtype, device=base.device))
            for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_favor_features(s[0], wp, s[1])

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    return {"workload": "favor_features_rows%d_d%d_m%d" % (rows, w.dk, m), "value": round(rows / t, 1),
            "unit": "rows/s", "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps,
            "roofline": roofline(favor_flops(rows, w.dk, m), nbytes, t, peaks, src, ncu_traffic("favor_features")),
            "l2": "%d rotating buffer sets" % R}


def bench_path_noncausal_favor(torch, la, reps, peaks, src):
    """la_forward_noncausal_favor on the non-causal workload (B=8 H=12 N=4096 d=64, bf16), m = 64."""
    w = workloads.NONCAUSAL_BF16
    m = 64
    q, k, v = workloads.random_inputs(w.seed, w.B, w.H, w.N, w.dk, w.dv, "bf16", sigma=FAVOR_SIGMA)
    wp = dev_copy(torch, workloads.favor_projection(w.seed + 1, m, w.dk, "bf16"), "bf16")
    nbytes = forward_bytes(w.BH, w.N, w.dk, w.dv, 2) + m * w.dk * 2
    R = n_rotations(nbytes + 2 * w.BH * w.N * m * 2)
    base = [dev_copy(torch, x, "bf16") for x in (q, k, v)]
    sets = [[t.clone() for t in base] + [torch.empty_like(base[2])] for _ in range(R)]

    def step(i):
        s = sets[i % R]
        la.la_forward_noncausal_favor(s[0], s[1], s[2], wp, s[3], eps=w.eps)

    secs, launches, _ = time_graph_steps(torch, la, step, reps, 3, Dist())
    t = secs / reps
    fl = favor_flops(2 * w.BH * w.N, w.dk, m) + noncausal_flops(w.BH, w.N, m, w.dv)
    return {"workload": w.name + "_favor_m%d" % m, "value": round(w.B * w.N / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 4), "launches_per_step": launches / reps, "m": m,
            "sigma": FAVOR_SIGMA,
            "roofline": roofline(fl, nbytes, t, peaks, src, None),
            "l2": "%d rotating buffer sets" % R}


def bench_path_decode_favor(torch, la, steps, peaks, src):
    """la_decode_step_favor on the decode workload (128 x 32 heads, d = 128, fp32 state) with
    m = 128 features: the features of the step's q and k (8192 rows, one launch) and the
    decode step on them.  The prefill state comes from la_prefill_state_favor.  Inputs are
    scaled to sigma = 0.5 (the FAVOR+ input scale)."""
    w = workloads.DECODE_BF16
    m = 128
    (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
    for t in (qd, kd):
        t.mul_(FAVOR_SIGMA)
    kp.mul_(FAVOR_SIGMA)
    wp = dev_copy(torch, workloads.favor_projection(w.seed + 1, m, w.dk, "bf16"), "bf16")
    S, z = la.la_prefill_state_favor(kp, vp, wp)
    del qp, kp, vp
    o = torch.empty((w.B, w.H, w.dv), dtype=torch.bfloat16, device="cuda")

    def step(i):
        la.la_decode_step_favor(S, z, qd[i], kd[i], vd[i], wp, o, eps=w.eps)

    n = min(steps, w.steps)
    secs, launches, _ = time_graph_steps(torch, la, step, n, 3, Dist())
    t = secs / n
    nbytes = decode_bytes_per_step(w.BH, m, w.dv, 2) + m * w.dk * 2
    fl = decode_flops_per_step(w.BH, m, w.dv) + favor_flops(2 * w.BH, w.dk, m)
    return {"workload": w.name + "_favor_m%d" % m, "value": round(w.B / t, 1), "unit": "tokens/s",
            "head_steps_per_s": round(w.BH / t, 1), "ms_per_step": round(t * 1e3, 5), "steps": n,
            "launches_per_step": launches / n, "m": m, "sigma": FAVOR_SIGMA,
            "roofline": roofline(fl, nbytes, t, peaks, src, None),
            "l2": "state 270 MB > L2"}


def bench_path_decode_decay(torch, la, steps, peaks, src):
    """la_decode_step_decay on the decode workload (4096 heads, d = 128, fp32 state)."""
    w = workloads.DECODE_BF16
    (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
    g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda()
    S, z = la.la_prefill_state_decay(kp, vp, g)
    del qp, kp, vp
    o = torch.empty((w.B, w.H, w.dv), dtype=torch.bfloat16, device="cuda")

    def step(i):
        la.la_decode_step_decay(S, z, qd[i], kd[i], vd[i], g, o, eps=w.eps)

    n = min(steps, w.steps)
    secs, launches, _ = time_graph_steps(torch, la, step, n, 3, Dist())
    t = secs / n
    nbytes = decode_bytes_per_step(w.BH, w.dk, w.dv, 2)
    fl = decode_flops_per_step(w.BH, w.dk, w.dv)
    return {"workload": w.name + "_decay", "value": round(w.B / t, 1), "unit": "tokens/s",
            "ms_per_step": round(t * 1e3, 5), "steps": n, "launches_per_step": launches / n,
            "roofline": roofline(fl, nbytes, t, peaks, src, ncu_traffic("decode_decay")),
            "l2": "state 270 MB > L2"}


# --------------------------------------------------------------------------- CPU oracle
def oracle_causal_sample(w, target_s=10.0, max_reps=100000):
    """The float64 oracle (as it stands) on a bounded sample of workload w:
    whole (b,h) sequences, repeated until about target_s seconds.  Returns
    (tokens/s scaled to full positions, threads, description)."""
    import oracle
    orc = oracle.get()
    q, k, v = workloads.forward_inputs(w)
    qh, kh, vh = (x.reshape((w.BH,) + x.shape[2:]) for x in (q, k, v))
    nh = w.BH
    t0 = time.time()
    reps = 0
    while True:
        orc.causal_recurrent(qh[:nh], kh[:nh], vh[:nh], w.eps)
        reps += 1
        el = time.time() - t0
        if el >= target_s or reps >= max_reps:
            break
    head_tokens = reps * nh * w.N
    value = head_tokens / w.H / el
    desc = "%d pass(es) of all %d (b,h) sequences x %d positions, float64 recurrence, %.1f s" % (
        reps, nh, w.N, el)
    return value, orc.num_threads(), desc, el


def run_reference(args, dist):
    """Reference arm: the float64 CPU oracle on the host cores, same metric and
    config; each step is a bounded sample (8 of the 32 sequences)."""
    if dist.rank != 0:
        return 0
    import oracle
    w = workloads.CAUSAL_BF16
    orc = oracle.get()
    q, k, v = workloads.forward_inputs(w)
    qh, kh, vh = (x.reshape((w.BH,) + x.shape[2:]) for x in (q, k, v))
    nh = 8
    for _ in range(args.warmup):
        orc.causal_recurrent(qh[:nh], kh[:nh], vh[:nh], w.eps)
    t0 = time.time()
    for _ in range(args.steps):
        orc.causal_recurrent(qh[:nh], kh[:nh], vh[:nh], w.eps)
    el = time.time() - t0
    value = args.steps * nh * w.N / w.H / el
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "dk": w.dk, "dv": w.dv,
                   "chunk": w.chunk, "inputs": "bf16, seed %d" % w.seed},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": orc.num_threads(),
                         "kind": "oracle",
                         "sample": "each step: %d of %d (b,h) sequences x %d positions; value scaled per "
                                   "full position (/H)" % (nh, w.BH, w.N)},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, dist):
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    from causal_kernelized_attention_gb300 import build as la_build
    if dist.local_rank == 0:
        la_build.build()
    dist.barrier()
    import causal_kernelized_attention_gb300 as la
    la.load_library()
    peaks, src = load_peaks()
    w = workloads.CAUSAL_BF16

    sampler = ClockSampler(gpu_index=torch.cuda.current_device()) if dist.rank == 0 else None
    secs, launches, nbytes, R, clocks = bench_causal_headline(torch, la, w, args.steps, args.warmup, dist, peaks,
                                                              src, sampler)
    secs_max = dist.max(secs)
    t_step = secs_max / args.steps
    value = whole_job_throughput(dist.world, w.B * w.N, args.steps, secs_max)
    fl = causal_flops(w.BH, w.N, w.dk, w.dv, w.chunk)
    roof = roofline(fl, nbytes, secs / args.steps, peaks, src, ncu_traffic("causal_headline"))

    e2e_secs, h2d, d2h = bench_causal_e2e_pipelined(torch, la, w, max(10, min(args.steps, 200)), args.warmup, dist)
    e2e_steps = max(10, min(args.steps, 200))
    e2e_value = whole_job_throughput(dist.world, w.B * w.N, e2e_steps, dist.max(e2e_secs))

    # The headline again over a window of >= 200 ms (the same graphs replayed), so
    # that the clock record has samples inside the timed region.
    window = None
    if not args.headline_only and args.window_steps > 0:
        s3 = ClockSampler(gpu_index=torch.cuda.current_device()) if dist.rank == 0 else None
        wsecs, _, _, _, wclocks = bench_causal_headline(torch, la, w, args.window_steps, args.warmup, dist, peaks,
                                                        src, s3)
        wt = dist.max(wsecs) / args.window_steps
        window = {"steps": args.window_steps, "seconds": round(dist.max(wsecs), 4), "ms_per_step": round(wt * 1e3, 5),
                  "value": round(whole_job_throughput(dist.world, w.B * w.N, args.window_steps, dist.max(wsecs)), 1),
                  "frac": roofline(fl, nbytes, wt, peaks, src)["frac"], "clocks": wclocks}

    paths = {}
    if not args.headline_only:
        s2 = ClockSampler(gpu_index=torch.cuda.current_device(), period_ms=100).start() if dist.rank == 0 else None
        t_paths = time.time()
        paths["causal_long"] = bench_path_causal_long(torch, la, args.path_reps, peaks, src)
        paths["noncausal"] = bench_path_noncausal(torch, la, max(args.path_reps, 20), peaks, src)
        paths["decode"] = bench_path_decode(torch, la, 1024, peaks, src)
        paths["prefill_state"] = bench_path_prefill(torch, la, max(args.path_reps, 20), peaks, src)
        paths["causal_decay"] = bench_path_causal_decay(torch, la, max(args.path_reps, 20), peaks, src)
        paths["decode_decay"] = bench_path_decode_decay(torch, la, 1024, peaks, src)
        paths["prefill_state_decay"] = bench_path_prefill_decay(torch, la, max(args.path_reps, 20), peaks, src)
        paths["causal_gated"] = bench_path_causal_gated(torch, la, max(args.path_reps, 20), peaks, src)
        reps = max(args.path_reps, 20)
        paths["causal_relu"] = bench_path_causal_variant(torch, la, reps, peaks, src, "relu", False, "relu", 0.0, True)
        paths["causal_retention"] = bench_path_causal_variant(torch, la, reps, peaks, src, "retention", True,
                                                              "identity", 0.0, False)
        paths["noncausal_relu_nonorm"] = bench_path_noncausal_variant(torch, la, reps, peaks, src, "relu_nonorm",
                                                                      "relu", 0.0, False)
        paths["backward"] = bench_path_backward(torch, la, reps, peaks, src)
        paths["favor_features"] = bench_path_favor_features(torch, la, reps, peaks, src)
        paths["causal_favor"] = bench_path_causal_favor(torch, la, reps, peaks, src)
        paths["noncausal_favor"] = bench_path_noncausal_favor(torch, la, reps, peaks, src)
        paths["decode_favor"] = bench_path_decode_favor(torch, la, 256, peaks, src)
        if s2:
            paths["clocks"] = s2.stop(window=(t_paths, time.time()))

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "dk": w.dk, "dv": w.dv,
                   "chunk": w.chunk, "accumulate": "fp32", "global_batch": w.B * dist.world,
                   "seq_len": w.N, "parallelism": "replicas x%d" % dist.world,
                   "l2": "%d rotating input/output sets (%.0f MB > 4x L2)" % (R, R * nbytes / 1e6),
                   "timing": "CUDA graph replay, CUDA events on the launch stream"},
        "tflops": roof["tflops"],
        "roofline": roof,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "overlap": "2 device buffer sets; step i's copies in, step i-1's compute and step i-2's "
                           "copy out on three streams (pinned host buffers)"},
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        val, cores, desc, el = oracle_causal_sample(w, target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(val, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    if window is not None:
        line["headline_window"] = window
    # Every secondary path in compact form, the gated ones (long causal, decode) last,
    # then the three gate fractions: the end of the line is what a truncated log keeps.
    if paths:
        order = [n for n in paths if n not in ("causal_long", "decode", "clocks")] + ["causal_long", "decode"]
        line["paths"] = {n: compact_path(paths[n], peaks) for n in order if n in paths}
        if "clocks" in paths:
            line["paths_clocks"] = paths["clocks"]
        line["gates"] = {"causal_headline_frac": roof["frac"],
                         "causal_long_frac": paths["causal_long"]["roofline"]["frac"],
                         "decode_hbm_frac": paths["decode"]["roofline"]["frac"],
                         "decode_dram_frac": compact_path(paths["decode"], peaks).get("dram_frac")}
    if args.details and dist.rank == 0:
        with open(args.details, "w") as f:
            json.dump({"headline_roofline": roof, "paths": paths, "headline_window": window}, f, indent=1)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def compact_path(p, peaks):
    """One secondary path in a few keys: throughput, time per step, roofline
    fraction (of algorithmic bytes or flop) and, where an ncu capture of the
    current kernel gives its DRAM bytes per launch, the fraction of the copy
    bandwidth those bytes reach (`dram_frac`)."""
    r = p["roofline"]
    c = {"workload": p["workload"], "value": p["value"], "unit": p["unit"], "ms": p["ms_per_step"],
         "bound": r["bound"], "frac": r["frac"]}
    if r.get("traffic"):
        secs = p["ms_per_step"] / 1e3
        c["dram_frac"] = round(r["traffic"] / secs / 1e9 / peaks["hbm_gbs"], 4)
    return c


PROFILE_CASES = ("headline", "causal_long", "causal_long_quarter", "noncausal", "decode", "prefill_state_quarter",
                 "causal_decay", "decode_decay", "prefill_state_decay_quarter", "causal_relu", "causal_retention",
                 "noncausal_relu_nonorm", "backward", "favor_features", "causal_favor")


def run_profile_case(name: str, launches: int) -> int:
    """A few plain launches of one workload (no graphs, no timing), for ncu.

    causal_long_quarter is the long causal workload at N = 16384 (537 MB of
    q, k, v, o: above L2, small enough for multi-pass profiling);
    prefill_state_quarter is the decode workload's prefill state with a quarter
    of its heads (B = 32: 268 MB of k, v)."""
    import torch
    import causal_kernelized_attention_gb300 as la
    from causal_kernelized_attention_gb300 import build as la_build
    la_build.build()
    la.load_library()
    if name in ("favor_features", "causal_favor"):
        # favor_features: x [64, 8, 2048, 64] bf16 (268 MB of x and phi, above L2), m = 64;
        # causal_favor: the headline causal shape through la_forward_causal_favor, m = 64
        w = workloads.CAUSAL_BF16
        g = torch.Generator(device="cuda").manual_seed(w.seed)
        wp = torch.from_numpy(workloads.favor_projection(w.seed + 1, 64, w.dk, "bf16").view(np.int16)).cuda()
        wp = wp.view(torch.bfloat16)
        if name == "favor_features":
            x = (torch.randn((64, w.H, w.N, w.dk), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
            phi = torch.empty((64, w.H, w.N, 64), dtype=torch.bfloat16, device="cuda")
            for _ in range(launches):
                la.la_favor_features(x, wp, phi)
        else:
            q, k, v = ((torch.randn((w.B, w.H, w.N, w.dk), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
                       for _ in range(3))
            o = torch.empty_like(v)
            for _ in range(launches):
                la.la_forward_causal_favor(q, k, v, wp, o, chunk=w.chunk, eps=w.eps)
    elif name == "backward":
        w = workloads.CAUSAL_BF16
        q, k, v = workloads.device_forward_inputs(w)
        dout = torch.randn(v.shape, device="cuda").to(torch.bfloat16)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        for _ in range(launches):
            la.la_backward_causal(q, k, v, dout, dq, dk, dv, eps=w.eps)
    elif name in ("causal_relu", "causal_retention"):
        w = workloads.CAUSAL_BF16
        q, k, v = workloads.device_forward_inputs(w)
        o = torch.empty_like(v)
        retention = name == "causal_retention"
        g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda() if retention else None
        for _ in range(launches):
            la.la_forward_causal_ex(q, k, v, o, gamma=g, feature_map="identity" if retention else "relu",
                                    normalize=not retention, chunk=w.chunk, eps=w.eps)
    elif name == "noncausal_relu_nonorm":
        w = workloads.NONCAUSAL_BF16
        q, k, v = workloads.device_forward_inputs(w)
        o = torch.empty_like(v)
        for _ in range(launches):
            la.la_forward_noncausal_ex(q, k, v, o, feature_map="relu", normalize=False, eps=w.eps)
    elif name == "causal_decay":
        w = workloads.CAUSAL_BF16
        q, k, v = workloads.device_forward_inputs(w)
        o = torch.empty_like(v)
        g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda()
        for _ in range(launches):
            la.la_forward_causal_decay(q, k, v, g, o, chunk=w.chunk, eps=w.eps)
    elif name == "decode_decay":
        import dataclasses
        w = dataclasses.replace(workloads.DECODE_BF16, steps=launches)
        (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
        g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda()
        S, z = la.la_prefill_state_decay(kp, vp, g)
        o = torch.empty((w.B, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
        for t in range(launches):
            la.la_decode_step_decay(S, z, qd[t], kd[t], vd[t], g, o, eps=w.eps)
    elif name in ("headline", "causal_long", "causal_long_quarter"):
        w = workloads.CAUSAL_BF16 if name == "headline" else workloads.CAUSAL_BF16_LONG
        if name == "causal_long_quarter":
            import dataclasses
            w = dataclasses.replace(w, N=16384)
        q, k, v = workloads.device_forward_inputs(w)
        o = torch.empty_like(v)
        for _ in range(launches):
            la.la_forward_causal(q, k, v, o, chunk=w.chunk, eps=w.eps)
    elif name == "noncausal":
        w = workloads.NONCAUSAL_BF16
        q, k, v = workloads.device_forward_inputs(w)
        o = torch.empty_like(v)
        for _ in range(launches):
            la.la_forward_noncausal(q, k, v, o, eps=w.eps)
    elif name == "prefill_state_decay_quarter":
        import dataclasses
        w = dataclasses.replace(workloads.DECODE_BF16, B=workloads.DECODE_BF16.B // 4, steps=1)
        (qp, kp, vp), _ = workloads.device_decode_inputs(w)
        g = torch.from_numpy(workloads.decay_gammas(w.H)).cuda()
        S, z = la.la_prefill_state_decay(kp, vp, g)
        for _ in range(launches - 1):
            la.la_prefill_state_decay(kp, vp, g, S, z)
    elif name == "prefill_state_quarter":
        import dataclasses
        w = dataclasses.replace(workloads.DECODE_BF16, B=workloads.DECODE_BF16.B // 4, steps=1)
        (qp, kp, vp), _ = workloads.device_decode_inputs(w)
        S, z = la.la_prefill_state(kp, vp)
        for _ in range(launches - 1):
            la.la_prefill_state(kp, vp, S, z)
    else:
        import dataclasses
        w = dataclasses.replace(workloads.DECODE_BF16, steps=launches)
        (qp, kp, vp), (qd, kd, vd) = workloads.device_decode_inputs(w)
        S, z = la.la_prefill_state(kp, vp)
        o = torch.empty((w.B, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
        for t in range(launches):
            la.la_decode_step(S, z, qd[t], kd[t], vd[t], o, eps=w.eps)
    torch.cuda.synchronize()
    print("profile case %s: %d launches ok" % (name, launches))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--headline-only", action="store_true", help="skip the secondary paths")
    ap.add_argument("--path-reps", type=int, default=20, help="timed steps of the long causal path")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--window-steps", type=int, default=16384,
                    help="steps of the second, long-window headline timing (0: skip)")
    ap.add_argument("--details", default=None, help="write every path's full record (JSON) to this file")
    ap.add_argument("--profile-case", choices=PROFILE_CASES, default=None,
                    help="run a few plain launches of one workload (for ncu) instead of the benchmark")
    ap.add_argument("--profile-launches", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args.profile_case, args.profile_launches)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps; the line reports the count used
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)
    return run_gpu(args, dist)


if __name__ == "__main__":
    sys.exit(main())
