#!/usr/bin/env python
"""Batched Soft-DTW forward + backward throughput on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: the headline shape B=32, N=M=512, D=64, x,y ~ N(0,1), gamma=1, loss =
batch mean (SoftDTW-CUDA (PyTorch + Numba) README, "Key Benchmark"). One step =
forward + backward with input gradients in the unfused mode, then the same in the
fused mode, i.e. 2*B*N*M DP cells. Metric: DP cells per second (B*N*M per
forward+backward). Inputs are resident in HBM before the timed region; the L2 is
flushed (a 256 MiB write) between timed steps, outside the per-step events.

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample
of the same workload (the method has no runnable reference implementation).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SoftDTW fwd+bwd DP cells/s at B=32,N=M=512,D=64 (fused & unfused); peak MB"
B, N, M, D, GAMMA = 32, 512, 512, 64, 1.0
CELLS = B * N * M
WORKLOAD = "softdtw fwd+bwd B=32 N=M=512 D=64 gamma=1, unfused then fused"
FALLBACK_HBM_GBS = 6800.0
# Per-cell accounting of the method for the roofline (one forward + backward):
#   HBM bytes: unfused 28 (cost written, then read by the forward and by the
#   backward; R written and read; E written and read once for both contractions),
#   fused 8 (R written and read; costs recomputed on chip). The double-float state
#   counts R and the stored cost at 8 bytes: unfused 48, fused 16. Inputs read
#   and gradients written once come on top.
#   SFU operations: forward 2 ex2 + 1 lg2 (the three-term soft-min), backward
#   2 ex2 + 1 lg2 (the log-sum-exp of the three messages) + 1 ex2 (E itself).
ALG_BYTES = {("unfused", False): 28, ("fused", False): 8, ("unfused", True): 48, ("fused", True): 16}
FWD_EX2, FWD_LG2, BWD_EX2, BWD_LG2 = 2, 1, 3, 1
# SFU issue rate per SM and clock on this part: ex2 32, lg2 16 (a one-instruction
# microbenchmark with 8 independent chains per thread measured 31.7 and 15.9).
EX2_PER_SM_CLK, LG2_PER_SM_CLK = 32, 16
FALLBACK_SM_MHZ = 2070.0
# DRAM bytes (read + write) of one bwd_kernel launch of this workload's fused step
# from one ncu capture (`dram__bytes_read.sum + dram__bytes_write.sum`), with the
# SHA-256 of the sources that build the kernel at the time of the capture; the
# bench reports it only while those sources are unchanged (else null).
# profiles/bwd_kernel_headline.md: 71,442,432 read + 7,738,624 written.
BWD_TRAFFIC = {"sha256": "8c55defe62301a7354beda158f4df6f74b1d95c2a659e06e6ed3d9d7e5ca57c2", "bytes": 79181056}
BWD_SOURCES = ("wavefront.cu", "common.cuh", "channel.cuh", "kernels.h")
# kernels per step: unfused forward (operand images, cost tensor, wavefront) + backward
# (wavefront, gradient operand images, two gradient contractions), fused forward
# (operand images, wavefront with tensor-core costs) + backward (4)
LAUNCHES_PER_STEP = 3 + 4 + 2 + 4
# chunks of the batch in the end-to-end (host buffer) step
E2E_CHUNKS = 2


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------- reference arm

def time_max_over_ranks(total_ms, device=None):
    """The slowest rank's timed total (ms): every rank gets the max, so the job's
    throughput is the units all ranks processed over the longest time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(total_ms)
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, steps, cells_per_step, total_ms):
    """Whole-job cells/s: every rank runs `steps` steps of its own batch (weak scaling)."""
    return world * steps * cells_per_step / (total_ms * 1e-3)


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:  # rank 0 alone times the oracle; the others exit without work
        return 0
    import oracle
    from differentiable_series_alignment_gb300 import synth
    x, y = synth.iid_normal_pair(B, N, M, D, 1)
    cores = oracle.threads_used(0)
    sample = max(1, min(cores, B))  # problems per step: one per host core, run in parallel
    gl = np.full(sample, 1.0 / B)
    for _ in range(args.warmup):
        oracle.batch(x[:sample], y[:sample], GAMMA, grad_loss=gl)
    t0 = time.perf_counter()
    for k in range(args.steps):
        idx = [(k * sample + q) % B for q in range(sample)]
        oracle.batch(x[idx], y[idx], GAMMA, grad_loss=gl)
    dt = time.perf_counter() - t0
    value = args.steps * sample * N * M / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "cells/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD + f"; oracle sample {sample} problems per step", "B": B, "N": N, "M": M,
                   "D": D, "gamma": GAMMA},
        "cpu_baseline": {"value": value, "unit": "cells/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} of {B} problems per step, fwd+bwd with gradients, fp64"},
        "e2e": {"value": value, "unit": "cells/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- helpers

class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.rows = []
        self.proc = None
        self.uuid = uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=2)
        if not self.rows:
            return None
        sm = [float(r[1]) for r in self.rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) > 8:
                for n_, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n_)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def sm_clock_mhz():
    """Maximum SM clock: MEASURED_PEAKS.json's, else the part's nominal maximum."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(p)).get("sm_max_mhz") or 0)
        if v > 0:
            return v
    except Exception:
        pass
    return FALLBACK_SM_MHZ


def sfu_rates(num_sms):
    """(ex2/s, lg2/s) at the maximum SM clock."""
    hz = sm_clock_mhz() * 1e6
    return num_sms * EX2_PER_SM_CLK * hz, num_sms * LG2_PER_SM_CLK * hz


def sources_sha256(names):
    import hashlib
    h = hashlib.sha256()
    for n_ in names:
        with open(os.path.join(ROOT, "differentiable_series_alignment_gb300", "csrc", n_), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def roofline_bound(cells, hbm_bytes, ex2, lg2, hbm_gbs, rates):
    """The roofline time of `cells` DP cells moving `hbm_bytes` and issuing ex2/lg2
    per cell: the slower of HBM at its measured peak and the SFU at its issue rate."""
    t_hbm = hbm_bytes / (hbm_gbs * 1e9)
    t_sfu = cells * (ex2 / rates[0] + lg2 / rates[1])
    return {"hbm_us": t_hbm * 1e6, "sfu_us": t_sfu * 1e6, "bound": "hbm" if t_hbm >= t_sfu else "sfu",
            "bound_us": max(t_hbm, t_sfu) * 1e6}


def step_roofline(cells, io_bytes, mode_name, ext, hbm_gbs, rates, ms):
    """Roofline fraction of one forward + backward (both directions of the DP)."""
    r = roofline_bound(cells, cells * ALG_BYTES[(mode_name, ext)] + io_bytes, FWD_EX2 + BWD_EX2,
                       FWD_LG2 + BWD_LG2, hbm_gbs, rates)
    r["frac"] = r["bound_us"] / (ms * 1e3)
    return r


def cpu_baseline():
    import oracle
    from differentiable_series_alignment_gb300 import synth
    x, y = synth.iid_normal_pair(B, N, M, D, 1)
    cores = oracle.threads_used(0)
    gl = np.full(B, 1.0 / B)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.batch(x, y, GAMMA, grad_loss=gl)
        reps += 1
        dt = time.perf_counter() - t0
        if dt > 8.0 or reps >= 20:
            break
    # the same on one core: two problems of the batch, repeated for about a second
    t1 = time.perf_counter()
    reps1 = 0
    while True:
        oracle.batch(x[:2], y[:2], GAMMA, grad_loss=gl[:2], nthreads=1)
        reps1 += 1
        dt1 = time.perf_counter() - t1
        if dt1 > 1.0:
            break
    return {"value": reps * CELLS / dt, "unit": "cells/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x the full batch B=32 N=M=512 D=64, fwd+bwd with gradients, fp64, {dt:.1f} s",
            "single_core": {"value": reps1 * 2 * N * M / dt1, "unit": "cells/s", "cores": 1,
                            "sample": f"{reps1} x 2 problems of the batch, {dt1:.1f} s"}}


# --------------------------------------------------------------------------- the other workloads

def measure_per_config(L, synth, dev, flush, stream, hbm, rates, step_ns):
    """DP cells/s, peak device memory above the resident inputs and gradient buffers,
    and the roofline fraction (slower of HBM at the method's bytes and the SFU at its
    ex2/lg2 count, over the measured forward + backward) of every workload beside the
    headline: the small one, the length and width sweep in both modes, the long
    time-warped pairs at three gammas plus their normalized form, and 100 barycenter
    steps (with and without early stopping). The precision mode is the one the
    high-level API picks for the workload's batch-mean loss."""
    import torch
    from differentiable_series_alignment_gb300 import softdtw_barycenter

    def median_ms(fn, reps, warm=1):
        for _ in range(warm):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for k in range(reps):
            flush.fill_(k & 0xff)
            ev[k][0].record(stream)
            fn()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in ev]))

    def point(x, y, gamma, mode, reps, normalized=False):
        B_, N_, D_ = x.shape
        M_ = y.shape[1]
        gx, gy = torch.empty_like(x), torch.empty_like(y)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        op = L.OP_NORMALIZED if normalized else L.OP_FWD_BWD
        ws = L.workspace(op, B_, N_, M_, D_, mode, dev)
        loss = torch.empty(B_, device=dev)
        g = torch.full((B_,), 1.0 / B_, device=dev)
        if normalized:
            def fb():
                L.sdtw_normalized(x, y, gamma, mode, loss, g, gx, gy, ws)
        else:
            def fb():
                L.sdtw_forward(x, y, gamma, mode, loss, ws)
                L.sdtw_backward(x, y, gamma, mode, g, gx, gy, ws)
        ms = median_ms(fb, reps)
        assert L.sdtw_last_device_status(ws) == 0
        assert bool(torch.isfinite(loss).all()) and bool(torch.isfinite(gx).all())
        peak = (torch.cuda.max_memory_allocated(dev) - base) / 2**20
        cells = (3 if normalized else 1) * B_ * N_ * M_
        name = "fused" if mode & L.FUSED else "unfused"
        ext = bool(mode & L.EXTENDED)
        r = step_roofline(cells, 2 * B_ * (N_ + M_) * D_ * 4, name, ext, hbm, rates, ms)
        floor = 2 * (N_ + M_ - 1) * step_ns * 1e-6
        out = {"mode": name + ("+extended" if ext else ""), "ms": ms, "cells": cells,
               "cells_per_s": cells / (ms * 1e-3), "peak_MB_above_inputs": peak,
               "workspace_MB": ws.numel() / 2**20, "roofline_frac": r["frac"], "roofline": r,
               "latency_floor_ms": floor, "latency_frac": floor / ms}
        del ws, loss, gx, gy
        return out

    res = {}
    t0 = time.perf_counter()
    c = synth.WORKLOADS["small"]
    x, y = (torch.from_numpy(a).to(dev) for a in synth.iid_normal_pair(c["B"], c["N"], c["M"], c["D"], c["seed"]))
    prec = L.auto_precision(1.0, c["N"], c["M"], c["D"], c["B"])
    res["small"] = [dict(point(x, y, 1.0, m | prec, 20), B=c["B"], N=c["N"], M=c["M"], D=c["D"], gamma=1.0)
                    for m in (L.UNFUSED, L.FUSED)]

    c = synth.WORKLOADS["sweep"]
    pts = [(Ls, c["D_at_L"]) for Ls in c["L_sweep"]] + [(c["L_at_D"], Ds) for Ds in c["D_sweep"]]
    res["sweep"] = []
    for Ls, Ds in pts:
        x, y = (torch.from_numpy(a).to(dev)
                for a in synth.iid_normal_pair(32, Ls, Ls, Ds, c["seed"], repeat=Ls * 1000 + Ds))
        auto = L.auto_precision(1.0, Ls, Ls, Ds, 32)
        for prec in (0, L.EXTENDED):   # both precisions; `auto` marks the one the high-level API picks
            for m in (L.UNFUSED, L.FUSED):
                res["sweep"].append(dict(point(x, y, 1.0, m | prec, 5 if Ls <= 512 else 3), B=32, L=Ls, D=Ds,
                                         gamma=1.0, auto=(prec == auto)))
        del x, y

    c = synth.WORKLOADS["long_warped"]
    xn, yn = synth.warped_pair(c["B"], c["N"], c["D"], c["seed"])
    x, y = torch.from_numpy(xn).to(dev), torch.from_numpy(yn).to(dev)
    res["long_warped"] = []
    for gamma in c["gammas"]:
        m = L.FUSED | L.auto_precision(gamma, c["N"], c["M"], c["D"], c["B"])
        res["long_warped"].append(dict(point(x, y, gamma, m, 2), B=c["B"], N=c["N"], D=c["D"], gamma=gamma))
        res["long_warped"].append(dict(point(x, y, gamma, m, 2, normalized=True), B=c["B"], N=c["N"], D=c["D"],
                                       gamma=gamma, variant="normalized"))
    del x, y

    c = synth.WORKLOADS["barycenter"]
    X = torch.from_numpy(synth.block_waves(c["K"], c["T"], c["D"], c["seed"])).to(dev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    softdtw_barycenter(X, gamma=1.0, max_iter=3, lr=c["lr"], fused=True)          # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    z, lo = softdtw_barycenter(X, gamma=1.0, max_iter=c["steps"], lr=c["lr"], fused=True, return_losses=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    peak = (torch.cuda.max_memory_allocated(dev) - base) / 2**20
    cells = c["steps"] * c["K"] * c["T"] * c["T"]
    r = step_roofline(cells, c["steps"] * 2 * c["K"] * 2 * c["T"] * c["D"] * 4, "fused", False, hbm, rates, ms)
    lo = lo.cpu().numpy()
    _, lo_es = softdtw_barycenter(X, gamma=1.0, max_iter=c["steps"], lr=c["lr"], fused=True, early_stopping=True,
                                  return_losses=True)
    lo_es = lo_es.cpu().numpy()
    res["barycenter"] = {"K": c["K"], "T": c["T"], "D": c["D"], "steps": c["steps"], "lr": c["lr"], "gamma": 1.0,
                         "mode": "fused", "ms": ms, "ms_per_step": ms / c["steps"], "cells": cells,
                         "cells_per_s": cells / (ms * 1e-3), "peak_MB_above_inputs": peak,
                         "roofline_frac": r["frac"], "roofline": r, "loss_first": float(lo[0]),
                         "loss_last": float(lo[-1]),
                         "early_stopping": {"iterations": int(len(lo_es)), "of": c["steps"],
                                            "saved_frac": 1.0 - len(lo_es) / c["steps"],
                                            "loss_last": float(lo_es[-1]),
                                            "rule": "tol=1e-4 relative improvement, patience=10, checked every 10"}}
    res["wall_s"] = time.perf_counter() - t0
    return res


# --------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import torch.distributed as dist
    from differentiable_series_alignment_gb300 import _lib as L, synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    L.load()
    dev = torch.device("cuda", local)
    x_np, y_np = synth.iid_normal_pair(B, N, M, D, 1, repeat=rank)
    x = torch.from_numpy(x_np).to(dev)
    y = torch.from_numpy(y_np).to(dev)
    g = torch.full((B,), 1.0 / B, device=dev)
    bufs = {}
    for mode in (L.UNFUSED, L.FUSED):
        bufs[mode] = dict(ws=L.workspace(L.OP_FWD_BWD, B, N, M, D, mode, dev),
                          loss=torch.empty(B, device=dev), gx=torch.empty_like(x), gy=torch.empty_like(y))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        for mode in (L.UNFUSED, L.FUSED):
            b = bufs[mode]
            L.sdtw_forward(x, y, GAMMA, mode, b["loss"], b["ws"])
            L.sdtw_backward(x, y, GAMMA, mode, g, b["gx"], b["gy"], b["ws"])

    for _ in range(max(args.warmup, 3)):
        step()
    for mode in (L.UNFUSED, L.FUSED):
        assert L.sdtw_last_device_status(bufs[mode]["ws"]) == 0
    # The step's library calls (their launches, memsets and side-stream forks) captured
    # once into a CUDA graph and replayed: the same kernels with the same arguments,
    # without the host round trips and launch gaps between them.
    launch = "eager"
    run_step = step
    if args.graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            graph.replay()
            torch.cuda.synchronize()
            for mode in (L.UNFUSED, L.FUSED):
                assert L.sdtw_last_device_status(bufs[mode]["ws"]) == 0
            run_step, launch = graph.replay, "cuda_graph"
        except Exception as e:  # capture unsupported here: time the calls as issued
            launch = f"eager (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()

    uuid = None
    try:
        u = torch.cuda.get_device_properties(local).uuid
        uuid = "GPU-" + str(u) if not str(u).startswith("GPU-") else str(u)
    except Exception:
        uuid = None
    clk = ClockSampler(uuid)
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk.start()
    t_wall0 = time.perf_counter()
    for k in range(K):
        flush.fill_(k & 0xff)
        starts[k].record(stream)
        run_step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    clocks = clk.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = time_max_over_ranks(float(np.sum(step_ms)), dev)
    for mode in (L.UNFUSED, L.FUSED):
        assert L.sdtw_last_device_status(bufs[mode]["ws"]) == 0
    cells_per_step = 2 * CELLS
    value = job_value(world, K, cells_per_step, total_ms)

    # ---- per mode, per kernel (events on the launching stream), L2 flushed between iterations
    def timed(fn, iters):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for k in range(iters):
            flush.fill_(k & 0xff)
            ev[k][0].record(stream)
            fn()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ev]))

    iters = max(20, min(200, K))
    per_mode = {}
    for mode, name in ((L.UNFUSED, "unfused"), (L.FUSED, "fused")):
        b = bufs[mode]
        f_ms = timed(lambda: L.sdtw_forward(x, y, GAMMA, mode, b["loss"], b["ws"]), iters)
        bw_ms = timed(lambda: L.sdtw_backward(x, y, GAMMA, mode, g, None, None, b["ws"]), iters)
        fb_ms = timed(lambda: (L.sdtw_forward(x, y, GAMMA, mode, b["loss"], b["ws"]),
                               L.sdtw_backward(x, y, GAMMA, mode, g, b["gx"], b["gy"], b["ws"])), iters)
        per_mode[name] = {"fwd_ms": f_ms, "bwd_wavefront_ms": bw_ms, "fwd_bwd_ms": fb_ms,
                          "cells_per_s": CELLS / (fb_ms * 1e-3)}
        assert L.sdtw_last_device_status(b["ws"]) == 0

    # the double-float state (SDTW_EXTENDED: robust to near ties at any upstream weight)
    # at the same workload, both modes
    for mode, name in ((L.UNFUSED | L.EXTENDED, "unfused+extended"), (L.FUSED | L.EXTENDED, "fused+extended")):
        bx = {"ws": L.workspace(L.OP_FWD_BWD, B, N, M, D, mode, dev), "loss": torch.empty(B, device=dev),
              "gx": torch.empty_like(x), "gy": torch.empty_like(y)}
        xi = max(10, min(50, K))
        f_ms = timed(lambda: L.sdtw_forward(x, y, GAMMA, mode, bx["loss"], bx["ws"]), xi)
        fb_ms = timed(lambda: (L.sdtw_forward(x, y, GAMMA, mode, bx["loss"], bx["ws"]),
                               L.sdtw_backward(x, y, GAMMA, mode, g, bx["gx"], bx["gy"], bx["ws"])), xi)
        per_mode[name] = {"fwd_ms": f_ms, "fwd_bwd_ms": fb_ms, "cells_per_s": CELLS / (fb_ms * 1e-3),
                          "workspace_MB": bx["ws"].numel() / 2**20}
        assert L.sdtw_last_device_status(bx["ws"]) == 0
        del bx

    # the checkpointed fused mode (no per-cell forward state; bands recomputed in the
    # backward): reported beside the two modes of the step, not part of it
    ck = L.FUSED | L.CHECKPOINT
    bufs[ck] = {"ws": L.workspace(L.OP_FWD_BWD, B, N, M, D, ck, dev), "loss": torch.empty(B, device=dev),
                "gx": torch.empty_like(x), "gy": torch.empty_like(y)}
    b = bufs[ck]
    ck_iters = max(10, min(50, K))
    f_ms = timed(lambda: L.sdtw_forward(x, y, GAMMA, ck, b["loss"], b["ws"]), ck_iters)
    fb_ms = timed(lambda: (L.sdtw_forward(x, y, GAMMA, ck, b["loss"], b["ws"]),
                           L.sdtw_backward(x, y, GAMMA, ck, g, b["gx"], b["gy"], b["ws"])), ck_iters)
    per_mode["fused_checkpoint"] = {"fwd_ms": f_ms, "fwd_bwd_ms": fb_ms, "cells_per_s": CELLS / (fb_ms * 1e-3)}
    assert L.sdtw_last_device_status(b["ws"]) == 0

    # peak memory of one fwd+bwd per mode, inputs and gradient buffers resident
    for mode, name in ((L.UNFUSED, "unfused"), (L.FUSED, "fused"), (ck, "fused_checkpoint")):
        del bufs[mode]
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        gx_, gy_ = torch.empty_like(x), torch.empty_like(y)
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        ws = L.workspace(L.OP_FWD_BWD, B, N, M, D, mode, dev)
        loss = torch.empty(B, device=dev)
        L.sdtw_forward(x, y, GAMMA, mode, loss, ws)
        L.sdtw_backward(x, y, GAMMA, mode, g, gx_, gy_, ws)
        torch.cuda.synchronize()
        per_mode[name]["peak_MB"] = torch.cuda.max_memory_allocated(dev) / 2**20
        per_mode[name]["peak_MB_above_inputs"] = (torch.cuda.max_memory_allocated(dev) - base) / 2**20
        per_mode[name]["workspace_MB"] = ws.numel() / 2**20
        del ws, loss, gx_, gy_

    # ---- roofline of the dominant kernel: the backward wavefront (the largest share of a
    # step's kernel time in the launch list), timed alone through sdtw_backward without input
    # gradients (fused workspace). Its roofline is the slower of two bounds per launch:
    # HBM at the method's bytes for the fused backward (R read once, 4 B per cell; E stays
    # on chip) and the SFU at the method's 3 ex2 + 1 lg2 per cell.
    hbm, src = measured_peaks()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rates = sfu_rates(num_sms)
    bw_ms = per_mode["fused"]["bwd_wavefront_ms"]
    bytes_bwd = CELLS * 4
    rb = roofline_bound(CELLS, bytes_bwd, BWD_EX2, BWD_LG2, hbm, rates)
    if rb["bound"] == "hbm":
        achieved, peak, unit = bytes_bwd / (bw_ms * 1e-3) / 1e9, hbm, "GB/s"
    else:
        achieved = CELLS * (BWD_EX2 + BWD_LG2) / (bw_ms * 1e-3) / 1e12
        peak = CELLS * (BWD_EX2 + BWD_LG2) / (rb["sfu_us"] * 1e-6) / 1e12
        unit = "Tops/s (ex2 + lg2)"
    sha = sources_sha256(BWD_SOURCES)
    traffic = BWD_TRAFFIC["bytes"] if BWD_TRAFFIC["sha256"] == sha else None
    impl_bytes = CELLS * (8 + 4)   # what this kernel moves: the stored (v_left, h_up) pair, E written
    roofline = {"bound": rb["bound"], "achieved": achieved, "peak": peak, "unit": unit,
                "frac": rb["bound_us"] / (bw_ms * 1e3), "traffic": traffic,
                "kernel": "bwd_kernel (log-space backward wavefront, fused step)",
                "peak_source": f"HBM {src} ({hbm:.0f} GB/s); SFU ex2 {rates[0]:.3g}/s, lg2 {rates[1]:.3g}/s "
                               f"({EX2_PER_SM_CLK} and {LG2_PER_SM_CLK} per SM and clock at "
                               f"{sm_clock_mhz():.0f} MHz x {num_sms} SMs)",
                "algorithmic_bytes_per_launch": bytes_bwd, "sfu_ops_per_cell": {"ex2": BWD_EX2, "lg2": BWD_LG2},
                "hbm_us": rb["hbm_us"], "sfu_us": rb["sfu_us"], "launch_ms": bw_ms,
                "implementation_bytes_per_launch": impl_bytes,
                "traffic_over_algorithmic": (traffic / bytes_bwd) if traffic else None,
                "traffic_sources_sha256": sha}

    # ---- the same kernel against its latency floor. One 32-row strip over a long row
    # has no neighbour to wait for, so its time per step is the free-running step of
    # the backward recursion; a pass over one N x M problem takes at least N+M-1 of
    # them. Timed through the library like the rest (one warp, fused workspace).
    Lc = 8192
    x1_np, y1_np = synth.iid_normal_pair(1, 32, Lc, D, 5)
    x1, y1 = torch.from_numpy(x1_np).to(dev), torch.from_numpy(y1_np).to(dev)
    ws1 = L.workspace(L.OP_FWD_BWD, 1, 32, Lc, D, L.FUSED, dev)
    loss1, g1 = torch.empty(1, device=dev), torch.ones(1, device=dev)
    L.sdtw_forward(x1, y1, GAMMA, L.FUSED, loss1, ws1)
    strip_ms = timed(lambda: L.sdtw_backward(x1, y1, GAMMA, L.FUSED, g1, None, None, ws1), 20)
    assert L.sdtw_last_device_status(ws1) == 0
    steps1 = ((Lc + 31 + 15) // 16) * 16          # skewed steps of one strip
    step_ns = strip_ms * 1e6 / steps1
    floor_ms = (N + M - 1) * step_ns * 1e-6
    roofline["latency"] = {"chain_steps": N + M - 1, "free_step_ns": step_ns, "floor_ms": floor_ms,
                           "frac": floor_ms / bw_ms,
                           "note": "free-running step measured on one 32 x 8192 strip (whole launch / its "
                                   "8224 steps); frac = floor_ms / launch_ms"}
    del ws1

    # the whole step per mode against the same two bounds (both directions, inputs and
    # gradients moved once)
    io = 2 * B * (N + M) * D * 4
    for name in ("unfused", "fused"):
        per_mode[name]["roofline"] = step_roofline(CELLS, io, name, False, hbm, rates, per_mode[name]["fwd_bwd_ms"])
        per_mode[name]["latency_floor_ms"] = 2 * floor_ms

    per_config = None
    if args.per_config:
        per_config = measure_per_config(L, synth, dev, flush, stream, hbm, rates, step_ns)

    # ---- end to end through the C ABI with HOST buffers, both modes: every step copies the
    # batch in from pinned host memory and the losses and gradients back out
    # (sdtw_value_and_grad_host: the batch runs as E2E_CHUNKS chunks on side streams, so the
    # copies of one chunk overlap the kernels of the others)
    xh = torch.from_numpy(x_np).pin_memory()
    yh = torch.from_numpy(y_np).pin_memory()
    glh = torch.full((B,), 1.0 / B).pin_memory()
    hbuf = {m_: (torch.empty(B).pin_memory(), torch.empty_like(xh).pin_memory(), torch.empty_like(yh).pin_memory(),
                 L.host_workspace(B, N, M, D, m_, E2E_CHUNKS, device=dev))
            for m_ in (L.UNFUSED, L.FUSED)}

    def e2e_step():
        for mode in (L.UNFUSED, L.FUSED):
            lo, gxo, gyo, wsh = hbuf[mode]
            L.sdtw_value_and_grad_host(xh, yh, glh, GAMMA, mode, lo, gxo, gyo, E2E_CHUNKS, wsh, stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    ke = max(10, min(100, K))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(ke):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / ke
    for mode in (L.UNFUSED, L.FUSED):
        assert L.sdtw_last_device_status(hbuf[mode][3], stream) == 0
    h2d = 2 * (xh.numel() + yh.numel() + B) * 4
    d2h = 2 * (B + xh.numel() + yh.numel()) * 4

    if rank != 0:
        return 0
    cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": "cells/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "N": N, "M": M, "D": D, "gamma": GAMMA,
                   "cells_per_step": cells_per_step, "l2": "flushed between timed steps (256 MiB write)",
                   "launch": launch},
        "per_mode": per_mode,
        "roofline": roofline,
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": {"value": world * 2 * CELLS / (e2e_ms * 1e-3), "unit": "cells/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": K * LAUNCHES_PER_STEP,
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(args):
    """K untimed steps of the workload (unfused, then fused), for wrapping in ncu; in
    the fp32 modes of the timed step or in the extended ones."""
    import torch
    from differentiable_series_alignment_gb300 import _lib as L, synth
    L.load()
    x_np, y_np = synth.iid_normal_pair(B, N, M, D, 1)
    x, y = torch.from_numpy(x_np).cuda(), torch.from_numpy(y_np).cuda()
    g = torch.full((B,), 1.0 / B, device="cuda")
    prec = L.EXTENDED if args.profile_precision == "extended" else 0
    for mode in (L.UNFUSED | prec, L.FUSED | prec):
        ws = L.workspace(L.OP_FWD_BWD, B, N, M, D, mode)
        loss, gx, gy = torch.empty(B, device="cuda"), torch.empty_like(x), torch.empty_like(y)
        for _ in range(args.profile):
            L.sdtw_forward(x, y, GAMMA, mode, loss, ws)
            L.sdtw_backward(x, y, GAMMA, mode, g, gx, gy, ws)
        assert L.sdtw_last_device_status(ws) == 0
    torch.cuda.synchronize()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--profile", type=int, default=0, help="run this many untimed steps (for ncu) and exit")
    ap.add_argument("--profile-precision", choices=("fp32", "extended"), default="fp32",
                    help="precision of the --profile steps")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time the step's library calls as issued instead of replaying them as a CUDA graph")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the throughput / peak-memory / roofline figures of the other workloads")
    args = ap.parse_args()
    if args.profile:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
