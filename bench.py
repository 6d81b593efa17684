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
# DRAM bytes (read + write) of one bwd_kernel launch at this workload, from one
# `ncu --set full` capture of it: 71.55 MB read + 8.00 MB written. Set to None
# whenever the kernel changes until it is captured again.
BWD_DRAM_BYTES = 76.41e6
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
        step()
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

    # ---- roofline of the dominant kernel: the backward wavefront (38% of the kernel time of a step in
    # the launch list), timed alone through sdtw_backward without input gradients (fused workspace)
    hbm, src = measured_peaks()
    bw_ms = per_mode["fused"]["bwd_wavefront_ms"]
    slots = B * ((N + 31) // 32) * (M + 31) * 32
    bytes_bwd = CELLS * (8 + 4)  # (v_left, h_up) pair read + E written, per cell
    achieved = bytes_bwd / (bw_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": BWD_DRAM_BYTES, "kernel": "bwd_kernel (log-space backward wavefront)",
                "peak_source": src, "algorithmic_bytes_per_launch": bytes_bwd, "skewed_slots": slots,
                "launch_ms": bw_ms,
                "note": "latency-bound: N+M-1 dependent DP steps; traffic from one ncu capture of this kernel"}

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
                   "cells_per_step": cells_per_step, "l2": "flushed between timed steps (256 MiB write)"},
        "per_mode": per_mode,
        "roofline": roofline,
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
    """K untimed steps of the workload (both modes), for wrapping in ncu."""
    import torch
    from differentiable_series_alignment_gb300 import _lib as L, synth
    L.load()
    x_np, y_np = synth.iid_normal_pair(B, N, M, D, 1)
    x, y = torch.from_numpy(x_np).cuda(), torch.from_numpy(y_np).cuda()
    g = torch.full((B,), 1.0 / B, device="cuda")
    for mode in (L.UNFUSED, L.FUSED):
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
    args = ap.parse_args()
    if args.profile:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
