#!/usr/bin/env python3
"""Benchmark of the GB300 Gated DeltaNet layer (one JSON line on rank 0).

Step = one decode step of the layer for 256 sequences x 1 token (16 QK / 32 V
heads, head_dim 128, bf16 activations, fp32 state pool of 1024 slots):
causal_conv1d_update over the 8192-channel qkv stream -> gdn_gating ->
gdn_decode_recurrent reading q/k/v straight out of the conv output.  value =
decode tokens/s of the whole job; the decode kernel's state traffic is the
roofline line (HBM bound).  Extra keys report the chunked prefill (8
sequences, 512..8192 tokens: conv fwd -> gating -> prefill) and the MTP step
(128 x 4 tokens with per-token snapshots and an accept copy).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run, one independent replica per GPU
(weak scaling: sequences are independent, the path has no collective); the
process group only carries the barrier and the max-over-ranks time.
--impl reference times the CPU oracle (the only reference implementation
there is) on a bounded sample of the same workload, on rank 0.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode tokens/s + state HBM GB/s; chunked prefill tokens/s; % roofline"
UNIT = "tokens/s"
DECODE_WORKLOAD = ("decode step: 256 sequences x 1 token, causal conv update (8192 ch, width 4) "
                   "+ gating + q/k L2 norm + recurrent decode (gdn_decode_step_fused with its "
                   "workspace: the conv / gates kernel, then the streaming decode behind it by "
                   "programmatic dependent launch), 16 QK / 32 V heads, head_dim 128, "
                   "bf16 activations, fp32 state pool 1024 slots x 32 x 128 x 128")


# --------------------------------------------------------------------- util --

def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true", help="skip the prefill / MTP extras")
    p.add_argument("--only", choices=["mtp", "prefill", "long"], default=None,
                   help="profiling aid: run just this extra (its own JSON line, no decode step)")
    p.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    p.add_argument("--long-tokens", type=int, default=65536,
                   help="length of the long-context sequence (profiling aid with --only long)")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend, init_method="env://")


def reduce_max(x: float, device) -> float:
    """Max of x over ranks (x itself without a process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def whole_job(units_per_rank: float, max_seconds: float, world: int) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


SPLIT_SOURCES = ["gated_deltanet_linear_10_gb300/csrc/" + f for f in
                 ("prefill_split.cu", "prefill_common.cuh", "tc.cuh", "common.cuh")]


def profile_traffic(kernel_key: str, source_files):
    """DRAM bytes per launch recorded from an ncu capture in profiles/traffic.txt
    (lines: key bytes sha256-of-sources), or None when the kernel's sources
    changed since the capture or there is none."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in source_files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kernel_key and parts[2] == digest:
                return float(parts[1])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[c.strip() for c in line.split(",")] for line in out.strip().splitlines()]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s in sm if s >= 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- our kernels --

def decode_step_bytes(n, hqk, hv, channels, width=4):
    """Algorithmic bytes of the fused decode step (bf16 activations, dk = dv
    = 128): the state read + written once, the conv state read + written,
    x, a, b, o, the conv weights once, A_log / dt_bias, slot ids."""
    state = 2 * n * hv * 128 * 128 * 4
    conv_state = 2 * n * (width - 1) * channels * 2
    x = n * channels * 2
    ab = 2 * n * hv * 2
    o = n * hv * 128 * 2
    return state + conv_state + x + ab + o + channels * width * 2 + 2 * hv * 4 + n * 4


def decode_kernel_bytes(n, hqk, hv, dk, dv, io_bytes):
    """Algorithmic bytes of one decode launch (1 token per sequence): the
    state read + written once, q/k per QK head, v, o, g, beta, slot ids."""
    state = 2 * n * hv * dv * dk * 4
    qk = 2 * n * hqk * dk * io_bytes
    vo = 2 * n * hv * dv * io_bytes
    gb = 2 * n * hv * 4
    return state + qk + vo + gb + n * 4


def run_only(args):
    """One extra workload alone (for profiler captures of its kernels)."""
    import gated_deltanet_linear_10_gb300 as gdn
    import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    if args.only == "mtp":
        res = bench_mtp(gdn, workloads, dev, flush, steps=max(1, args.steps))
    elif args.only == "long":
        res = bench_long(gdn, workloads, dev, flush, load_peaks(), steps=max(1, args.steps),
                         T=args.long_tokens)
    else:
        res = bench_prefill(gdn, workloads, dev, flush, load_peaks(), steps=max(1, args.steps))
    assert gdn.gdn_get_device_status(clear=True) == 0
    print(json.dumps({"only": args.only, **res}), flush=True)


def run_ours(args):
    import gated_deltanet_linear_10_gb300 as gdn
    import workloads

    if args.only:
        return run_only(args)
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    peaks = load_peaks()

    w = workloads.decode(pool_device=dev)
    d = w.dims
    x, a, b = w.x.to(dev), w.a.to(dev), w.b.to(dev)
    conv_w, A_log, dt_bias = w.conv_w.to(dev), w.A_log.to(dev), w.dt_bias.to(dev)
    cpool, spool, slots = w.conv_pool.to(dev), w.state_pool, w.slots.to(dev)
    N = w.n_seqs
    y = torch.empty_like(x)
    g = torch.empty((N, d.hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    o = torch.empty((N, d.hv, d.dv), dtype=x.dtype, device=dev)
    nq = d.hqk * d.dk
    qv = y.narrow(1, 0, nq).unflatten(1, (d.hqk, d.dk))
    kv = y.narrow(1, nq, nq).unflatten(1, (d.hqk, d.dk))
    vv = y.narrow(1, 2 * nq, d.hv * d.dv).unflatten(1, (d.hv, d.dv))
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # 256 MiB > L2

    stream = torch.cuda.current_stream(dev)

    ws = torch.empty(gdn.gdn_decode_step_workspace_size(N, d.hqk, d.hv), dtype=torch.uint8,
                     device=dev)

    def step(ev=None, workspace=ws):   # the decode step (two launches with the workspace)
        if ev is not None:
            ev[0].record(stream)
        gdn.gdn_decode_step_fused(x, conv_w, cpool, a, b, A_log, dt_bias, d.hqk, spool, slots,
                                  scale=w.scale, o=o, workspace=workspace)
        if ev is not None:
            ev[1].record(stream)

    def step_unfused(ev=None):   # the same step as three calls
        if ev is not None:
            ev[0].record(stream)
        gdn.causal_conv1d_update(x, 1, conv_w, cpool, slots, y=y)
        if ev is not None:
            ev[1].record(stream)
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
        if ev is not None:
            ev[2].record(stream)
        gdn.gdn_decode_recurrent(qv, kv, vv, g, beta, 1, spool, slots, scale=w.scale, o=o)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
        flush.zero_()
    torch.cuda.synchronize(dev)
    assert gdn.gdn_get_device_status(clear=True) == 0

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    gc.disable()                                 # no collector pause while the host enqueues
    t0 = time.perf_counter()
    torch.cuda._sleep(2_000_000)                 # head start: the host enqueues ahead of the GPU
    for i in range(K):
        step(evs[i])
        flush.zero_()
    torch.cuda.synchronize(dev)
    barrier()
    wall = time.perf_counter() - t0
    gc.enable()
    clocks = sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms_step = sum(step_ms) / K
    ms_step_median = sorted(step_ms)[K // 2]
    ms_step_max = reduce_max(ms_step, dev)
    value = whole_job(N, ms_step_max / 1e3, world)
    # the roofline unit is the whole step (both kernels, the fused step's
    # algorithmic bytes: the y / gates round trip through the workspace is
    # not counted)
    dec_avg = ms_step
    dec_bytes = decode_step_bytes(N, d.hqk, d.hv, d.channels)
    achieved = dec_bytes / (dec_avg / 1e3) / 1e9
    traffic = profile_traffic("decode_step_two_kernels",
                              ["gated_deltanet_linear_10_gb300/csrc/" + f for f in
                               ("decode_step.cu", "decode.cu", "common.cuh", "tc.cuh")])

    # ---- the same step without a workspace: one kernel
    Ko = min(K, 300)
    evo = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ko)]
    for _ in range(3):
        step(workspace=False)
        flush.zero_()
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(2_000_000)
    for i in range(Ko):
        step(evo[i], workspace=False)
        flush.zero_()
    torch.cuda.synchronize(dev)
    one_ms = sum(e[0].elapsed_time(e[1]) for e in evo) / Ko
    one_kernel = {"ms_per_step": round(one_ms, 5),
                  "frac_hbm": round(dec_bytes / (one_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                  "traffic": profile_traffic("decode_step_kernel",
                                             ["gated_deltanet_linear_10_gb300/csrc/" + f for f in
                                              ("decode_step.cu", "common.cuh", "tc.cuh")])}

    # ---- the same step as three calls (conv update, gating, decode)
    Ku = min(K, 200)
    evu = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Ku)]
    for _ in range(3):
        step_unfused()
        flush.zero_()
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(2_000_000)
    for i in range(Ku):
        step_unfused(evu[i])
        flush.zero_()
    torch.cuda.synchronize(dev)
    unf_dec = sum(e[2].elapsed_time(e[3]) for e in evu) / Ku
    unfused = {"ms_per_step": round(sum(e[0].elapsed_time(e[3]) for e in evu) / Ku, 5),
               "causal_conv1d_update_ms": round(sum(e[0].elapsed_time(e[1]) for e in evu) / Ku, 5),
               "gdn_gating_ms": round(sum(e[1].elapsed_time(e[2]) for e in evu) / Ku, 5),
               "gdn_decode_recurrent_ms": round(unf_dec, 5),
               "decode_kernel_frac_hbm": round(
                   decode_kernel_bytes(N, d.hqk, d.hv, d.dk, d.dv, 2) / (unf_dec / 1e3) / 1e9 /
                   peaks["hbm_gbs"], 4)}

    # ---- end to end: host -> device inputs, the three calls, o -> host
    x_h = w.x.pin_memory()
    a_h, b_h = w.a.pin_memory(), w.b.pin_memory()
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    Ke = max(10, min(K, 500))
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(2_000_000)
    for i in range(Ke):
        e2e_ev[i][0].record(stream)
        x.copy_(x_h, non_blocking=True)
        a.copy_(a_h, non_blocking=True)
        b.copy_(b_h, non_blocking=True)
        step()
        o_h.copy_(o, non_blocking=True)
        e2e_ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize(dev)
    e2e_serial_ms = reduce_max(sum(e[0].elapsed_time(e[1]) for e in e2e_ev) / Ke, dev)
    h2d = x_h.numel() * 2 + a_h.numel() * 2 + b_h.numel() * 2
    d2h = o_h.numel() * 2
    assert gdn.gdn_get_device_status(clear=True) == 0

    # ---- end to end as a serving loop runs it: a copy stream brings step
    # i + 1's inputs into the other of two device buffers and reads step
    # i - 1's o back while step i runs; every step's copies are inside the
    # timed loop.  No L2 flush: each step streams 1.1 GB of state (> L2).
    e2e_ms = e2e_pipelined(gdn, w, d, conv_w, A_log, dt_bias, cpool, spool, slots, dev, Ke)

    extras = {}
    if not args.no_extras:
        extras["mtp"] = bench_mtp(gdn, workloads, dev, flush)
        extras["prefill"] = bench_prefill(gdn, workloads, dev, flush, peaks)
        extras["decode_gated"] = bench_decode_gated(gdn, workloads, dev, flush)
        extras["mixed"] = bench_mixed(gdn, workloads, dev, flush)
        extras["long"] = bench_long(gdn, workloads, dev, flush, peaks)

    cpu = None
    if rank == 0:
        del flush
        cpu = cpu_baseline(w, args.cpu_budget)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "global_batch": N * world, "seq_len": 1,
                   "io_dtype": "bf16", "l2": "flushed between steps (256 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": "decode_front_kernel + decode_stream_kernel (one step)",
                     "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "algorithmic_bytes": dec_bytes, "avg_launch_ms": round(dec_avg, 5),
                     "peak_source": peaks["source"]},
        "kernels_ms": {"gdn_decode_step_fused": round(dec_avg, 5)},
        "median_ms_per_step": round(ms_step_median, 5),
        "state_gbs": round(achieved, 1),
        "step_one_kernel": one_kernel,
        "step_unfused": unfused,
        "e2e": {"value": round(whole_job(N, e2e_ms / 1e3, world), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "overlap": "H2D of step i+1 and D2H of step i-1 on a copy stream during step i "
                           "(double-buffered inputs / outputs); L2 not flushed (1.1 GB of state "
                           "per step)",
                "serial_ms_per_step": round(e2e_serial_ms, 5),
                "serial_value": round(whole_job(N, e2e_serial_ms / 1e3, world), 1)},
        "gpu_launches": 2 * K,
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
        "cpu_baseline": cpu,
    }
    line.update(extras)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def e2e_pipelined(gdn, w, d, conv_w, A_log, dt_bias, cpool, spool, slots, dev, steps):
    """ms per decode step of a loop that copies each step's x, a, b from pinned
    host memory and reads its o back, with the copies of neighbouring steps
    overlapping the step on a second stream.  Returns the max over ranks."""
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    n = w.n_seqs
    xs_h = [w.x.clone().pin_memory() for _ in range(2)]
    as_h = [w.a.clone().pin_memory() for _ in range(2)]
    bs_h = [w.b.clone().pin_memory() for _ in range(2)]
    os_h = [torch.empty((n, d.hv, d.dv), dtype=w.x.dtype).pin_memory() for _ in range(2)]
    xs = [torch.empty_like(w.x, device=dev) for _ in range(2)]
    as_ = [torch.empty_like(w.a, device=dev) for _ in range(2)]
    bs = [torch.empty_like(w.b, device=dev) for _ in range(2)]
    os_ = [torch.empty((n, d.hv, d.dv), dtype=w.x.dtype, device=dev) for _ in range(2)]
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    ws = torch.empty(gdn.gdn_decode_step_workspace_size(n, d.hqk, d.hv), dtype=torch.uint8,
                     device=dev)

    def h2d(i):                 # on the copy stream, once buffer i % 2 is consumed
        j = i & 1
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(step_done[j])
            xs[j].copy_(xs_h[j], non_blocking=True)
            as_[j].copy_(as_h[j], non_blocking=True)
            bs[j].copy_(bs_h[j], non_blocking=True)
            h2d_done[j].record(copy)

    def run(k, start=None):
        # copy-stream order: H2D(0), H2D(1), D2H(0), H2D(2), D2H(1), ...: the
        # inputs of step i + 1 and the output of step i - 1 move during step i
        if start is not None:
            copy.wait_event(start)             # the first copy is inside the timed region
        h2d(0)
        for i in range(k):
            j = i & 1
            if i + 1 < k:
                h2d(i + 1)
            comp.wait_event(h2d_done[j])
            if i >= 2:
                comp.wait_event(d2h_done[j])    # o buffer j of step i - 2 is read back
            gdn.gdn_decode_step_fused(xs[j], conv_w, cpool, as_[j], bs[j], A_log, dt_bias, d.hqk,
                                      spool, slots, scale=w.scale, o=os_[j], workspace=ws)
            step_done[j].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(step_done[j])
                os_h[j].copy_(os_[j], non_blocking=True)
                d2h_done[j].record(copy)
        comp.wait_stream(copy)

    run(4)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(2_000_000)
    e0.record(comp)
    run(steps, e0)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    return reduce_max(e0.elapsed_time(e1) / steps, dev)


def bench_mtp(gdn, workloads, dev, flush, steps=50):
    """MTP step: conv update (4 tokens, per-token conv snapshots), gating and
    the decode with per-token state snapshots in one kernel
    (gdn_mtp_step_fused), then the accept copies into the source slots.  The
    same step through the three separate calls is timed beside it."""
    w = workloads.mtp(pool_device=dev)
    d = w.dims
    x, a, b = w.x.to(dev), w.a.to(dev), w.b.to(dev)
    conv_w, A_log, dt_bias = w.conv_w.to(dev), w.A_log.to(dev), w.dt_bias.to(dev)
    cpool, spool, slots, snap = w.conv_pool.to(dev), w.state_pool, w.slots.to(dev), w.snap.to(dev)
    acc_src = w.snap[torch.arange(w.n_seqs), w.extra["accept"].long()].to(torch.int32).to(dev)
    y = torch.empty_like(x)
    nq = d.hqk * d.dk
    qv = y.narrow(1, 0, nq).unflatten(1, (d.hqk, d.dk))
    kv = y.narrow(1, nq, nq).unflatten(1, (d.hqk, d.dk))
    vv = y.narrow(1, 2 * nq, d.hv * d.dv).unflatten(1, (d.hv, d.dv))
    T = w.n_seqs * 4
    g = torch.empty((T, d.hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    o = torch.empty((T, d.hv, d.dv), dtype=x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def accept():
        gdn.gdn_state_snapshot(spool, acc_src, slots)
        gdn.gdn_state_snapshot(cpool, acc_src, slots)

    def fused(e):
        gdn.gdn_mtp_step_fused(x, 4, conv_w, cpool, a, b, A_log, dt_bias, d.hqk, spool, slots,
                               snap, scale=w.scale, o=o)
        e[1].record(stream)
        e[2].record(stream)
        accept()

    def three_calls(e):
        gdn.causal_conv1d_update(x, 4, conv_w, cpool, slots, snap_indices=snap, y=y)
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
        e[1].record(stream)
        gdn.gdn_decode_recurrent(qv, kv, vv, g, beta, 4, spool, slots, snap_indices=snap,
                                 scale=w.scale, o=o)
        e[2].record(stream)
        accept()

    def timed(body):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(3):
            body(ev[i % steps])
            flush.zero_()
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(1_000_000)
        for e in ev:
            e[0].record(stream)
            body(e)
            e[3].record(stream)
            flush.zero_()
        torch.cuda.synchronize(dev)
        mean = lambda u, v: sum(e[u].elapsed_time(e[v]) for e in ev) / steps
        return mean(0, 3), mean(0, 1), mean(1, 2), mean(2, 3)

    f_whole, f_kernel, _, f_accept = timed(fused)
    c_whole, c_front, c_dec, c_accept = timed(three_calls)

    # algorithmic bytes.  state: the source read once, 4 snapshots written;
    # conv state: the same for the slot's 3 x channels bf16 conv state
    st = w.n_seqs * d.hv * d.dv * d.dk * 4
    conv_state = d.channels * 3 * 2
    ab = 2 * T * d.hv * 2
    o_bytes = T * d.hv * d.dv * 2
    # the fused kernel: x, conv weights, a, b read; both states; o written
    fused_bytes = (st * 5 + w.n_seqs * conv_state * 5 + T * d.channels * 2
                   + d.channels * 4 * 2 + ab + o_bytes)
    accept_bytes = 2 * w.n_seqs * (d.hv * d.dv * d.dk * 4 + conv_state)
    step_bytes = fused_bytes + accept_bytes
    # the three calls: conv update (x read, y written, conv states), gating
    # (a, b read, g, beta written), decode (q, k, v, g, beta read, o written)
    io = T * (2 * d.hqk * d.dk + d.hv * d.dv) * 2 + o_bytes + 2 * T * d.hv * 4
    dec_bytes = st * 5 + io
    peak = load_peaks()["hbm_gbs"]
    gbs = lambda nbytes, ms: nbytes / (ms / 1e3) / 1e9
    del spool, w
    return {"workload": "MTP: 128 sequences x 4 tokens, per-token state + conv snapshots, "
                        "accept copy",
            "step_ms": round(f_whole, 5),
            "tokens_per_s": round(T / (f_whole / 1e3), 1),
            "step_bytes": step_bytes,
            "step_gbs": round(gbs(step_bytes, f_whole), 1),
            "step_frac_hbm": round(gbs(step_bytes, f_whole) / peak, 4),
            "gpu_launches_per_step": 3,
            "fused_kernel_ms": round(f_kernel, 5),
            "fused_kernel_algorithmic_bytes": fused_bytes,
            "fused_kernel_gbs": round(gbs(fused_bytes, f_kernel), 1),
            "fused_kernel_frac_hbm": round(gbs(fused_bytes, f_kernel) / peak, 4),
            "fused_kernel_traffic_bytes": profile_traffic(
                "mtp_step_kernel", ["gated_deltanet_linear_10_gb300/csrc/" + f for f in
                                    ("mtp_step.cu", "common.cuh")]),
            "accept_copies_ms": round(f_accept, 5),
            "three_calls": {
                "step_ms": round(c_whole, 5),
                "tokens_per_s": round(T / (c_whole / 1e3), 1),
                "gpu_launches_per_step": 5,
                "conv_update_gating_ms": round(c_front, 5),
                "decode_kernel_ms": round(c_dec, 5),
                "decode_kernel_gbs": round(gbs(dec_bytes, c_dec), 1),
                "decode_kernel_frac_hbm": round(gbs(dec_bytes, c_dec) / peak, 4),
                "decode_kernel_algorithmic_bytes": dec_bytes,
                "decode_kernel_traffic_bytes": profile_traffic(
                    "decode_kernel_mtp", ["gated_deltanet_linear_10_gb300/csrc/" + f for f in
                                          ("decode.cu", "common.cuh", "tc.cuh")]),
                "accept_copies_ms": round(c_accept, 5)}}


def bench_mixed(gdn, workloads, dev, flush, steps=20):
    """A serving step's mixed batch (256 decode rows + two 2048-token prompts)
    through gdn_mixed_batch (decode rows on the streaming decode kernel, in
    place, beside the prompts' chunked prefill), the same call with the two
    halves one after the other, and the same batch through one
    gdn_prefill_chunked call."""
    w = workloads.mixed(pool_device=dev)
    d = w.dims
    q, k, v, a, b = (t.to(dev) for t in (w.q, w.k, w.v, w.a, w.b))
    cu = w.cu_seqlens.to(dev)
    nd = w.extra["n_decode"]
    g, beta = gdn.gdn_gating(a, b, w.A_log.to(dev), w.dt_bias.to(dev))
    slots = w.slots.to(dev)
    # decode rows continue their slot in place; prompts start from zero and
    # end in their slot
    init = torch.where(w.has_initial_state.to(dev).bool(), slots, torch.full_like(slots, -1))
    T = q.shape[0]
    o = torch.empty((T, d.hv, d.dv), dtype=q.dtype, device=dev)
    need = gdn.gdn_prefill_workspace_size(w.n_seqs - nd, T, d.hv, d.dk, d.dv, 64)
    # + 512 bytes: the decode runs beside the prefill's chains; without them
    # the two halves run one after the other
    ws_mixed = torch.empty(need + 512, dtype=torch.uint8, device=dev)
    ws_serial = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_all = torch.empty(gdn.gdn_prefill_workspace_size(w.n_seqs, T, d.hv, d.dk, d.dv, 64),
                         dtype=torch.uint8, device=dev)
    def mixed():
        gdn.gdn_mixed_batch(q, k, v, g, beta, cu, nd, w.state_pool, init, slots, w.scale,
                            decode_in_place=True, o=o, workspace=ws_mixed)

    def serial():
        gdn.gdn_mixed_batch(q, k, v, g, beta, cu, nd, w.state_pool, init, slots, w.scale,
                            decode_in_place=True, o=o, workspace=ws_serial)

    def one_call():
        gdn.gdn_prefill_chunked(q, k, v, g, beta, cu, w.state_pool, init, slots, w.scale, o=o,
                                workspace=ws_all)

    res = {}
    for name, fn in (("mixed_batch", mixed), ("serial", serial), ("prefill_call", one_call)):
        for _ in range(3):
            fn()
            flush.zero_()
        torch.cuda.synchronize(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record()
            fn()
            ev[i][1].record()
            flush.zero_()
        torch.cuda.synchronize(dev)
        res[name] = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    assert gdn.gdn_get_device_status(clear=True) == 0
    return {"workload": f"mixed step: {nd} decode rows (1 token, state in place) + prompts of "
                        f"{[int(x) for x in w.extra['lengths'][nd:]]} tokens, 16 QK / 32 V heads, "
                        "head_dim 128, bf16",
            "tokens_per_s": round(T / (res["mixed_batch"] / 1e3), 1),
            "mixed_batch_ms": round(res["mixed_batch"], 4),
            "path": "prefill, then the streaming decode beside its chains (work counter)",
            "halves_one_after_the_other_ms": round(res["serial"], 4),
            "prefill_call_ms": round(res["prefill_call"], 4),
            "gpu_launches_per_step": 5}


def bench_decode_gated(gdn, workloads, dev, flush, steps=50):
    """The decode step's recurrence with the gated RMSNorm on its output
    (gdn_decode_recurrent_gated: at dv = 128 decode, then the norm kernel in
    place) against the plain decode, and the norm kernel alone."""
    w = workloads.decode(pool_device=dev)
    d = w.dims
    gen = torch.Generator().manual_seed(2024)
    z = torch.randn(w.q.shape[0], d.hv, d.dv, generator=gen).to(w.q.dtype).to(dev)
    nw = (torch.rand(d.dv, generator=gen) + 0.5).to(dev)
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    g, beta = gdn.gdn_gating(w.a.to(dev), w.b.to(dev), w.A_log.to(dev), w.dt_bias.to(dev))
    spool, slots = w.state_pool, w.slots.to(dev)
    o = torch.empty((q.shape[0], d.hv, d.dv), dtype=q.dtype, device=dev)
    y = torch.empty_like(o)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for _ in range(3):
            fn()
            flush.zero_()
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(1_000_000)
        for i in range(steps):
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
            flush.zero_()
        torch.cuda.synchronize(dev)
        return sum(e[0].elapsed_time(e[1]) for e in ev) / steps

    def plain():
        gdn.gdn_decode_recurrent(q, k, v, g, beta, 1, spool, slots, scale=w.scale, o=o)

    def gated():
        gdn.gdn_decode_recurrent_gated(q, k, v, g, beta, 1, spool, slots, z, nw, 1e-6,
                                       scale=w.scale, y=y)

    def norm():
        gdn.gdn_gated_rmsnorm(o, z, nw, 1e-6, y=y)

    t_plain, t_gated, t_norm = timed(plain), timed(gated), timed(norm)
    nbytes = 3 * o.numel() * o.element_size()       # o and z read, y written
    del spool, w
    return {"workload": "decode 256 x 1 token + gated RMSNorm (dv 128) of its output",
            "gated_decode_ms": round(t_gated, 5), "plain_decode_ms": round(t_plain, 5),
            "norm_kernel_ms": round(t_norm, 5),
            "norm_kernel_gbs": round(nbytes / (t_norm / 1e3) / 1e9, 1),
            "gated_tokens_per_s": round(256 / (t_gated / 1e3), 1)}


def prefill_flops_per_token(hv, dk, dv, chunk, causal=False):
    """Flops of the chunked form per token, full chunk x chunk tiles:
    hv * (6 dk dv + 2 C (3 dk + 2 dv)); with causal, the C x C tiles count
    half: hv * (6 dk dv + C (3 dk + 2 dv))."""
    return hv * (6 * dk * dv + (1 if causal else 2) * chunk * (3 * dk + 2 * dv))


def bench_prefill(gdn, workloads, dev, flush, peaks, steps=5):
    w = workloads.prefill()
    d = w.dims
    x = w.x.to(dev)
    conv_w, A_log, dt_bias = w.conv_w.to(dev), w.A_log.to(dev), w.dt_bias.to(dev)
    a, b = w.a.to(dev), w.b.to(dev)
    cu, slots = w.cu_seqlens.to(dev), w.slots.to(dev)
    has = w.has_initial_state.to(dev)
    cpool = w.conv_pool.to(dev)
    spool = torch.zeros((64, d.hv, d.dv, d.dk), dtype=torch.float32, device=dev)
    sslots = (slots % 64).to(torch.int32)      # final-state slots in the 64-slot pool
    none = torch.full_like(slots, -1)
    T = x.shape[0]
    y = torch.empty_like(x)
    nq = d.hqk * d.dk
    qv = y.narrow(1, 0, nq).unflatten(1, (d.hqk, d.dk))
    kv = y.narrow(1, nq, nq).unflatten(1, (d.hqk, d.dk))
    vv = y.narrow(1, 2 * nq, d.hv * d.dv).unflatten(1, (d.hv, d.dv))
    g = torch.empty((T, d.hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    o = torch.empty((T, d.hv, d.dv), dtype=x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    need = gdn.gdn_prefill_workspace_size(cu.numel() - 1, T, d.hv, d.dk, d.dv, w.chunk)
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else False

    def step(e=None, workspace=ws):
        if e is not None:
            e[0].record(stream)
        gdn.causal_conv1d_fwd(x, conv_w, cu, cpool, slots, has, y=y)
        if e is not None:
            e[1].record(stream)
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
        if e is not None:
            e[2].record(stream)
        gdn.gdn_prefill_chunked(qv, kv, vv, g, beta, cu, spool, none, sslots, w.scale,
                                chunk=w.chunk, o=o, workspace=workspace)
        if e is not None:
            e[3].record(stream)

    # the single fused kernel (no workspace), for comparison
    for _ in range(2):
        step(workspace=False)
        flush.zero_()
    torch.cuda.synchronize(dev)
    for i in range(steps):
        step(ev[i], workspace=False)
        flush.zero_()
    torch.cuda.synchronize(dev)
    pre_fused = sum(e[2].elapsed_time(e[3]) for e in ev) / steps

    def call_ms(fn):
        """Mean time of one call of fn, L2 flushed between calls."""
        for _ in range(2):
            fn()
            flush.zero_()
        torch.cuda.synchronize(dev)
        for i in range(steps):
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
            flush.zero_()
        torch.cuda.synchronize(dev)
        return sum(e[0].elapsed_time(e[1]) for e in ev) / steps

    # the gated RMSNorm of the prefill output (standalone kernel, in place)
    z = torch.randn(o.shape, generator=torch.Generator().manual_seed(7)).to(o.dtype).to(dev)
    nw = torch.ones(d.dv, device=dev)
    norm_ms = call_ms(lambda: gdn.gdn_gated_rmsnorm(o, z, nw, 1e-6, y=o))
    norm_bytes = 3 * o.numel() * o.element_size()

    # the prefill with the gated RMSNorm in the chain kernel's epilogue (y
    # instead of o), after the layer's conv and gating
    y_gated = torch.empty_like(o)

    def gated():
        gdn.gdn_prefill_chunked_gated(qv, kv, vv, g, beta, cu, spool, none, sslots, w.scale, z,
                                      nw, 1e-6, chunk=w.chunk, y=y_gated, workspace=ws)

    step()
    gated_ms = call_ms(gated)

    # the same layer in one call: gdn_prefill_layer (conv, then the prefill
    # with the gates formed in its prep kernel)
    lneed = gdn.gdn_prefill_layer_workspace_size(cu.numel() - 1, T, d.hqk, d.hv)
    lws_raw = torch.empty(lneed + 1024, dtype=torch.uint8, device=dev)
    loff = (-lws_raw.data_ptr()) % 1024
    lws = lws_raw[loff:loff + lneed]

    layer_call_ms = call_ms(lambda: gdn.gdn_prefill_layer(
        x, conv_w, cpool, slots, has, a, b, A_log, dt_bias, cu, d.hqk, spool, none, sslots,
        scale=w.scale, o=o, workspace=lws))
    # and the gated layer in one call (gdn_prefill_layer_gated: y instead of o)
    gated_layer_call_ms = call_ms(lambda: gdn.gdn_prefill_layer_gated(
        x, conv_w, cpool, slots, has, a, b, A_log, dt_bias, cu, d.hqk, spool, none, sslots, z,
        nw, 1e-6, scale=w.scale, y=y_gated, workspace=lws))

    for _ in range(2):
        step()
        flush.zero_()
    torch.cuda.synchronize(dev)
    for i in range(steps):
        step(ev[i])
        flush.zero_()
    torch.cuda.synchronize(dev)
    total = sum(e[0].elapsed_time(e[3]) for e in ev) / steps
    conv = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    pre = sum(e[2].elapsed_time(e[3]) for e in ev) / steps
    flops = prefill_flops_per_token(d.hv, d.dk, d.dv, w.chunk) * T
    tf = flops / (pre / 1e3) / 1e12
    conv_bytes = 2 * T * d.channels * 2
    return {"workload": f"prefill: 8 sequences, {T} tokens (lengths U[512, 8192]), conv fwd + "
                        "gating + chunked prefill (chunk 64)",
            "tokens_per_s": round(T / (min(total, layer_call_ms) / 1e3), 1),
            "layer_ms": round(total, 4), "prefill_kernel_ms": round(pre, 4),
            "layer_call_ms": round(layer_call_ms, 4),
            "layer_path": "gdn_prefill_layer (conv, then the prefill with its gates formed in "
                          "the prep kernel)" if layer_call_ms < total else
                          "conv fwd + gating + prefill (three calls)",
            "prefill_path": "prep kernel + chain kernel (workspace %.1f MiB)" % (need / 2**20),
            "prefill_fused_kernel_ms": round(pre_fused, 4),
            "conv_kernel_ms": round(conv, 4),
            "conv_gbs": round(conv_bytes / (conv / 1e3) / 1e9, 1),
            "prefill_tflops": round(tf, 2),
            "gated_norm_ms": round(norm_ms, 4),
            "gated_norm_gbs": round(norm_bytes / (norm_ms / 1e3) / 1e9, 1),
            "prefill_gated_kernel_ms": round(gated_ms, 4),
            "gated_layer_ms": round(total - pre + gated_ms, 4),
            "gated_layer_call_ms": round(gated_layer_call_ms, 4),
            "gated_layer_tokens_per_s": round(
                T / (min(total - pre + gated_ms, gated_layer_call_ms) / 1e3), 1),
            "prep_kernel_traffic_bytes": profile_traffic("prep_kernel", SPLIT_SOURCES),
            "chain_kernel_traffic_bytes": profile_traffic("chain_kernel", SPLIT_SOURCES),
            "prefill_frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "flops_per_token": prefill_flops_per_token(d.hv, d.dk, d.dv, w.chunk),
            # the same at the causal-half count of the C x C tiles (4.46 MFLOP/token)
            "prefill_tflops_causal": round(
                prefill_flops_per_token(d.hv, d.dk, d.dv, w.chunk, causal=True) * T
                / (pre / 1e3) / 1e12, 2)}


def bench_long(gdn, workloads, dev, flush, peaks, steps=3, T=65536):
    """Long-context prefill: one sequence of T = 65,536 tokens, 16 QK / 32 V
    heads, head_dim 128, bf16, nonzero initial state (gating + chunked
    prefill), and the split at T / 2 with the state carried through a pool
    slot against the single pass."""
    w = workloads.long_context(device=dev, T=T)
    d = w.dims
    T = w.q.shape[0]
    q, k, v, a, b = w.q, w.k, w.v, w.a, w.b
    A_log, dt_bias = w.A_log.to(dev), w.dt_bias.to(dev)
    pool = torch.zeros((4, d.hv, d.dv, d.dk), dtype=torch.float32, device=dev)
    pool[0] = w.state_pool[0]
    g = torch.empty((T, d.hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    o = torch.empty((T, d.hv, d.dv), dtype=q.dtype, device=dev)
    i32 = lambda *x: torch.tensor(x, dtype=torch.int32, device=dev)
    cu, s0, s1, s2, s3 = i32(0, T), i32(0), i32(1), i32(2), i32(3)
    need = gdn.gdn_prefill_workspace_size(1, T, d.hv, d.dk, d.dv, w.chunk)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(e=None):
        if e is not None:
            e[0].record(stream)
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
        if e is not None:
            e[1].record(stream)
        gdn.gdn_prefill_chunked(q, k, v, g, beta, cu, pool, s0, s1, w.scale, o=o, workspace=ws)
        if e is not None:
            e[2].record(stream)

    for _ in range(2):
        step()
        flush.zero_()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        step(ev[i])
        flush.zero_()
    torch.cuda.synchronize(dev)
    total = sum(e[0].elapsed_time(e[2]) for e in ev) / steps
    pre = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    # the same sequence on the serial chain (a workspace without the scan's part)
    serial_ws = torch.empty(1024 + ((T + 63) // 64 + 1) * d.hv * 33 * 1024, dtype=torch.uint8,
                            device=dev)
    o_serial = torch.empty_like(o)
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    for i in range(steps + 1):
        if i:
            ev_s[2 * i - 2].record(stream)
        gdn.gdn_prefill_chunked(q, k, v, g, beta, cu, pool, s0, s3, w.scale, o=o_serial,
                                workspace=serial_ws)
        if i:
            ev_s[2 * i - 1].record(stream)
        flush.zero_()
    torch.cuda.synchronize(dev)
    pre_serial = sum(ev_s[2 * i].elapsed_time(ev_s[2 * i + 1]) for i in range(steps)) / steps
    del serial_ws
    # split at T/2: [0, T/2) from slot 0 into slot 2, then [T/2, T) from slot 2
    half = T // 2
    cu_h = torch.tensor([0, half], dtype=torch.int32, device=dev)
    o_split = torch.empty_like(o)
    gdn.gdn_prefill_chunked(q[:half], k[:half], v[:half], g[:half], beta[:half], cu_h, pool, s0,
                            s2, w.scale, o=o_split[:half], workspace=ws)
    gdn.gdn_prefill_chunked(q[half:], k[half:], v[half:], g[half:], beta[half:], cu_h, pool, s2,
                            s2, w.scale, o=o_split[half:], workspace=ws)
    torch.cuda.synchronize(dev)
    assert gdn.gdn_get_device_status(clear=True) == 0
    rel = lambda x, y: float((x.float() - y.float()).abs().max() / y.float().abs().max())
    flops = prefill_flops_per_token(d.hv, d.dk, d.dv, w.chunk) * T
    tf = flops / (pre / 1e3) / 1e12
    res = {"workload": f"long-context prefill: 1 sequence x {T} tokens, nonzero initial state, "
                       "gating + chunked prefill (chunk 64), 16 QK / 32 V heads, head_dim 128, bf16",
           "tokens_per_s": round(T / (total / 1e3), 1),
           "layer_ms": round(total, 4), "prefill_kernel_ms": round(pre, 4),
           "prefill_tflops": round(tf, 2),
           "prefill_frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
           "prefill_path": "chunk-state scan: two segments, 3 x 32 chain CTAs",
           "serial_prefill_kernel_ms": round(pre_serial, 4),
           "scan_vs_serial_rel_err_o": rel(o, o_serial),
           "scan_vs_serial_rel_err_state": rel(pool[1], pool[3]),
           "split_at": half,
           "split_rel_err_o": rel(o_split, o),
           "split_rel_err_state": rel(pool[2], pool[1]),
           "workspace_mib": round(need / 2**20, 1)}
    del w, q, k, v, o, o_split, o_serial, ws
    return res


# ------------------------------------------------------------ oracle (CPU) --

def _oracle_decode_step(w, n, sub_pool, threads=None):
    """The CPU oracle on the first n sequences of a decode step: conv update,
    gating, recurrent decode (the same three steps the GPU step runs)."""
    import numpy as np

    import oracle
    d = w.dims
    x = w.x[:n].double().numpy()
    y, _ = oracle.conv1d_update(x, 1, w.conv_w.double().numpy(), None, w.conv_pool,
                                w.slots[:n].numpy().astype(np.int64))
    q, k, v = oracle.split_qkv(y, d.hqk, d.hv, d.dk, d.dv)
    g, beta = oracle.gating(w.a[:n], w.b[:n], w.A_log, w.dt_bias)
    oracle.gdn_decode(q, k, v, g, beta, 1, sub_pool, np.arange(n), scale=w.scale, threads=threads)


def cpu_baseline(w, budget_s, n=None):
    """Time the oracle as it stands on the host cores on whole decode steps
    of the same workload, repeated until about budget_s seconds."""
    n = w.n_seqs if n is None else n
    sub = w.state_pool[w.slots[:n].long().to(w.state_pool.device)].cpu()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    reps = 0
    while True:
        _oracle_decode_step(w, n, sub)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    # one thread: the first 16 sequences of the step, repeated for ~1/4 of the budget
    n1 = min(16, n)
    sub1 = sub[:n1].clone()
    t1 = time.perf_counter()
    reps1 = 0
    while True:
        _oracle_decode_step(w, n1, sub1, threads=1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 4 or reps1 >= 1000:
            break
    return {"value": round(reps * n / el, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} x decode step of {n} sequences (conv update + gating + "
                      f"recurrent decode, fp64 C oracle, {cores} threads), {el:.1f} s",
            "single_thread": {"value": round(reps1 * n1 / el1, 2), "unit": UNIT, "cores": 1,
                              "sample": f"{reps1} x the first {n1} sequences of the step, "
                                        f"1 thread, {el1:.1f} s"}}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import workloads
    w = workloads.decode()
    n_probe = 8
    sub = w.state_pool[w.slots[:n_probe].long()]
    t0 = time.perf_counter()
    _oracle_decode_step(w, n_probe, sub)
    per_seq = (time.perf_counter() - t0) / n_probe
    budget = 150.0
    K, Wm = args.steps, args.warmup
    n = int(max(1, min(w.n_seqs, budget / max(1, K + Wm) / per_seq)))
    sub = w.state_pool[w.slots[:n].long()]
    for _ in range(Wm):
        _oracle_decode_step(w, n, sub)
    t0 = time.perf_counter()
    for _ in range(K):
        _oracle_decode_step(w, n, sub)
    el = time.perf_counter() - t0
    value = K * n / el
    cores = os.cpu_count() or 1
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(el / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": DECODE_WORKLOAD, "global_batch": n, "seq_len": 1,
                       "sample": f"each step: the first {n} of the 256 sequences"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": f"{K} steps x {n} sequences of the decode step"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
