#!/usr/bin/env python
"""Benchmark of the Flint decode MoE layer on one GB300 (or N replicas).

Headline: one BF16 MoE decode layer (hidden 2048, 256 routed experts, sigmoid
top-6 + 1 shared, intermediate 512) at batch 8 with i.i.d. unit-RMS tokens,
timed as CUDA-graph replay with CUDA events, with a cold L2 for every step
(default: 8 distinct copies of the layer rotated per step; --l2 flush writes a
512 MiB buffer between steps instead).  Metric: HBM GB/s over the bytes the layer needs --
(U+1) experts x 6 MiB + the 1 MiB router, U = distinct selected experts -- and
the layer latency in microseconds.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the host instead (the comparison arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import flint_synth as fs  # noqa: E402

METRIC = "MoE decode-layer µs and HBM GB/s (selected-expert bytes) at batch 1/8/32/128"
EXPERT_BYTES_BF16 = 3 * 512 * 2048 * 2          # 6,291,456
ROUTER_BYTES = 256 * 2048 * 2                   # 1,048,576
EXPERT_BYTES_NVFP4 = 3 * 512 * 2048 // 2 + 3 * 512 * 2048 // 16   # 1,769,472 (+12 B of scales)
GATEUP_BYTES_BF16 = 2 * 512 * 2048 * 2          # 4,194,304
DOWN_BYTES_BF16 = 512 * 2048 * 2                # 2,097,152
L2_FLUSH_BYTES = 512 << 20
SPACER_CYCLES = 100_000
FALLBACK_HBM_GBS = 6800.0
LAYER_SEED, TOKEN_SEED, OFFSET_SEED = 1001, 2000, 1003
SMALL_BATCH_MAX = 8      # batches the library runs as one persistent kernel


def needed_bytes_bf16(U: int) -> int:
    return (U + 1) * EXPERT_BYTES_BF16 + ROUTER_BYTES


def needed_bytes_nvfp4(U: int) -> int:
    return (U + 1) * (EXPERT_BYTES_NVFP4 + 12) + ROUTER_BYTES


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = None
        if sel is None:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            sel = vis.split(",")[device_index] if vis else str(device_index)
        self.sel = sel

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, "--query-gpu=" + self.FIELDS, "--format=csv",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.strip().split(",")]
                if len(parts) < 9 or not parts[1].split()[0].isdigit():
                    continue
                rows.append(parts)
        os.unlink(self.path)
        sm = [int(r[1].split()[0]) for r in rows]
        mx = [int(r[2].split()[0]) for r in rows if r[2].split()[0].isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(self.REASONS, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- helpers

def stats_us(ms_list):
    us = sorted(1000.0 * t for t in ms_list)
    n = len(us)
    return {"mean": sum(us) / n, "p10": us[int(0.1 * (n - 1))], "p50": us[int(0.5 * (n - 1))],
            "p90": us[int(0.9 * (n - 1))]}


class Cold:
    """Keeps the L2 cold for every timed step.

    rotate (default): R distinct copies of the layer's weights (R x 1.6 GB,
      inputs far larger than L2); step i uses copy i mod R, so the weights a
      step reads were last touched R-1 steps (>= 7 x 45 MB > L2) earlier.
    flush: one copy; before each step a 512 MiB buffer is written (outside the
      events).  The write leaves ~L2-sized dirty data whose write-back then
      overlaps the timed step, so this mode over-states the layer's time.
    """

    def __init__(self, mode, W, device, copies=8):
        self.mode = mode
        if mode == "rotate":
            self.Ws = [W] + [{k: v.clone() for k, v in W.items()} for _ in range(copies - 1)]
            self.buf = None
        else:
            self.Ws = [W]
            self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.v = 0

    def weights(self, i):
        return self.Ws[i % len(self.Ws)]

    def before(self, i):
        if self.buf is not None:
            self.v = (self.v + 1) & 0xFF
            self.buf.fill_(self.v)
        else:
            # A ~50 us spin kernel (no memory traffic) between steps keeps the
            # GPU busy while the host enqueues the next step, so host launch
            # latency never lands inside the timed events.
            torch.cuda._sleep(SPACER_CYCLES)

    def describe(self):
        if self.mode == "rotate":
            return ("inputs larger than L2: %d distinct copies of the layer weights (%.1f GB), "
                    "rotated per step" % (len(self.Ws), len(self.Ws) * 1.618))
        return "flushed between timed steps (512 MiB write, outside the events)"


def timed_steps(fn, steps, warmup, cold, stream, barrier=None, sampler=None):
    """warmup untimed calls, then `steps` timed calls fn(i), each bracketed by
    CUDA events on `stream`; cold.before(i) runs outside the events."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            cold.before(i)
            fn(i)
        torch.cuda.synchronize()
        if barrier:
            barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        t0 = time.perf_counter()
        for i, (s, e) in enumerate(ev):
            cold.before(warmup + i)
            s.record(stream)
            fn(warmup + i)
            e.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        clocks = sampler.stop() if sampler else None
        if barrier:
            barrier()
    return [s.elapsed_time(e) for s, e in ev], wall, clocks


class Chain:
    """CUDA graphs of k consecutive calls call(0), ..., call(k - 1), k = 1..n,
    where call(i) runs one step on weight copy i: one replay times k steps
    between one pair of events.  An event pair around a one-launch graph costs
    ~5.6 us on a GB300 even for an empty kernel, ~1.2 us per launch when eight
    run back to back; chaining the steps (as a decode step chains its layers)
    keeps that fixed cost out of the per-step time.  With one weight copy
    (L2 flush mode) n is 1: every step is its own replay after a flush."""

    def __init__(self, call, n, stream):
        self.call, self.n, self.stream = call, n, stream
        self.graphs = {}
        with torch.cuda.stream(stream):
            for i in range(n):
                call(i)
            stream.synchronize()

    def replay(self, k):
        if k not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(k):
                        self.call(i)
            self.graphs[k] = g
        self.graphs[k].replay()


def chain_blocks(steps: int, n: int):
    """Replay sizes for exactly `steps` steps in replays of at most n."""
    return [n] * (steps // n) + ([steps % n] if steps % n else [])


def timed_chain(chain, steps, warmup, cold, stream, barrier=None, sampler=None):
    """Exactly `steps` timed steps as replays of up to chain.n chained steps
    (the last replay takes the remainder), after >= warmup untimed steps;
    cold.before runs before each replay, outside the events.  Returns one
    per-step time (replay time / its steps) for every step."""
    blocks = chain_blocks(steps, chain.n)
    for k in set(blocks):
        chain.replay(k)  # capture outside the timed region
    torch.cuda.synchronize()
    nwarm = -(-max(warmup, 1) // chain.n)
    times, wall, clocks = timed_steps(lambda j: chain.replay(blocks[j - nwarm] if j >= nwarm else chain.n),
                                      len(blocks), nwarm, cold, stream, barrier, sampler)
    per_step = []
    for k, t in zip(blocks, times):
        per_step += [t / k] * k
    return per_step, wall, clocks


class BF16Layer:
    def __init__(self, m, cold, B, bias_on, device, seed):
        self.m, self.cold, self.B = m, cold, B
        self.x, self.res = fs.tokens(seed, B, device=device)
        self.bias = fs.logit_offsets(OFFSET_SEED, device=device) if bias_on else None
        self.out = torch.empty_like(self.res)
        self.idx = torch.empty((B, 6), dtype=torch.int32, device=device)
        self.w = torch.empty((B, 6), dtype=torch.float32, device=device)
        self.ws = m.new_workspace(B, device=device)
        self.graphs = []

    def call(self, i=0, stream=None):
        W = self.cold.weights(i)
        self.m.flint_moe_decode_bf16(self.x, self.res, W["wr"], self.bias, W["w13"], W["w2"],
                                     W["ws13"], W["ws2"], self.out, self.ws, self.idx, self.w,
                                     stream=stream)

    def unique_experts(self) -> int:
        self.call()
        torch.cuda.synchronize()
        st = self.m.flint_moe_get_device_status(self.ws)
        if st != self.m.FLINT_OK:
            raise RuntimeError("device status " + self.m.status_string(st))
        return int(torch.unique(self.idx).numel())

    def capture(self, stream):
        """One CUDA graph per weight copy."""
        self.graphs = []
        with torch.cuda.stream(stream):
            for i in range(len(self.cold.Ws)):
                self.call(i, stream)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    self.call(i, stream)
                self.graphs.append(g)

    def replay(self, i):
        self.graphs[i % len(self.graphs)].replay()


def measure_bf16(m, cold, B, bias_on, seed, steps, warmup, stream, barrier=None, sampler=None):
    L = BF16Layer(m, cold, B, bias_on, cold.Ws[0]["wr"].device, seed)
    U = L.unique_experts()
    chain = Chain(lambda i: L.call(i, stream), len(cold.Ws), stream)
    times, wall, clocks = timed_chain(chain, steps, warmup, cold, stream, barrier, sampler)
    st = stats_us(times)
    nb = needed_bytes_bf16(U)
    return L, U, nb, times, st, wall, clocks


def single_call_us(L, steps, warmup, stream):
    """The same layer with an event pair around every one-call replay (the
    per-step fixed cost of events and graph launch included)."""
    L.capture(stream)
    times, _, _ = timed_steps(L.replay, steps, warmup, L.cold, stream)
    return stats_us(times)["mean"]


def stage_times(m, L, steps, warmup, stream):
    """Per-kernel CUDA-event durations of the three kernels, each launched alone
    on `stream` (route -> gate/up -> down on a routed workspace), chained over
    the weight copies like the layer steps."""
    cold = L.cold
    idx = torch.empty_like(L.idx)
    w = torch.empty_like(L.w)
    out = torch.empty_like(L.res)

    def route(i):
        W = cold.weights(i)
        m.flint_moe_route(L.x, W["wr"], L.bias, idx, w, L.ws, stream=stream)

    def gate(i):
        W = cold.weights(i)
        m.flint_moe_gateup_bf16(L.x, W["w13"], W["ws13"], L.ws, stream=stream)

    def down(i):
        W = cold.weights(i)
        m.flint_moe_down_bf16(L.res, W["w2"], W["ws2"], out, L.ws, stream=stream)

    res = {}
    for name, fn in (("router", route), ("gateup", gate), ("down", down)):
        with torch.cuda.stream(stream):
            route(0)
            gate(0)
        times, _, _ = timed_chain(Chain(fn, len(cold.Ws), stream), steps, warmup, cold, stream)
        res[name] = stats_us(times)
    torch.cuda.synchronize()
    return res


def e2e_measure(m, L, steps, warmup, stream):
    """Same layer through the public call with host buffers: pinned H2D of x and
    residual (kept next to each other, so one copy brings both), the decode
    call, D2H of out -- all inside the events."""
    x0, r0 = L.x, L.res
    xr = torch.stack([x0, r0])          # [2, B, H]: x, then the residual
    L.x, L.res = xr[0], xr[1]           # contiguous views the call reads
    xrh = xr.cpu().pin_memory()
    oh = torch.empty_like(L.out, device="cpu").pin_memory()

    def step(i):
        xr.copy_(xrh, non_blocking=True)
        L.call(i, stream)
        oh.copy_(L.out, non_blocking=True)

    try:
        times, _, _ = timed_steps(step, steps, warmup, L.cold, stream)
    finally:
        L.x, L.res = x0, r0
    return times, xrh.numel() * 2, oh.numel() * 2


def cpu_baseline(L, W_host, budget_s=10.0):
    import oracle
    x = L.x.cpu()
    res = L.res.cpu()
    bias = None if L.bias is None else L.bias.cpu()
    threads = oracle.max_threads()
    reps, t_tot = 0, 0.0
    while t_tot < budget_s and reps < 200:
        t0 = time.perf_counter()
        out, idx, _ = oracle.moe_bf16(fs.FULL, x, res, W_host["wr"], bias, W_host["w13"],
                                      W_host["w2"], W_host["ws13"], W_host["ws2"], nthreads=threads)
        t_tot += time.perf_counter() - t0
        reps += 1
    U = len(set(idx.reshape(-1).tolist()))
    per = t_tot / reps
    return {"value": needed_bytes_bf16(U) / per / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "us_per_layer": per * 1e6,
            "sample": "fp64 C oracle (selected experts only) on the full batch-%d layer, %d "
                      "repetitions, OpenMP over tokens" % (L.B, reps)}


# ---------------------------------------------------------------- arms

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    barrier = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        barrier = dist.barrier
    return world, rank, local, barrier


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, world, rank, local, barrier):
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as m
    m.lib()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peak, peak_kind = peaks()
    B = args.batch
    W = fs.layer_weights(LAYER_SEED, fs.FULL, device=device)
    cold = Cold(args.l2, W, device)
    sampler = ClockSampler(local)
    L, U, nb, times, st, wall, clocks = measure_bf16(
        m, cold, B, False, TOKEN_SEED + B, args.steps, args.warmup, stream, barrier, sampler)
    mean_ms = st["mean"] / 1000.0
    t_max = max_over_ranks(mean_ms, world)
    value = world * nb / (t_max / 1e3) / 1e9

    roof_steps = min(args.steps, 400)
    kern = stage_times(m, L, roof_steps, max(3, args.warmup // 4), stream)
    single_us = single_call_us(L, roof_steps, max(3, args.warmup // 4), stream)
    if B <= SMALL_BATCH_MAX:
        # The whole layer is one launch of the persistent kernel: the chained
        # steps time back-to-back launches of exactly that kernel on its stream.
        roof_kernel = "moe_small_bf16_kernel"
        alg_bytes = nb + 3 * B * 2048 * 2          # weights + x, residual, out
        dur_us = st["mean"]
    else:
        roof_kernel = "gateup_bf16_kernel"
        alg_bytes = (U + 1) * GATEUP_BYTES_BF16 + B * 2048 * 2 + 7 * B * 512 * 4
        dur_us = kern["gateup"]["mean"]
    achieved = alg_bytes / (dur_us * 1e-6) / 1e9
    traffic = recorded_traffic(roof_kernel, B)

    e2e_times, h2d, d2h = e2e_measure(m, L, min(args.steps, 1000), max(3, args.warmup // 4),
                                      stream)
    e2e_mean = stats_us(e2e_times)["mean"]
    e2e_t = max_over_ranks(e2e_mean, world)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "one BF16 Flint MoE decode layer, batch %d: hidden 2048, 256 routed "
                        "experts sigmoid top-6 + 1 shared, intermediate 512, N(0,0.02) weights, "
                        "unit-RMS N(0,1) tokens" % B,
            "batch": B, "unique_experts": U, "needed_bytes": nb,
            "l2": cold.describe(),
            "timing": "CUDA events around CUDA-graph replays of %d consecutive layer steps "
                      "(one per weight copy, %s per layer); time per step = replay time / %d"
                      % (len(cold.Ws), "one persistent kernel" if B <= SMALL_BATCH_MAX
                         else "3 kernels", len(cold.Ws)),
            "us_single_call": round(single_us, 3),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "us_per_layer": round(st["mean"], 3),
        "us_p10_p50_p90": [round(st["p10"], 3), round(st["p50"], 3), round(st["p90"], 3)],
        "frac_of_peak": round(nb / (st["mean"] * 1e-6) / 1e9 / peak, 4),
        "peak_gbs": peak, "peak_kind": peak_kind,
        "kernels_us": {k: round(v["mean"], 3) for k, v in kern.items()},
        "roofline": {"bound": "hbm", "kernel": roof_kernel, "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": alg_bytes,
                     "launch_us": round(dur_us, 3),
                     "note": "peak = %s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind},
        "e2e": {"value": round(world * nb / (e2e_t * 1e-6) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_t, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": (1 if B <= SMALL_BATCH_MAX else 3) * args.steps,
        "clocks": clocks,
        "wall_s_timed": round(wall, 4),
    }
    if args.extras and rank == 0:
        line["per_config"] = extras(m, cold, stream, args)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        W_host = {k: v.cpu() for k, v in W.items()}
        line["cpu_baseline"] = cpu_baseline(L, W_host)
    if rank == 0:
        print(json.dumps(line), flush=True)


def extras(m, cold, stream, args):
    """Secondary configurations (reported, not the headline)."""
    out = {}
    steps = max(50, min(args.steps, 500))
    for B, bias_on in ((1, False), (8, False), (32, True), (128, True)):
        L, U, nb, times, st, _, _ = measure_bf16(m, cold, B, bias_on, TOKEN_SEED + B, steps,
                                                 args.warmup, stream)
        out["bf16_b%d%s" % (B, "_skew" if bias_on else "")] = {
            "us": round(st["mean"], 3), "p50_us": round(st["p50"], 3), "unique_experts": U,
            "needed_bytes": nb, "gbs": round(nb / (st["mean"] * 1e-6) / 1e9, 1)}
        del L
    out.update(nvfp4_configs(m, cold, stream, steps, args.warmup))
    out.update(attn_configs(m, stream, steps, args.warmup))
    if args.stack:
        out.update(stack_configs(m, stream, args.warmup))
    return out


def nvfp4_configs(m, cold, stream, steps, warmup):
    """NVFP4 W4A16 layer at batch 1 and 8, and at 32 and 128 with skewed
    routing (weights packed from each bf16 copy)."""
    nvs = [fs.nvfp4_layer(W) for W in cold.Ws]
    torch.cuda.synchronize()
    out = {}
    for B, bias_on in ((1, False), (8, False), (32, True), (128, True)):
        x, res = fs.tokens(TOKEN_SEED + B, B, device=x_device(cold))
        bias = fs.logit_offsets(OFFSET_SEED, device=x_device(cold)) if bias_on else None
        o = torch.empty_like(res)
        idx = torch.empty((B, 6), dtype=torch.int32, device=x.device)
        ws = m.new_workspace(B, device=x.device)
        chain = Chain(lambda i: m.flint_moe_decode_nvfp4_w4a16(
            x, res, cold.Ws[i]["wr"], bias, nvs[i], o, ws, idx, None, stream=stream),
            len(cold.Ws), stream)
        torch.cuda.synchronize()
        U = int(torch.unique(idx).numel())
        times, _, _ = timed_chain(chain, steps, warmup, cold, stream)
        st = stats_us(times)
        nb = needed_bytes_nvfp4(U)
        out["nvfp4_b%d%s" % (B, "_skew" if bias_on else "")] = {
                                "us": round(st["mean"], 3), "p50_us": round(st["p50"], 3),
                                "unique_experts": U, "needed_bytes": nb,
                                "gbs": round(nb / (st["mean"] * 1e-6) / 1e9, 1)}
    del nvs
    return out


def attn_configs(m, stream, steps, warmup):
    """The attention side of a decode step (per-head Q/K RMSNorm + RoPE + bf16
    KV-cache write, one kernel) at batch 1 / 8 / 32 / 128: 8 distinct input
    sets (positions up to 2^18, a 4096-row cache each) chained per replay like
    the layer steps.  Its bytes (~20 KiB per token) stay in L2, so the figure is
    the kernel's latency, not a bandwidth claim."""
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {}
    for B in (1, 8, 32, 128):
        sets = []
        for i in range(8):
            d = {k: v.to(dev) for k, v in fs.attn_inputs(900 + 16 * B + i, B, 4096).items()}
            d["q"] = torch.empty((B, m.N_Q_HEADS, m.HEAD_DIM), dtype=torch.bfloat16, device=dev)
            sets.append(d)

        def call(i, sets=sets):
            d = sets[i]
            m.flint_qk_norm_rope_kv_bf16(d["qkv"], d["q_norm"], d["k_norm"], d["positions"],
                                         d["slot_mapping"], d["q"], d["k_cache"], d["v_cache"],
                                         1.0e6, 1e-6, stream=stream)

        class _Spacer:
            def before(self, i):
                torch.cuda._sleep(SPACER_CYCLES)

        times, _, _ = timed_chain(Chain(call, len(sets), stream), steps, warmup, _Spacer(), stream)
        st = stats_us(times)
        row = (m.N_Q_HEADS + 2 * m.N_KV_HEADS) * m.HEAD_DIM
        nbytes = B * row * 2 + 2 * m.HEAD_DIM * 2 + B * (m.N_Q_HEADS + 2 * m.N_KV_HEADS) * m.HEAD_DIM * 2
        out["qk_norm_rope_kv_b%d" % B] = {"us": round(st["mean"], 3), "p50_us": round(st["p50"], 3),
                                          "bytes": nbytes,
                                          "gbs": round(nbytes / (st["mean"] * 1e-6) / 1e9, 1)}
    return out


def x_device(cold):
    return cold.Ws[0]["wr"].device


STACK_LAYERS = 47


def stack_configs(m, stream, warmup, steps=20):
    """47 distinct BF16 MoE layers resident (~76 GB) applied in sequence, each
    taking the RMSNorm of the previous layer's output as its input (folded
    into the layer call): one decode step's MoE work, naturally cold in L2."""
    device = torch.device("cuda", torch.cuda.current_device())
    free, _ = torch.cuda.mem_get_info(device)
    need = STACK_LAYERS * 1.62e9 + 8e9
    if free < need:
        return {"stack47": {"skipped": "needs %.0f GB free, %.0f GB available"
                            % (need / 1e9, free / 1e9)}}
    layers = [fs.layer_weights(5000 + l, fs.FULL, device=device) for l in range(STACK_LAYERS)]
    torch.cuda.synchronize()
    out = {}
    for B in (1, 8, 32):
        _, r0 = fs.tokens(6000 + B, B, device=device)
        outs = [torch.empty_like(r0) for _ in range(STACK_LAYERS)]
        idx = torch.empty((STACK_LAYERS, B, 6), dtype=torch.int32, device=device)
        ws = m.new_workspace(B, device=device)

        def step_once():
            res = r0
            for l, W in enumerate(layers):
                m.flint_moe_decode_bf16_prenorm(res, W["wr"], None, W["w13"], W["w2"],
                                                W["ws13"], W["ws2"], outs[l], ws, 1e-6, idx[l],
                                                None, stream=stream)
                res = outs[l]

        with torch.cuda.stream(stream):
            step_once()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_once()
        torch.cuda.synchronize()
        nb = sum(needed_bytes_bf16(int(torch.unique(idx[l]).numel())) for l in range(STACK_LAYERS))

        class _Spacer:
            def before(self, i):
                torch.cuda._sleep(SPACER_CYCLES)

        times, _, _ = timed_steps(lambda i: g.replay(), steps, warmup, _Spacer(), stream)
        st = stats_us(times)
        out["stack47_b%d" % B] = {"us_per_step": round(st["mean"], 2), "p50_us": round(st["p50"], 2),
                                  "needed_bytes": nb, "gbs": round(nb / (st["mean"] * 1e-6) / 1e9, 1),
                                  "us_per_layer": round(st["mean"] / STACK_LAYERS, 3),
                                  # per layer: the RMSNorm folded into the persistent
                                  # kernel, or run before it / the three chained kernels
                                  "gpu_launches_per_step":
                                      (1 if B <= m.PRENORM_FUSED_MAX_BATCH else
                                       2 if B <= SMALL_BATCH_MAX else 4) * STACK_LAYERS}
        del g
    del layers
    torch.cuda.empty_cache()
    return out


def source_closure(tu: str):
    """The translation unit `tu` (a file under csrc/) and every header it
    includes, transitively, from csrc/ and include/ -- the files its kernels
    are compiled from."""
    import re
    dirs = [os.path.join(ROOT, "moe_decode_sigmoid_gb300", "csrc"), os.path.join(ROOT, "include")]
    seen, todo = {}, [tu]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        for d in dirs:
            path = os.path.join(d, name)
            if os.path.exists(path):
                seen[name] = path
                with open(path) as f:
                    todo += re.findall(r'^\s*#\s*include\s+"([^"]+)"', f.read(), re.M)
                break
    return [seen[n] for n in sorted(seen)]


def sources_sha(tu: str = None) -> str:
    """Hash of the CUDA sources a kernel is built from (the closure of its
    translation unit `tu`; every CUDA source when None): recorded ncu traffic
    only counts while it matches."""
    import hashlib
    h = hashlib.sha256()
    if tu is None:
        csrc = os.path.join(ROOT, "moe_decode_sigmoid_gb300", "csrc")
        paths = [os.path.join(csrc, n) for n in sorted(os.listdir(csrc))]
    else:
        paths = source_closure(tu)
    for path in paths:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, batch: int):
    """dram bytes (read + write) per launch from profiles/traffic.json, or None
    when no capture matches this kernel, batch and source revision."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get("%s_b%d" % (kernel, batch))
        if rec and rec.get("sources_sha") == sources_sha(rec.get("tu")):
            return rec.get("traffic_bytes")
    except Exception:
        pass
    return None


def run_reference(args, world, rank):
    """The comparison arm: the fp64 CPU oracle on the host cores, on the same
    workload as the GPU arm -- each step is the whole batch-B layer (router,
    selection, the selected and shared experts, combine), the computation the
    cpu_baseline of the GPU arm times, with OpenMP over the host's threads."""
    if rank != 0:
        return
    import oracle
    B = args.batch
    W = fs.layer_weights(LAYER_SEED, fs.FULL, device="cpu")
    x, res = fs.tokens(TOKEN_SEED + B, B, device="cpu")
    threads = oracle.max_threads()
    state = {}

    def step(i):
        out, idx, _ = oracle.moe_bf16(fs.FULL, x, res, W["wr"], None, W["w13"], W["w2"],
                                      W["ws13"], W["ws2"], nthreads=threads)
        state["idx"] = idx

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    wall = time.perf_counter() - t0
    per = wall / args.steps
    U = len(set(state["idx"].reshape(-1).tolist()))
    nb = needed_bytes_bf16(U)
    value = nb / per / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "one BF16 Flint MoE decode layer, batch %d: hidden 2048, 256 routed "
                               "experts sigmoid top-6 + 1 shared, intermediate 512, N(0,0.02) "
                               "weights, unit-RMS N(0,1) tokens" % B,
                   "batch": B, "unique_experts": U, "needed_bytes": nb},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "the whole batch-%d layer per step (fp64 C oracle, selected "
                                   "experts only, OpenMP over tokens on %d host threads)"
                                   % (B, threads)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(spec: str, calls: int):
    """A few decode calls of one layer (one weight copy, a couple of GB on the
    device), for small profiler captures: FMT:B with FMT bf16 or nvfp4.
    Prints one status line, not a bench line."""
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as m
    fmt, B = spec.split(":")
    B = int(B)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    W = fs.layer_weights(LAYER_SEED, fs.FULL, device=dev)
    nv = fs.nvfp4_layer(W) if fmt == "nvfp4" else None
    x, res = fs.tokens(TOKEN_SEED + B, B, device=dev)
    out = torch.empty_like(res)
    ws = m.new_workspace(B, device=dev)
    for _ in range(calls):
        if fmt == "nvfp4":
            m.flint_moe_decode_nvfp4_w4a16(x, res, W["wr"], None, nv, out, ws)
        else:
            m.flint_moe_decode_bf16(x, res, W["wr"], None, W["w13"], W["w2"], W["ws13"],
                                    W["ws2"], out, ws)
    torch.cuda.synchronize()
    st = m.flint_moe_get_device_status(ws)
    print("profile case %s: %d calls, device status %d" % (spec, calls, st), flush=True)
    if st != m.FLINT_OK:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--extras", action="store_true", default=True)
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stack", action="store_true", default=True,
                    help="also time the 47-layer stack (needs ~85 GB free)")
    ap.add_argument("--no-stack", dest="stack", action="store_false")
    ap.add_argument("--l2", choices=("rotate", "flush"), default="rotate",
                    help="cold-L2 method between timed steps")
    ap.add_argument("--profile-case", default=None, metavar="FMT:B",
                    help="only run --steps decode calls of one bf16|nvfp4 layer at batch B "
                         "(for profiler captures) and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.steps)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local, barrier = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local, barrier)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
