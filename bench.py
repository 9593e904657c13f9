#!/usr/bin/env python3
"""Benchmark of the recurrent-state decode step on GB300.

One step = one decode token of the serving workload (GDN, B = 256 requests,
H = 48 heads, d = 128, four independent layer pools, states pre-warmed by 256
eager updates) through all three storage variants, i.e. every step of the hot
path: eager FP32 (read / update / write the dense state), deferred FP32 base +
log (merge interval M = 16), per-window INT8 (window W = 16; appends, and the
window-end fold + requantization on the tensor cores on every 16th token).  The same tokens feed
the three variants.

Prints one JSON line.  ``value`` = head-steps (B * H * tokens * pools *
variants) per second over all ranks, inputs resident in HBM; ``e2e`` = the
same through ``ls_decode_step_host`` with host buffers; ``roofline`` = the
dominant kernel (the eager step) against the measured HBM copy bandwidth.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "state-update decode steps/sec (B*H*tokens) and achieved HBM GB/s vs GB300 peak"
UNIT = "head-steps/s"
WORKLOAD = "gdn_serving_b256_h48_4pools"
VARIANTS = (("eager", 0), ("deferred", 16), ("int8", 16))
SWEEP_W = (8, 16, 32, 64, 128)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling runs)")
    ap.add_argument("--only", default=None, help="comma list of variants to run")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip e2e, window sweep and CPU baseline (profiling runs)")
    ap.add_argument("--ring", type=int, default=64, help="distinct token inputs kept in HBM")
    ap.add_argument("--pools", type=int, default=None, help="override the pool count (profiling runs)")
    ap.add_argument("--window", type=int, default=None,
                    help="override the window / merge interval of the log variants (profiling runs)")
    ap.add_argument("--col-scales", action="store_true",
                    help="INT8 pools in the smoothed per-value-column format (profiling runs)")
    ap.add_argument("--compensators", type=int, default=0,
                    help="Compensator Tokens per INT8 state (profiling runs)")
    return ap.parse_args()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world: int) -> None:
    """Barrier over the ranks (no-op on one rank)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the timed interval)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (max_ms * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# sources each profiled kernel is compiled from (a change voids its counters)
KERNEL_SOURCES = {"eager_step_kernel": ("ls_eager.cu", "ls_device.cuh", "ls_internal.cuh")}


def kernel_sources_digest(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "recurrent_state_quantization_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, heads_per_launch: int):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, scaled
    to `heads_per_launch`; None when the kernel's sources changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = kernel_sources_digest(kernel)
    for line in open(path):
        m = dict(re.findall(r"(\w+)=(\S+)", line))
        if m.get("kernel") == kernel and m.get("sources") == digest:
            return float(m["dram_bytes_per_head"]) * heads_per_launch
    return None


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def make_pools(w, variant, window, dev, col_scales=False, compensators=0, k16=False, r16=False):
    from recurrent_state_quantization_gb300 import StatePool
    return [StatePool(w.num_slots, w.heads, variant, w.gate, window, device=dev,
                      col_scales=col_scales, compensators=compensators, k16=k16, r16=r16)
            for _ in range(w.pools)]


def prewarm(w, pools_by_variant, slot_idx, masks, dev):
    """Warm every pool's states with `prewarm_tokens` eager updates (the eager
    kernel), then copy the warmed states into the other variants' pools."""
    import torch
    from recurrent_state_quantization_gb300 import workloads as wl
    all_slots = torch.arange(w.num_slots, dtype=torch.int32, device=dev)
    eager = pools_by_variant["eager"]
    for p, pool in enumerate(eager):
        for t in range(-w.prewarm_tokens, 0):
            pool.decode_step(slot_idx, *wl.step_inputs(w, t, pool=p, device=dev, masks=masks))
        warm = pool.read(all_slots)
        for name, pools in pools_by_variant.items():
            if name != "eager":
                pools[p].load(all_slots, warm)
        del warm
    torch.cuda.synchronize()


def run_native(args, rank, world, local):
    import torch
    import __graft_entry__
    from recurrent_state_quantization_gb300 import bytemodel as bm
    from recurrent_state_quantization_gb300 import workloads as wl

    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    base = wl.WORKLOAD_BY_NAME[WORKLOAD]
    over = {}
    if args.batch is not None:
        over.update(batch=args.batch, num_slots=args.batch)
    if args.pools is not None:
        over.update(pools=args.pools)
    w = wl.Workload(**{**base.__dict__, **over}) if over else base
    only = set(args.only.split(",")) if args.only else None
    variants = [(n, W if (args.window is None or not W) else args.window)
                for n, W in VARIANTS if only is None or n in only]
    heads = w.batch * w.heads
    slot_idx = wl.slot_index(w, dev)
    masks = wl.static_masks(w, dev)

    fmt = {"col_scales": args.col_scales, "compensators": args.compensators}
    pools = {n: make_pools(w, n, W, dev, **(fmt if n == "int8" else {})) for n, W in variants}
    if "eager" not in pools:
        pools["eager"] = make_pools(w, "eager", 0, dev)
    prewarm(w, pools, slot_idx, masks, dev)

    # token inputs resident in HBM: a ring of distinct tokens per pool
    ring = max(1, min(args.ring, args.steps + args.warmup))
    inputs = [[wl.step_inputs(w, t, pool=p, device=dev, masks=masks) for t in range(ring)]
              for p in range(w.pools)]
    ys = {n: [torch.empty(w.batch, w.heads, w.d_v, device=dev) for _ in range(w.pools)]
          for n, _ in variants}
    stream = torch.cuda.current_stream()

    def one_step(t, ev=None):
        for vi, (n, _) in enumerate(variants):
            if ev is not None:
                ev[vi][0].record(stream)
            for p in range(w.pools):
                pools[n][p].decode_step(slot_idx, *inputs[p][t % ring], y=ys[n][p])
            if ev is not None:
                ev[vi][1].record(stream)

    for t in range(args.warmup):
        one_step(t)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in variants] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches
    start.record(stream)
    for t in range(args.steps):
        one_step(args.warmup + t, evs[t])
    stop.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = reduce_max(start.elapsed_time(stop), world, dev)

    hbm_peak, peak_kind = peaks()
    # per-variant figures: each variant timed on its own over whole windows
    # (a multiple of every window / merge interval), so they do not depend on
    # how --steps meets the windows; the headline stays the timed region above
    period = 1
    for _, W in variants:
        if W:
            period = period * W // math.gcd(period, W)
    per_tokens = period * max(1, -(-64 // period))
    per_variant = {}
    for n, W in variants:
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = args.warmup + args.steps
        torch.cuda.synchronize()
        a_ev.record(stream)
        for t in range(per_tokens):
            for p in range(w.pools):
                pools[n][p].decode_step(slot_idx, *inputs[p][(t0 + t) % ring], y=ys[n][p])
        b_ev.record(stream)
        torch.cuda.synchronize()
        ms = a_ev.elapsed_time(b_ev)
        hs = heads * w.pools * per_tokens
        per_hs = (bm.int8_bytes(w.gate, W, col_scales=args.col_scales, compensators=args.compensators)
                  if n == "int8" else bm.variant_bytes(n, w.gate, W))
        bytes_ = per_hs * hs
        gbs = bytes_ / (ms * 1e-3) / 1e9
        per_variant[n] = {"window": W or None, "tokens": per_tokens,
                          "ms_per_token_all_pools": ms / per_tokens,
                          "head_steps_per_s": hs / (ms * 1e-3),
                          "algorithmic_bytes_per_head_step": per_hs,
                          "achieved_gbs": gbs, "frac_of_" + peak_kind + "_hbm": gbs / hbm_peak}
    value = job_throughput(heads * w.pools * len(variants) * args.steps, world, elapsed_ms)
    # windows that close inside the headline's timed region: the pools start
    # at a boundary, so token t closes a window when (t + 1) % W == 0
    window_ends = {n: sum(1 for t in range(args.warmup, args.warmup + args.steps) if (t + 1) % W == 0)
                   for n, W in variants if W}
    # kernel launches per decode call: one step kernel; an INT8 pool without
    # compensator pairs also launches the tensor-core window-end fold after it
    # (every token; it returns at once unless a window closed)
    launches_per_step = w.pools * sum(2 if (n == "int8" and not args.compensators) else 1 for n, _ in variants)

    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic",
           "config": {"workload": w.name, "gate": "scalar (Gated DeltaNet)", "batch": w.batch,
                      "heads": w.heads, "d_k": w.d_k, "d_v": w.d_v, "pools": w.pools,
                      "variants": [f"{n}" + (f" window={W}" if W else "") +
                                   (" smoothed per-value-column" if n == "int8" and args.col_scales else "") +
                                   (f" + {args.compensators} compensator tokens"
                                    if n == "int8" and args.compensators else "") for n, W in variants],
                      "prewarm_tokens": w.prewarm_tokens, "distinct_token_inputs": ring,
                      "l2": "inputs larger than L2: every pool's state is 0.2-0.8 GB and the "
                            "step streams 4 pools x 3 variants (about 5 GB) per token",
                      "parallelism": f"{world} independent replica(s), no collective",
                      "window_ends_in_timed_region": window_ends,
                      "per_variant_timing": f"each variant alone over {per_tokens} tokens "
                                            f"(whole windows), after the timed region"},
           "gpu_launches": launches_per_step * args.steps,
           "variants": per_variant}

    # five repeats inside the timed region: consecutive blocks of whole windows
    # (the slowest token of each window is its window end), ms per step each;
    # a region shorter than five whole windows is cut into five equal blocks
    blk = args.steps // 5 // period * period
    whole = blk > 0
    if not whole:
        blk = args.steps // 5
    if blk > 0:
        block_ms = [evs[r * blk][0][0].elapsed_time(evs[(r + 1) * blk - 1][-1][1]) / blk
                    for r in range(5)]
        out["repeats"] = {"blocks": 5, "steps_per_block": blk, "ms_per_step": block_ms,
                          "median_ms_per_step": statistics.median(block_ms),
                          "blocks_are": "whole windows" if whole else
                                        "equal token blocks (fewer than five whole windows timed)"}

    # roofline of the dominant kernel, the eager step (one launch per call):
    # a run of back-to-back eager launches (every pool, several tokens), so
    # the state each launch leaves dirty in L2 is written back inside the run
    # and the average launch carries its full read and write traffic
    if "eager" in per_variant:
        runs = 16 * w.pools
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a_ev.record(stream)
        for t in range(runs // w.pools):
            for p in range(w.pools):
                pools["eager"][p].decode_step(slot_idx, *inputs[p][t % ring], y=ys["eager"][p])
        b_ev.record(stream)
        torch.cuda.synchronize()
        launch_ms = a_ev.elapsed_time(b_ev) / runs
        in_step_ms = sum(evs[t][0][0].elapsed_time(evs[t][0][1]) for t in range(args.steps)) / (
            args.steps * w.pools) if variants[0][0] == "eager" else None
        bytes_launch = bm.eager_bytes(w.gate) * heads
        achieved = bytes_launch / (launch_ms * 1e-3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": "eager_step_kernel", "achieved": achieved,
                           "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                           "frac": achieved / hbm_peak,
                           "algorithmic_bytes_per_launch": bytes_launch,
                           "launch_ms": launch_ms,
                           "timing": f"{runs} back-to-back launches (CUDA events on the launching "
                                     f"stream), after the timed region",
                           "launch_ms_in_timed_region": in_step_ms,
                           "traffic": ncu_traffic("eager_step_kernel", heads)}
    if clk is not None:
        out["clocks"] = clk

    if not args.no_extras:
        out["int8_window_sweep"] = window_sweep(w, slot_idx, masks, inputs, ring, dev, hbm_peak,
                                                peak_kind, pools["eager"])
        out["e2e"] = e2e(w, variants, pools, slot_idx, dev, world)
        out["rwkv6"] = rwkv6(dev, hbm_peak, peak_kind)
        out["kda"] = kda(dev, hbm_peak, peak_kind)
        out["split_replay_ablation"] = split_ablation(dev)
        if rank == 0:
            out["cpu_baseline"] = cpu_baseline(w, variants, budget_s=6.0)
    return out


def window_sweep(w, slot_idx, masks, inputs, ring, dev, peak, peak_kind, eager_pools):
    """INT8 head-steps/s and achieved algorithmic GB/s for each window W (a
    whole number of windows, 4 pools, warmed states); for W = 16 in the
    smoothed per-value-column format, without and with 4 Compensator Tokens
    (the full LeapQuant boundary format), and per-key-row with 4 Compensator
    Tokens (the ladder of LeapQuant §4.4 Table 2); with bfloat16 key-side log factors
    (DeltaLog §3.4), INT8 W = 16 and deferred FP32 M = 16; and with FP16
    records (LeapQuant §4.1, §4.3), INT8 W = 16 per-key-row and in the full
    LeapQuant format (smoothed + 4 FP16 Compensator Tokens)."""
    import torch
    from recurrent_state_quantization_gb300 import bytemodel as bm
    all_slots = torch.arange(w.num_slots, dtype=torch.int32, device=dev)
    res = []
    stream = torch.cuda.current_stream()
    heads = w.batch * w.heads
    cases = ([("int8", W_, False, 0, False, False) for W_ in SWEEP_W]
             + [("int8", 16, True, 0, False, False), ("int8", 16, False, 4, False, False),
                ("int8", 16, True, 4, False, False),
                ("int8", 16, False, 0, True, False), ("deferred", 16, False, 0, True, False),
                ("int8", 16, False, 0, False, True), ("int8", 16, True, 4, False, True)])
    for variant, W, cols, comp, k16, r16 in cases:
        pools = make_pools(w, variant, W, dev, col_scales=cols, compensators=comp, k16=k16,
                           r16=r16)
        for p in range(w.pools):
            pools[p].load(all_slots, eager_pools[p].read(all_slots))
        y = torch.empty(w.batch, w.heads, w.d_v, device=dev)
        tokens = max(2 * W, 64)
        for t in range(W):  # warm-up: one window
            for p in range(w.pools):
                pools[p].decode_step(slot_idx, *inputs[p][t % ring], y=y)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for t in range(tokens):
            for p in range(w.pools):
                pools[p].decode_step(slot_idx, *inputs[p][t % ring], y=y)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        hs = heads * w.pools * tokens
        p_k = 2 if (k16 or r16) else 4
        per = (bm.deferred_bytes(w.gate, W, p_k=p_k) if variant == "deferred" else
               bm.int8_bytes(w.gate, W, col_scales=cols, compensators=comp, p_k=p_k,
                             p_u=2 if r16 else 4))
        gbs = per * hs / (ms * 1e-3) / 1e9
        fmt = ("fp32 base" if variant == "deferred" else
               "smoothed per-value-column" if cols else "per-key-row")
        res.append({"variant": variant, "window": W,
                    "format": fmt + (f" + {comp} compensator tokens" if comp else "") +
                    (" + bf16 key log" if k16 else "") + (" + fp16 records" if r16 else ""),
                    "algorithmic_bytes_per_head_step": per,
                    "tokens": tokens, "head_steps_per_s": hs / (ms * 1e-3),
                    "achieved_gbs": gbs, "frac_of_" + peak_kind + "_hbm": gbs / peak})
        del pools
        torch.cuda.empty_cache()
    return res


def split_ablation(dev, batch=256, heads=48, cycles=8, reps=3):
    """Split-vs-fused replay (DeltaLog §5.3, Fig. 9): amortized time per token
    over whole merge cycles of GDN, KDA and RWKV6 at M = 4 and 8 (deferred
    FP32) and of GDN at W = 16 (INT8), one batch x heads pool per path, the
    two entry points timed alternately (median of `reps`)."""
    import statistics as st
    import torch
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import workloads as wl
    ops = (("gdn", "scalar", False), ("kda", "per_key", False), ("rwkv6", "per_key", True))
    cases = [(n, g, p, "deferred", M) for n, g, p in ops for M in (4, 8)]
    cases.append(("gdn", "scalar", False, "int8", 16))
    stream = torch.cuda.current_stream()
    slots = torch.arange(batch, dtype=torch.int32, device=dev)
    res = []
    for name, gate, plain, variant, M in cases:
        w = wl.custom(f"{name}_b{batch}_h{heads}", gate=gate, batch=batch, heads=heads,
                      tokens=cycles * M, seed=11, lam_scale=0.05)
        ins = [wl.step_inputs(w, t, device=dev) for t in range(16)]
        y = torch.empty(batch, heads, w.d_v, device=dev)
        pools = {path: StatePool(batch, heads, variant, gate, M, device=dev, plain=plain)
                 for path in ("fused", "split")}
        call = {"fused": lambda t: pools["fused"].decode_step(slots, *ins[t % 16], y=y),
                "split": lambda t: pools["split"].decode_step_split(slots, *ins[t % 16], y=y)}
        for path in call:  # one cycle of warm-up (allocates the split scratch)
            for t in range(M):
                call[path](t)
        times = {"fused": [], "split": []}
        for _ in range(reps):
            for path in ("fused", "split"):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                a.record(stream)
                for t in range(cycles * M):
                    call[path](t)
                b.record(stream)
                torch.cuda.synchronize()
                times[path].append(a.elapsed_time(b) * 1e3 / (cycles * M))
        f, s = st.median(times["fused"]), st.median(times["split"])
        res.append({"operator": name, "variant": variant, "M": M, "batch": batch, "heads": heads,
                    "fused_us_per_token": f, "split_us_per_token": s,
                    "speedup_split_over_fused": f / s})
        del pools, call
        torch.cuda.empty_cache()
    return res


def rwkv6(dev, peak, peak_kind, tokens=64):
    """RWKV6 (per-key decay, raw (k, v) updates; DeltaLog Table 1) on one
    256 x 48-head pool: eager and deferred (M = 16) head-steps/s and
    algorithmic GB/s, states warmed by one merge cycle."""
    import torch
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import bytemodel as bm
    from recurrent_state_quantization_gb300 import workloads as wl
    w = wl.custom("rwkv6_b256_h48", gate="per_key", batch=256, heads=48, tokens=tokens,
                  seed=7, lam_scale=0.05)
    slots = torch.arange(w.batch, dtype=torch.int32, device=dev)
    ins = [wl.step_inputs(w, t, device=dev) for t in range(16)]
    stream = torch.cuda.current_stream()
    out = {"workload": w.name, "gate": "per_key", "update": "plain (k, v)"}
    for variant, M in (("eager", 0), ("deferred", 16)):
        pool = StatePool(w.num_slots, w.heads, variant, w.gate, M, device=dev, plain=True)
        y = torch.empty(w.batch, w.heads, w.d_v, device=dev)
        for t in range(16):
            pool.decode_step(slots, *ins[t % 16], y=y)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for t in range(tokens):
            pool.decode_step(slots, *ins[t % 16], y=y)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        hs = w.batch * w.heads * tokens
        byt = bm.variant_bytes(variant, "per_key", M or 1)
        gbs = byt * hs / (ms * 1e-3) / 1e9
        out[variant] = {"window": M or None, "head_steps_per_s": hs / (ms * 1e-3),
                        "algorithmic_bytes_per_head_step": byt, "achieved_gbs": gbs,
                        "frac_of_" + peak_kind + "_hbm": gbs / peak}
        del pool
    torch.cuda.empty_cache()
    return out


def kda(dev, peak, peak_kind, tokens=64):
    """The KDA workload (per-key gate with 10 % long-lived channels, 128
    requests x 32 heads, one pool of 256 MB FP32 states): eager, deferred
    (M = 16) and INT8 (W = 32) head-steps/s and algorithmic GB/s over two INT8
    windows, states warmed by one window."""
    import torch
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import bytemodel as bm
    from recurrent_state_quantization_gb300 import workloads as wl
    w = wl.WORKLOAD_BY_NAME["kda_b128_h32_t512_longlived"]
    slots = wl.slot_index(w, dev)
    masks = wl.static_masks(w, dev)
    ins = [wl.step_inputs(w, t, device=dev, masks=masks) for t in range(16)]
    stream = torch.cuda.current_stream()
    out = {"workload": w.name, "gate": "per_key (KDA)"}
    for variant, W in (("eager", 0), ("deferred", 16), ("int8", 32)):
        pool = StatePool(w.num_slots, w.heads, variant, w.gate, W, device=dev)
        y = torch.empty(w.batch, w.heads, w.d_v, device=dev)
        for t in range(32):
            pool.decode_step(slots, *ins[t % 16], y=y)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for t in range(tokens):
            pool.decode_step(slots, *ins[t % 16], y=y)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        hs = w.batch * w.heads * tokens
        byt = bm.variant_bytes(variant, "per_key", W or 1)
        gbs = byt * hs / (ms * 1e-3) / 1e9
        out[variant] = {"window": W or None, "head_steps_per_s": hs / (ms * 1e-3),
                        "algorithmic_bytes_per_head_step": byt, "achieved_gbs": gbs,
                        "frac_of_" + peak_kind + "_hbm": gbs / peak}
        del pool
    torch.cuda.empty_cache()
    return out


def e2e(w, variants, pools, slot_idx, dev, world=1, tokens=24):
    """The same step through ls_decode_step_host: inputs copied from pinned host
    memory and y copied back inside the timed region, every call.  Layer pool
    p is driven on its own stream (the layer pools are independent), so one
    pool's host copies overlap another pool's kernels; every pool has its own
    host output buffer."""
    import torch
    from recurrent_state_quantization_gb300 import workloads as wl
    host = []
    for p in range(w.pools):
        row = []
        for t in range(4):
            ins = wl.step_inputs(w, 10_000 + t, pool=p, device=dev)
            row.append([x.cpu().pin_memory() for x in ins])
        host.append(row)
    hslots = slot_idx.cpu().pin_memory()
    hy = {(n, p): torch.empty(w.batch, w.heads, w.d_v).pin_memory()
          for n, _ in variants for p in range(w.pools)}
    streams = [torch.cuda.Stream(device=dev) for _ in range(w.pools)]
    torch.cuda.synchronize()

    def step(t):
        for n, _ in variants:
            for p in range(w.pools):
                pools[n][p].decode_step_host(hslots, *host[p][t % 4], hy[(n, p)],
                                             stream=streams[p])
        for s in streams:
            s.synchronize()  # the step's results are on the host

    for t in range(2):
        step(t)
    barrier(world)
    t0 = time.perf_counter()
    for t in range(tokens):
        step(t)
    dt = reduce_max(time.perf_counter() - t0, world, dev)
    heads = w.batch * w.heads
    calls = len(variants) * w.pools
    h2d = calls * (4 * w.batch + 4 * heads * (w.d_k * 2 + w.d_v + w.dl + 1))
    d2h = calls * 4 * heads * w.d_v
    return {"value": job_throughput(heads * calls * tokens, world, dt * 1e3), "unit": UNIT, "tokens": tokens,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "ls_decode_step_host (pinned host buffers, cudaMemcpyAsync inside the "
                   "library; one stream per layer pool; the host synchronizes on every y "
                   "every token)"}


def cpu_baseline(w, variants, budget_s=6.0, steps=None):
    """The double-precision CPU oracle, as it stands, on a bounded sample of the
    workload: the 48 heads of one slot, token after token, for each variant
    until `budget_s` seconds (or `steps` tokens) have passed."""
    import numpy as np
    import torch
    import oracle
    from recurrent_state_quantization_gb300 import workloads as wl
    oracle.build_oracle()
    idx = np.arange(w.heads, dtype=np.int64)
    total_hs, total_s, toks = 0, 0.0, {}
    for n, W in variants:
        if n == "eager":
            o = oracle.EagerOracle(w.heads, w.d_k, w.d_v, w.dl)
        elif n == "deferred":
            o = oracle.DeferredOracle(w.heads, w.d_k, w.d_v, w.dl, W)
        else:
            o = oracle.WindowInt8Oracle(w.heads, w.d_k, w.d_v, w.dl, W)
        one = wl.Workload(**{**w.__dict__, "batch": 1, "num_slots": 1})
        t_spent, t = 0.0, 0
        while (steps is None and t_spent < budget_s) or (steps is not None and t < steps):
            q, k, v, lam, beta = wl.step_inputs(one, t, device="cpu")
            args = (q.reshape(w.heads, -1).numpy(), k.reshape(w.heads, -1).numpy(),
                    v.reshape(w.heads, -1).numpy(), lam.reshape(w.heads, -1).numpy(),
                    beta.reshape(-1).numpy())
            t0 = time.perf_counter()
            o.step(idx, *args)
            t_spent += time.perf_counter() - t0
            t += 1
        toks[n] = t
        total_hs += w.heads * t
        total_s += t_spent
    return {"value": total_hs / total_s, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle", "host_cpu": cpu_model(), "nproc": os.cpu_count(),
            "sample": f"the {w.heads} heads of one slot of {w.name}, "
                      + ", ".join(f"{n}: {toks[n]} tokens" for n, _ in variants)
                      + "; double precision, OpenMP over heads; host time of the oracle calls"}


def cpu_model() -> str:
    """The host CPU's model name, as lscpu reports it (else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def run_reference(args):
    """The CPU oracle as the reference arm: each step = one token of the
    48 heads of one slot through the three variants."""
    import oracle  # noqa: F401
    from recurrent_state_quantization_gb300 import workloads as wl
    w = wl.WORKLOAD_BY_NAME[WORKLOAD]
    variants = list(VARIANTS)
    cpu_baseline(w, variants, steps=args.warmup)
    t0 = time.perf_counter()
    res = cpu_baseline(w, variants, steps=args.steps)
    wall = time.perf_counter() - t0
    value = res["value"]
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * (w.heads * len(variants)) / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "d_k": w.d_k,
                       "d_v": w.d_v, "pools": w.pools,
                       "variants": ["eager", "deferred window=16", "int8 window=16"],
                       "sample_per_step": f"{w.heads} heads of one slot x 3 variants"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": res["cores"],
                             "kind": "oracle", "sample": res["sample"],
                             "host_cpu": res["host_cpu"], "nproc": res["nproc"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": wall}


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0
    rank, world, local = dist_setup(args)
    out = run_native(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
