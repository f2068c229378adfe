"""Benchmark of the trellis-quantized MoE grouped GEMM on GB300.

One step = one pass of the routed-expert hot path over one batch: zero the
fp32 accumulator, routing sort, m-tile map, grouped GEMM (trellis decode fused
into the tcgen05 multiply, router-weighted combine), bf16 combine.  Default
workload: DeepSeek-V4-shaped decode, 32 tokens x top-6 of 256 experts,
K=4096 -> N=2048, 2-bit trellis L=16, TILE_M=16 (192 pairs, ~136 woken experts).

Steps cycle over 4 independent weight sets (as successive layers would), so the
~285 MB of woken packed bytes a step streams never sits warm in the 129 MB L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import os

import argparse
import concurrent.futures
import json
import multiprocessing
import platform
import shutil
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402

METRIC = "trellis-MoE grouped GEMM us/call, pairs/s, packed-weight GB/s vs roofline"
DEFAULT_WORKLOAD = "v4_decode_n32"
NUM_WEIGHT_SETS = 4
# the 8192-token prefill projections (Zipf routing), timed beside the headline
PREFILL_WORKLOADS = ("v4_prefill_n8192_up", "v4_prefill_n8192_down")
BLAS_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


# --------------------------------------------------------------- traffic model

def grouped_algorithmic_bytes(num_tiles: int, n: int, top_k: int, K: int, N: int, L: int) -> int:
    """Bytes the grouped GEMM must move per launch: each m-tile stages its
    expert's packed rows once (N*K/4 bytes; the pages' bandwidth bound), each
    pair's activation row is read once (K bf16), the fp32 accumulator is read
    and written once (n*N*4 each way), plus the fp16 LUT."""
    return num_tiles * N * K // 4 + n * top_k * K * 2 + n * N * 8 + (2 << L)


def grouped_flops(n: int, top_k: int, K: int, N: int) -> int:
    return 2 * n * top_k * K * N


def recorded_traffic(workload: str):
    """DRAM bytes per grouped launch from the ncu capture recorded under
    profiles/, used only while the kernel source still has the recorded hash."""
    import hashlib
    src = os.path.join(ROOT, "trellis_quantized_moe_sort_gb300", "csrc", "tq_grouped.cu")
    rec = os.path.join(ROOT, "profiles", "grouped_kernel_traffic.txt")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(rec):
            f = line.split()
            if len(f) == 3 and not line.startswith("#") and f[0] == h and f[1] == workload:
                return int(f[2])
    except OSError:
        pass
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    replica sets the job's time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


# --------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, smax, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = max(smax, float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- our arm

def _cuda(torch, a):
    import warnings
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")     # read-only numpy buffers: copied to the device anyway
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_ours(args, rank, world, dist):
    import torch
    import trellis_quantized_moe_sort_gb300 as tq
    from trellis_quantized_moe_sort_gb300 import build as b

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(tq.lib_path):
        b.build()
    if dist is not None:
        dist.barrier()
    tq.tq_init(local)
    shp = moe_inputs.shape(args.workload)
    n, k, E, K, N, L, T = shp.n, shp.top_k, shp.E, shp.K, shp.N, shp.L, args.tile_m
    P = n * k

    # ---- resident inputs: args.weight_sets independent layers
    sets = []
    for layer in range(args.weight_sets):
        prob = moe_inputs.make_problem(args.workload, layer=layer)
        sets.append({"x": _cuda(torch, prob.x_bits.view(np.int16)), "ids": _cuda(torch, prob.topk_ids),
                     "w": _cuda(torch, prob.topk_w), "packed": _cuda(torch, prob.packed),
                     "lut": _cuda(torch, prob.lut_bits.view(np.int16)), "prob": prob})
    cap = tq.tq_tile_map_capacity(n, k, E, T)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sorted_pairs = torch.empty(P, dtype=torch.int32, device="cuda")
    tiles = torch.empty((cap, 3), dtype=torch.int32, device="cuda")
    num_tiles = torch.empty(1, dtype=torch.int32, device="cuda")
    y32 = torch.empty((n, N), dtype=torch.float32, device="cuda")
    y = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]

    # the activation layout tq_moe_forward uses for this m-tile: token rows
    # gathered by the kernel, or a pair-sorted copy made by the prepare launch
    lay = tq.X_TOKENS if T <= tq.GATHER_MAX_TILE_M else tq.X_PAIR_SORTED
    x_sorted = None if lay == tq.X_TOKENS else torch.empty((P, K), dtype=torch.int16, device="cuda")

    ws = torch.empty(tq.tq_moe_workspace_size(n, k, E, K, N, T), dtype=torch.uint8, device="cuda")

    def step(i):
        """One step as a caller runs it: the whole routed-expert product
        (route + tile map clearing y32, grouped GEMM, combine) through the
        public call, inputs resident, no allocation."""
        s = sets[i % args.weight_sets]
        tq.tq_moe_forward(s["x"], s["packed"], s["lut"], s["ids"], s["w"], tile_m=T, pin=tq.ARM_GROUPED,
                          workspace=ws, y=y)

    def kernel_step(i, timed_slot=None):
        """The same step from the separate calls, with CUDA events around the
        grouped kernel (events between launches cost the programmatic overlap
        the whole-product call has, so the step above is timed without them)."""
        s = sets[i % args.weight_sets]
        # route + tile map clearing y32 (one launch), and for large m-tiles the
        # pair-sorted copy of x (a second launch)
        tq.tq_prepare(s["ids"], s["x"], E, T, cap, counts, offsets, sorted_pairs, tiles, num_tiles, x_sorted, y32)
        if timed_slot is not None:
            gev[timed_slot][0].record(stream)
        tq.tq_grouped_gemm(s["x"] if x_sorted is None else x_sorted, s["packed"], s["lut"], sorted_pairs, s["w"],
                           tiles, num_tiles, k, T, y32, x_layout=lay)
        if timed_slot is not None:
            gev[timed_slot][1].record(stream)
        tq.tq_combine(y32, y)

    lut_rate = tq.tq_probe_lut_rate(8)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # the warm-up steps run right before the timed region, so the GPU does
    # not sit idle (and drop its clocks) between them
    for i in range(args.warmup):
        step(i)
        kernel_step(i)
    torch.cuda.synchronize()
    code, where = tq.tq_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where} during warm-up")

    # timed region 1: the steps (the headline value)
    counts_before = tq.tq_launch_counts()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    counts_after = tq.tq_launch_counts()
    # timed region 2: the grouped kernel's own duration (the roofline's denominator)
    for i in range(args.steps):
        kernel_step(i, timed_slot=i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    code, where = tq.tq_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where} during the timed steps")
    ms_step = t0.elapsed_time(t1) / args.steps
    grouped_ms = float(np.mean([a.elapsed_time(b_) for a, b_ in gev]))
    launches = sum(counts_after[key] - counts_before[key] for key in counts_after)
    if dist is not None:
        ms_step, grouped_ms = max_over_ranks([ms_step, grouped_ms], dist, "cuda")

    # tiles per set (device) for the traffic model; correctness spot check vs nothing on the hot path
    tiles_per_set = []
    for i in range(args.weight_sets):
        kernel_step(i)
        torch.cuda.synchronize()
        tiles_per_set.append(int(num_tiles.item()))
    mean_tiles = float(np.mean(tiles_per_set))

    # ---- end to end through the public call with host buffers
    e2e = run_e2e(args, tq, torch, sets, n, k, E, K, N, T)
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    del sets, ws, x_sorted, y32, y
    torch.cuda.empty_cache()

    # ---- the 8192-token prefill projections at the native m-tile
    prefill = None
    if args.prefill:
        prefill = {}
        for name in PREFILL_WORKLOADS:
            prefill[name] = run_prefill_leg(args, tq, torch, name, local, lut_rate, sms, dist)
            torch.cuda.empty_cache()

    if rank != 0:
        return None
    # each grouped launch is timed on its own (events around it): the burst
    # tensor peak is the matching denominator
    hbm, bf16, bf16_sus, peak_src = measured_peaks()
    alg_bytes = grouped_algorithmic_bytes(int(round(mean_tiles)), n, k, K, N, L)
    achieved = alg_bytes / (grouped_ms * 1e-3) / 1e9
    flops = grouped_flops(n, k, K, N)
    t_hbm_us = alg_bytes / (hbm * 1e9) * 1e6
    t_tc_us = flops / (bf16 * 1e12) * 1e6
    bound = "hbm" if t_hbm_us >= t_tc_us else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4)}
    else:
        tf = flops / (grouped_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 2), "peak": bf16, "unit": "TFLOP/s",
                "frac": round(tf / bf16, 4)}
    traffic = args.traffic if args.traffic is not None else recorded_traffic(args.workload)
    roof.update({"traffic": traffic, "peak_source": peak_src, "kernel": "grouped_kernel",
                 "algorithmic_bytes": alg_bytes, "kernel_us": round(grouped_ms * 1e3, 2)})

    us_call = ms_step * 1e3
    line = {
        "metric": METRIC,
        "value": round(us_call, 2),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; uniform random bitstreams, N(0,1/K) fp16 LUT, N(0,1) bf16 activations)",
        "config": {
            "workload": f"{args.workload}: E={E} top-{k}, n={n} tokens ({P} pairs), K={K} -> N={N}, "
                        f"2-bit trellis L={L}, TILE_M={T}",
            "global_batch": n, "pairs": P, "tile_m": T, "mean_m_tiles": mean_tiles,
            "l2": f"inputs larger than L2: {args.weight_sets} weight sets cycled, "
                  f"~{mean_tiles * N * K / 4 / 1e6:.0f} MB of woken packed bytes per step vs 129 MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "pairs_per_s": round(world * P / (ms_step * 1e-3), 1),
        "packed_GBps": round(mean_tiles * N * K / 4 / (grouped_ms * 1e-3) / 1e9, 1),
        "grouped_kernel_us": round(grouped_ms * 1e3, 2),
        "roofline": roof,
        "decode_ceiling": decode_ceiling(mean_tiles, N, K, clk, lut_rate, grouped_ms * 1e3, sms),
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": e2e,
    }
    if prefill is not None:
        line["prefill"] = prefill
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, moe_inputs.make_problem(args.workload, layer=0),
                                            budget_s=args.cpu_seconds)
    return line


def run_prefill_leg(args, tq, torch, name, local, lut_rate, sms, dist):
    """One 8192-token prefill projection (Zipf routing) as a caller runs it:
    tq_moe_forward at the native m-tile on the grouped arm, inputs resident
    (512 MiB of packed weights per call, all 256 experts woken: larger than
    L2).  The whole call is timed over the steps; then the same steps from
    the separate calls with CUDA events around each grouped launch.  Clocks
    are sampled throughout.  The roofline is the dense bf16 tensor roofline
    (2 * pairs * K * N flops) against the measured burst peak, since each
    launch is timed on its own."""
    prob = moe_inputs.make_problem(name)
    s = prob.shape
    n, k, E, K, N, L = s.n, s.top_k, s.E, s.K, s.N, s.L
    P = n * k
    d = {"x": _cuda(torch, prob.x_bits.view(np.int16)), "ids": _cuda(torch, prob.topk_ids),
         "w": _cuda(torch, prob.topk_w), "packed": _cuda(torch, prob.packed),
         "lut": _cuda(torch, prob.lut_bits.view(np.int16))}
    del prob
    T = tq.tq_native_tile_m(n, k, E)
    cap = tq.tq_tile_map_capacity(n, k, E, T)
    ws = torch.empty(tq.tq_moe_workspace_size(n, k, E, K, N, tq.TILE_NATIVE), dtype=torch.uint8, device="cuda")
    y = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sp = torch.empty(P, dtype=torch.int32, device="cuda")
    tiles = torch.empty((cap, 3), dtype=torch.int32, device="cuda")
    nt = torch.empty(1, dtype=torch.int32, device="cuda")
    y32 = torch.empty((n, N), dtype=torch.float32, device="cuda")
    lay = tq.X_TOKENS if T <= tq.GATHER_MAX_TILE_M else tq.X_PAIR_SORTED
    xs = None if lay == tq.X_TOKENS else torch.empty((P, K), dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()
    steps = args.prefill_steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def call():
        tq.tq_moe_forward(d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=tq.TILE_NATIVE,
                          pin=tq.ARM_GROUPED, workspace=ws, y=y)

    def kernel(ev=None):
        tq.tq_prepare(d["ids"], d["x"], E, T, cap, counts, offsets, sp, tiles, nt, xs, y32)
        if ev is not None:
            ev[0].record(stream)
        tq.tq_grouped_gemm(d["x"] if xs is None else xs, d["packed"], d["lut"], sp, d["w"], tiles, nt, k, T, y32,
                           x_layout=lay)
        if ev is not None:
            ev[1].record(stream)
        tq.tq_combine(y32, y)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # warm-up right before the timed region (the GPU does not idle in between)
    for _ in range(args.warmup):
        call()
        kernel()
    torch.cuda.synchronize()
    code, where = tq.tq_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where} during {name} warm-up")
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        call()
    t1.record(stream)
    for i in range(steps):
        kernel(evs[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    code, where = tq.tq_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where} during {name}")
    us_call = t0.elapsed_time(t1) / steps * 1e3
    kern_us = float(np.mean([a.elapsed_time(b_) for a, b_ in evs])) * 1e3
    if dist is not None:
        us_call, kern_us = max_over_ranks([us_call, kern_us], dist, "cuda")
    ntiles = int(nt.item())
    _, bf16, _, peak_src = measured_peaks()
    flops = grouped_flops(n, k, K, N)
    tf = flops / (kern_us * 1e-6) / 1e12
    lookups = ntiles * N * K
    mhz = (clk or {}).get("sm_mhz") or 2070.0
    ceiling_us = lookups / (sms * mhz * 1e6 * lut_rate) * 1e6
    return {
        "workload": f"{name}: E={E} top-{k} (Zipf s={s.zipf_s}), n={n} tokens ({P} pairs), K={K} -> N={N}, "
                    f"2-bit trellis L={L}, kernel TILE_M={T} (native)",
        "api": "tq_moe_forward (tile_m=TQ_TILE_NATIVE, pin=grouped)",
        "tile_m": T, "m_tiles": ntiles, "steps": steps,
        "us_per_call": round(us_call, 1),
        "grouped_kernel_us": round(kern_us, 1),
        "pairs_per_s": round(P / (us_call * 1e-6), 1),
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(tf / bf16, 4), "peak_kind": "burst (each launch timed on its own)",
                     "peak_source": peak_src, "kernel": "grouped_kernel", "flops": flops,
                     "traffic": recorded_traffic(name)},
        "lookups": lookups,
        "decode_ceiling": {"ceiling_us": round(ceiling_us, 1), "frac": round(ceiling_us / kern_us, 4),
                           "lookups_per_clk_per_sm_measured": round(lut_rate, 3)},
        "l2": "inputs larger than L2: 512 MiB of packed weights per call (every expert woken)",
        "clocks": clk,
    }


def decode_ceiling(mean_tiles, N, K, clk, rate, kernel_us, sms):
    """Every weight of every staged (m-tile, expert) is one random lookup in
    the 2^16-entry LUT held in shared memory; `rate` is that lookup rate as
    measured on this GPU by tq_probe_lut_rate (lookups per clock per SM).
    The decode cannot beat lookups / (SMs x rate x clock)."""
    lookups = mean_tiles * N * K
    mhz = (clk or {}).get("sm_mhz") or 2070.0
    ceiling_us = lookups / (sms * mhz * 1e6 * rate) * 1e6
    return {"lookups": int(lookups), "lookups_per_clk_per_sm_measured": round(rate, 3),
            "ceiling_us": round(ceiling_us, 1), "sm_mhz": mhz, "frac": round(ceiling_us / kernel_us, 4),
            "kernel_lookups_per_clk_per_sm": round(lookups / (kernel_us * 1e-6) / sms / (mhz * 1e6), 3)}


def run_e2e(args, tq, torch, sets, n, k, E, K, N, T):
    """Same step through tq_moe_forward with host buffers: every step copies
    its batch's activations and routing from pinned host memory, runs the
    call and reads y back.  The copies run on a second stream into two
    alternating device buffer sets, so step i+1's inputs travel while step i
    computes and step i's output travels while step i+1 computes; the timed
    region spans the first input copy to the last output copy."""
    hosts = []
    for s in sets:
        prob = s["prob"]
        hosts.append({
            "x": torch.from_numpy(prob.x_bits.view(np.int16).copy()).pin_memory(),
            "ids": torch.from_numpy(np.ascontiguousarray(prob.topk_ids)).pin_memory(),
            "w": torch.from_numpy(np.ascontiguousarray(prob.topk_w)).pin_memory(),
        })
    bufs = [{"x": torch.empty((n, K), dtype=torch.int16, device="cuda"),
             "ids": torch.empty((n, k), dtype=torch.int32, device="cuda"),
             "w": torch.empty((n, k), dtype=torch.float32, device="cuda"),
             "y": torch.empty((n, N), dtype=torch.bfloat16, device="cuda"),
             "yh": torch.empty((n, N), dtype=torch.bfloat16).pin_memory(),
             "ws": torch.empty(tq.tq_moe_workspace_size(n, k, E, K, N, T), dtype=torch.uint8, device="cuda"),
             "in_ready": torch.cuda.Event(), "done": torch.cuda.Event()} for _ in range(2)]
    compute = torch.cuda.current_stream()
    copies = torch.cuda.Stream()

    def h2d(i):
        b, h = bufs[i % 2], hosts[i % args.weight_sets]
        with torch.cuda.stream(copies):
            b["x"].copy_(h["x"], non_blocking=True)
            b["ids"].copy_(h["ids"], non_blocking=True)
            b["w"].copy_(h["w"], non_blocking=True)
            b["in_ready"].record(copies)

    def run(steps, first):
        h2d(first)
        for i in range(first, first + steps):
            b = bufs[i % 2]
            compute.wait_event(b["in_ready"])
            tq.tq_moe_forward(b["x"], sets[i % args.weight_sets]["packed"], sets[i % args.weight_sets]["lut"],
                              b["ids"], b["w"], tile_m=T, pin=tq.ARM_GROUPED, workspace=b["ws"], y=b["y"])
            b["done"].record(compute)
            # step i+1's inputs: issued after step i's call (so the GPU starts
            # step i first), queued on the copy stream after step i-1's output
            # copy, which waited for step i-1: that buffer set is free
            if i + 1 < first + steps:
                h2d(i + 1)
            copies.wait_event(b["done"])
            with torch.cuda.stream(copies):
                b["yh"].copy_(b["y"], non_blocking=True)
        compute.wait_stream(copies)

    run(args.warmup, 0)
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(compute)
    copies.wait_stream(compute)
    run(args.steps, args.warmup)
    b_.record(compute)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b_) / args.steps
    h2d_bytes = n * K * 2 + n * k * 4 + n * k * 4
    return {"value": round(ms * 1e3, 2), "unit": "us/call", "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": n * N * 2,
            "api": "tq_moe_forward (pin=grouped); copies on a second stream, overlapping the neighbouring steps"}


# --------------------------------------------------------------- CPU oracle

_ORACLE = {}


def _oracle_worker_init(folder, L):
    """Worker set-up: the batch's arrays, memory-mapped from the files the
    parent wrote (the packed weights are read only for the rows a task asks)."""
    for key in ("x", "ids", "w", "packed", "lut"):
        _ORACLE[key] = np.load(os.path.join(folder, key + ".npy"), mmap_mode="r")
    _ORACLE["L"] = L


def _oracle_worker_rows(rows):
    """One task: the oracle's product for every pair of the batch on the given
    output rows; returns the seconds it took on this worker's core."""
    import oracle.trellis_moe as O
    d = _ORACLE
    t0 = time.perf_counter()
    O.moe_forward(d["x"], d["ids"], d["w"], d["packed"], d["lut"], d["L"], rows=np.asarray(rows))
    return time.perf_counter() - t0


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


class OraclePool:
    """The CPU oracle, as it stands, on every host core: one worker process
    per core (started with spawn; single-threaded BLAS each, so the workers
    do not oversubscribe the cores), each computing a slice of the output rows
    of the same batch.  Throughput = output rows finished / wall time, scaled
    to the whole call (the oracle's cost is linear in the rows)."""

    def __init__(self, prob, cores=None):
        self.prob = prob
        self.cores = max(1, int(cores or os.cpu_count() or 1))
        self.dir = tempfile.mkdtemp(prefix="tq_oracle_")
        for key, arr in (("x", prob.x_bits), ("ids", prob.topk_ids), ("w", prob.topk_w),
                         ("packed", prob.packed), ("lut", prob.lut_bits)):
            np.save(os.path.join(self.dir, key + ".npy"), np.ascontiguousarray(arr))
        saved = {v: os.environ.get(v) for v in BLAS_THREAD_VARS}
        for v in BLAS_THREAD_VARS:
            os.environ[v] = "1"                      # inherited by the spawned workers
        try:
            self.pool = concurrent.futures.ProcessPoolExecutor(
                self.cores, mp_context=multiprocessing.get_context("spawn"),
                initializer=_oracle_worker_init, initargs=(self.dir, prob.shape.L))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
        # start every worker (imports, first call) outside any timed sample
        list(self.pool.map(_oracle_worker_rows, [[0]] * self.cores))

    def sample(self, budget_s, rows_per_task=16, seed=1):
        """Row slices on all workers until `budget_s` of wall time has passed
        (then the tasks in flight finish).  Returns (wall s, rows done, summed
        per-task seconds)."""
        N = self.prob.shape.N
        order = np.random.Generator(np.random.PCG64(seed)).permutation(N)
        chunks = [np.sort(order[i:i + rows_per_task]).tolist() for i in range(0, N, rows_per_task)]
        pending, done_rows, busy, nxt = {}, 0, 0.0, 0
        t0 = time.perf_counter()
        while True:
            while len(pending) < 2 * self.cores and time.perf_counter() - t0 < budget_s:
                rows = chunks[nxt % len(chunks)]
                nxt += 1
                pending[self.pool.submit(_oracle_worker_rows, rows)] = len(rows)
            if not pending:
                break
            finished, _ = concurrent.futures.wait(list(pending), return_when=concurrent.futures.FIRST_COMPLETED)
            for f in finished:
                busy += f.result()
                done_rows += pending.pop(f)
        return time.perf_counter() - t0, done_rows, busy

    def close(self):
        self.pool.shutdown(wait=True)
        shutil.rmtree(self.dir, ignore_errors=True)


def cpu_baseline(workload, prob, budget_s=15.0, pool=None):
    """The CPU oracle on every host core, on a bounded sample of the batch:
    all its pairs against as many output rows as the budget allows (rows
    cycle through a fixed permutation); us/call = wall time x N / rows.  The
    one-core figure (summed per-task seconds x N / rows) is reported beside."""
    own = pool is None
    pool = pool or OraclePool(prob)
    try:
        wall, rows, busy = pool.sample(budget_s)
    finally:
        if own:
            pool.close()
    s = prob.shape
    return {"value": round(wall / rows * s.N * 1e6, 1), "unit": "us/call", "cores": pool.cores, "kind": "oracle",
            "sample": f"{workload}: all {s.pairs} pairs x {rows} output rows (of {s.N}, cycling) on "
                      f"{pool.cores} worker processes in {wall:.1f} s wall, scaled by N/rows",
            "cpu": cpu_model(),
            "one_core_us_per_call": round(busy / rows * s.N * 1e6, 1)}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on every host core, each step a
    bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return None
    prob = moe_inputs.make_problem(args.workload)
    per_step = []
    pool = OraclePool(prob)
    try:
        for i in range(args.warmup + args.steps):
            r = cpu_baseline(args.workload, prob, budget_s=max(0.5, args.cpu_seconds / max(args.steps, 1)),
                             pool=pool)
            if i >= args.warmup:
                per_step.append(r)
    finally:
        pool.close()
    value = float(np.mean([r["value"] for r in per_step]))
    s = prob.shape
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"{args.workload}: E={s.E} top-{s.top_k}, n={s.n}, K={s.K} -> N={s.N}, "
                               f"L={s.L}, TILE_M={args.tile_m}"},
        "cpu_baseline": {"value": round(value, 1), "unit": "us/call", "cores": per_step[0]["cores"],
                         "kind": "oracle", "sample": per_step[0]["sample"], "cpu": per_step[0]["cpu"],
                         "one_core_us_per_call": round(float(np.mean([r["one_core_us_per_call"]
                                                                      for r in per_step])), 1)},
        "e2e": {"value": round(value, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_sweep(args):
    """Every workload, both arms, each launch timed alone after an L2 flush
    (median of args.steps); one JSON line per (workload, arm, TILE_M).  This
    is the per-configuration table and the GB300 gate study."""
    import torch
    import trellis_quantized_moe_sort_gb300 as tq
    from trellis_quantized_moe_sort_gb300 import build as b
    b.build()
    torch.cuda.set_device(0)
    tq.tq_init(0)
    hbm, bf16, bf16_sus, peak_src = measured_peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    names = args.sweep_workloads.split(",") if args.sweep_workloads else list(moe_inputs.WORKLOADS)
    for name in names:
        prob = moe_inputs.make_problem(name)
        s = prob.shape
        lines = []
        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        d = {"x": _cuda(torch, prob.x_bits.view(np.int16)), "ids": _cuda(torch, prob.topk_ids),
             "w": _cuda(torch, prob.topk_w), "packed": _cuda(torch, prob.packed),
             "lut": _cuda(torch, prob.lut_bits.view(np.int16))}
        y32 = torch.zeros((s.n, s.N), dtype=torch.float32, device="cuda")

        def timed(fn, flush_l2=True):
            fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(args.steps):
                if flush_l2:
                    flush.zero_()
                else:
                    fn()   # keeps the GPU busy while the timed launch is enqueued; leaves L2 warm
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b_.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b_) * 1e3)
            return float(np.median(ts))

        tiles_list = [int(t) for t in args.sweep_tiles.split(",")]
        auto_layout = lambda T: tq.X_TOKENS if T <= tq.GATHER_MAX_TILE_M else tq.X_PAIR_SORTED
        layouts = (lambda T: (tq.X_TOKENS, tq.X_PAIR_SORTED)) if args.sweep_both_layouts else \
            (lambda T: (auto_layout(T),))
        arms = [("grouped", T, lay) for T in tiles_list for lay in layouts(T)]
        if s.n <= 1024 and not args.sweep_no_gemv:
            arms.append(("gemv", None, None))
        if args.sweep_dequant:
            arms += [("dequant", T, auto_layout(T)) for T in tiles_list]
        w_dense = None
        for arm, T, lay in arms:
            extra = {}
            if arm == "grouped":
                _, offsets, sp = tq.tq_route(d["ids"], s.E)
                cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, T)
                tiles, nt = tq.tq_build_tile_map(offsets, T, cap)
                xin = d["x"]
                if lay == tq.X_PAIR_SORTED:
                    # the pair-sorted copy (one pass) the kernel then reads with box copies
                    xin = tq.tq_gather_rows(d["x"], sp, s.top_k)
                    extra["gather_us"] = round(timed(lambda: tq.tq_gather_rows(d["x"], sp, s.top_k, xin)), 1)
                torch.cuda.synchronize()
                ntiles = int(nt.item())
                call = lambda: tq.tq_grouped_gemm(xin, d["packed"], d["lut"], sp, d["w"], tiles, nt, s.top_k, T, y32,
                                                  x_layout=lay)
                us = timed(call)
                extra["x_layout"] = "tokens" if lay == tq.X_TOKENS else "pair_sorted"
                extra["hot_l2_us"] = round(timed(call, flush_l2=False), 1)
                # host cost of one call (Python binding + C ABI + launch), GPU kept busy
                torch.cuda.synchronize()
                flush.zero_()
                h0 = time.perf_counter()
                for _ in range(20):
                    call()
                extra["host_us_per_call"] = round((time.perf_counter() - h0) / 20 * 1e6, 1)
                torch.cuda.synchronize()
                staged = ntiles * s.N * s.K // 4
            elif arm == "dequant":
                # dequantize-materialize comparator: every woken expert decoded
                # to dense bf16 (slot = expert id; other slots skipped), then the
                # same grouped GEMM with A read from the dense copy
                _, offsets, sp = tq.tq_route(d["ids"], s.E)
                cap = tq.tq_tile_map_capacity(s.n, s.top_k, s.E, T)
                tiles, nt = tq.tq_build_tile_map(offsets, T, cap)
                xin = d["x"] if lay == tq.X_TOKENS else tq.tq_gather_rows(d["x"], sp, s.top_k)
                woken_ids = np.unique(prob.topk_ids)
                ids = np.full(s.E, -1, dtype=np.int32)
                ids[woken_ids] = woken_ids
                ids_d = _cuda(torch, ids)
                if w_dense is None:
                    w_dense = torch.empty((s.E, s.N, s.K), dtype=torch.bfloat16, device="cuda")
                torch.cuda.synchronize()
                ntiles = int(nt.item())
                deq_us = timed(lambda: tq.tq_dequantize(d["packed"], d["lut"], expert_ids=ids_d, w_out=w_dense))
                gemm_us = timed(lambda: tq.tq_grouped_gemm_dense(xin, w_dense, sp, d["w"], tiles, nt, s.top_k, T,
                                                                 y32, x_layout=lay))
                us = deq_us + gemm_us
                staged = ntiles * s.N * s.K // 4
                mat = len(woken_ids) * s.N * s.K * 2
                extra = {"dequant_us": round(deq_us, 1), "dense_gemm_us": round(gemm_us, 1),
                         "materialized_GB": round(mat / 1e9, 3),
                         "dequant_write_GBps": round(mat / (deq_us * 1e-6) / 1e9, 1),
                         "dense_gemm_weight_GBps": round(ntiles * s.N * s.K * 2 / (gemm_us * 1e-6) / 1e9, 1)}
            else:
                us = timed(lambda: tq.tq_gemv(d["x"], d["packed"], d["lut"], d["ids"], d["w"], y32))
                # the same arm as tq_moe_forward runs it: one launch writing bf16 y
                ws = torch.empty(max(256, tq.tq_moe_workspace_size(s.n, s.top_k, s.E, s.K, s.N, 16)),
                                 dtype=torch.uint8, device="cuda")
                y = torch.empty((s.n, s.N), dtype=torch.bfloat16, device="cuda")
                extra["forward_us"] = round(timed(lambda: tq.tq_moe_forward(
                    d["x"], d["packed"], d["lut"], d["ids"], d["w"], tile_m=16, pin=tq.ARM_GEMV, workspace=ws,
                    y=y)), 1)
                del ws, y
                ntiles = None
                staged = s.pairs * s.N * s.K // 4
            code, where = tq.tq_device_error()
            if code:
                raise RuntimeError(f"device error {code} at {where} ({name}, {arm})")
            woken = len(np.unique(prob.topk_ids))
            m_tiles = ntiles if ntiles is not None else woken
            alg = grouped_algorithmic_bytes(m_tiles, s.n, s.top_k, s.K, s.N, s.L)
            flops = grouped_flops(s.n, s.top_k, s.K, s.N)
            t_hbm = alg / (hbm * 1e9) * 1e6
            t_tc = flops / (bf16 * 1e12) * 1e6        # each launch timed alone: the burst peak
            lookups = (ntiles if ntiles is not None else s.pairs) * s.N * s.K
            if arm == "dequant":
                lookups = woken * s.N * s.K
            extra["dispatch_T16"] = {1: "gemv", 2: "grouped"}[tq.tq_select_arm(s.n, s.top_k, s.E, 16)]
            extra["dispatch_measured"] = {1: "gemv", 2: "grouped"}[tq.tq_select_arm(s.n, s.top_k, s.E, 16,
                                                                                    tq.ARM_MEASURED)]
            extra["native_tile_m"] = tq.tq_native_tile_m(s.n, s.top_k, s.E)
            lines.append(({**extra, 
                "workload": name, "arm": arm, "tile_m": T, "n": s.n, "pairs": s.pairs, "woken": woken,
                "m_tiles": ntiles, "us": round(us, 1), "pairs_per_s": round(s.pairs / (us * 1e-6), 1),
                "staged_packed_GBps": round(staged / (us * 1e-6) / 1e9, 1),
                "roofline_us": round(max(t_hbm, t_tc), 1), "bound": "hbm" if t_hbm >= t_tc else "tensor",
                "frac": round(max(t_hbm, t_tc) / us, 4),
                "decode_lookups_per_clk_per_sm": round(lookups / (us * 1e-6) / 152 / 2.07e9, 2),
                "peak_source": peak_src, "peak_kind": "burst"}))
        clk = clocks.stop()
        for line in lines:
            print(json.dumps({**line, "clocks": clk}), flush=True)
        del d, y32, w_dense
        torch.cuda.empty_cache()


def run_step_latency(args):
    """Latency of one whole decode step through tq_moe_forward (route + tile
    map clearing y32, [copy,] arm, combine) at the V4 up shape across token
    counts, under the default selection, the measured policy and the grouped
    pin, each at the native m-tile: the call captured in a CUDA graph and
    replayed after an L2 flush (median), clocks sampled."""
    import torch
    import trellis_quantized_moe_sort_gb300 as tq
    from trellis_quantized_moe_sort_gb300 import build as b
    b.build()
    torch.cuda.set_device(0)
    tq.tq_init(0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    base = moe_inputs.make_problem("v4_decode_n32")
    packed = _cuda(torch, base.packed)
    lut = _cuda(torch, base.lut_bits.view(np.int16))
    names = {tq.ARM_AUTO: "auto", tq.ARM_MEASURED: "measured", tq.ARM_GROUPED: "grouped"}
    for n in [int(v) for v in args.gate_ns.split(",")]:
        prob = moe_inputs.make_problem("v4_decode_n32", n=n, with_packed=False)
        s = prob.shape
        x, ids, w = _cuda(torch, prob.x_bits.view(np.int16)), _cuda(torch, prob.topk_ids), _cuda(torch, prob.topk_w)
        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        row = {"n": n, "native_tile_m": tq.tq_native_tile_m(n, s.top_k, s.E)}
        for pin in (tq.ARM_AUTO, tq.ARM_MEASURED, tq.ARM_GROUPED):
            ws = torch.empty(max(256, tq.tq_moe_workspace_size(n, s.top_k, s.E, s.K, s.N, tq.TILE_NATIVE)),
                             dtype=torch.uint8, device="cuda")
            y = torch.empty((n, s.N), dtype=torch.bfloat16, device="cuda")
            stream = torch.cuda.Stream()
            call = lambda: tq.tq_moe_forward(x, packed, lut, ids, w, tile_m=tq.TILE_NATIVE, pin=pin, workspace=ws,
                                             y=y)
            with torch.cuda.stream(stream):
                _, arm = call()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call()
            ts = []
            for _ in range(args.steps):
                flush.zero_()
                torch.cuda.synchronize()
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b_.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b_) * 1e3)
            us = float(np.median(ts))
            # host cost of one eager call (binding + C ABI + launches), the GPU kept busy
            with torch.cuda.stream(stream):
                flush.zero_()
                h0 = time.perf_counter()
                for _ in range(20):
                    call()
                host_us = (time.perf_counter() - h0) / 20 * 1e6
            stream.synchronize()
            row[names[pin]] = {"arm": {1: "gemv", 2: "grouped"}[arm], "us_per_step": round(us, 1),
                               "tokens_per_s": round(n / (us * 1e-6), 1), "host_us_per_call": round(host_us, 1)}
        row["clocks"] = clocks.stop()
        code, where = tq.tq_device_error()
        if code:
            raise RuntimeError(f"device error {code} at {where} (n={n})")
        print(json.dumps(row), flush=True)


def run_gate_study(args):
    """GB300 gate study: both arms of the routed-expert product (grouped GEMM
    at TILE_M 16 and 128, per-pair GEMV) across token counts at the
    DeepSeek-V4 up shape, each kernel launch timed alone after an L2 flush.
    The GEMV is timed twice: tq_gemv (fp32 atomics into y32) and the
    one-launch arm of tq_moe_forward (bf16 y).  The tile-fill predicate's
    choice (TILE_M 16) is printed beside."""
    import torch
    import trellis_quantized_moe_sort_gb300 as tq
    from trellis_quantized_moe_sort_gb300 import build as b
    b.build()
    torch.cuda.set_device(0)
    tq.tq_init(0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    base = moe_inputs.make_problem("v4_decode_n32")
    packed = _cuda(torch, base.packed)
    lut = _cuda(torch, base.lut_bits.view(np.int16))
    ns = [int(v) for v in args.gate_ns.split(",")]
    for n in ns:
        prob = moe_inputs.make_problem("v4_decode_n32", n=n, with_packed=False)
        s = prob.shape
        x, ids, w = _cuda(torch, prob.x_bits.view(np.int16)), _cuda(torch, prob.topk_ids), _cuda(torch, prob.topk_w)
        y32 = torch.zeros((n, s.N), dtype=torch.float32, device="cuda")

        graphed = []

        def timed(fn):
            """Median device time of fn, replayed from a CUDA graph (so host
            launch gaps do not count) when capture works, else launched."""
            fn()
            torch.cuda.synchronize()
            run = fn
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn()
                run = g.replay
                graphed.append(True)
            except Exception:
                torch.cuda.synchronize()
                graphed.append(False)
            ts = []
            for _ in range(args.steps):
                flush.zero_()
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                run()
                b_.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b_) * 1e3)
            return float(np.median(ts))

        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        row = {"n": n, "pairs": n * s.top_k, "woken": int(len(np.unique(prob.topk_ids))),
               "pairs_per_woken_expert": round(tq.tq_pairs_per_woken_expert(n, s.top_k, s.E), 3),
               "predicate_arm_T16": {1: "gemv", 2: "grouped"}[tq.tq_select_arm(n, s.top_k, s.E, 16)],
               "measured_policy_arm": {1: "gemv", 2: "grouped"}[tq.tq_select_arm(n, s.top_k, s.E, 16,
                                                                                  tq.ARM_MEASURED)]}
        row["gemv_us"] = round(timed(lambda: tq.tq_gemv(x, packed, lut, ids, w, y32)), 1)
        # the GEMV arm as tq_moe_forward runs it: one launch that sums each
        # token's pairs in registers and writes bf16 y
        ws = torch.empty(max(256, tq.tq_moe_workspace_size(n, s.top_k, s.E, s.K, s.N, 16)), dtype=torch.uint8,
                         device="cuda")
        y = torch.empty((n, s.N), dtype=torch.bfloat16, device="cuda")
        row["gemv_forward_us"] = round(timed(lambda: tq.tq_moe_forward(x, packed, lut, ids, w, tile_m=16,
                                                                         pin=tq.ARM_GEMV, workspace=ws, y=y)), 1)
        for T in (16, 128):
            _, offsets, sp = tq.tq_route(ids, s.E)
            cap = tq.tq_tile_map_capacity(n, s.top_k, s.E, T)
            tiles, nt = tq.tq_build_tile_map(offsets, T, cap)

            counts = torch.empty(s.E, dtype=torch.int32, device="cuda")
            # the activation layout tq_moe_forward uses at this m-tile
            lay = tq.X_TOKENS if T <= tq.GATHER_MAX_TILE_M else tq.X_PAIR_SORTED
            xs = None if lay == tq.X_TOKENS else tq.tq_gather_rows(x, sp, s.top_k)

            def whole():  # route + tile map (+ pair-sorted copy) + grouped GEMM: the arm's device work
                tq.tq_route(ids, s.E, counts, offsets, sp)
                tq.tq_build_tile_map(offsets, T, cap, tiles, nt)
                if xs is not None:
                    tq.tq_gather_rows(x, sp, s.top_k, xs)
                tq.tq_grouped_gemm(x if xs is None else xs, packed, lut, sp, w, tiles, nt, s.top_k, T, y32,
                                   x_layout=lay)
            row[f"grouped_T{T}_us"] = round(timed(whole), 1)
        row["clocks"] = clocks.stop()
        code, where = tq.tq_device_error()
        if code:
            raise RuntimeError(f"device error {code} at {where} (n={n})")
        best = min(("gemv", row["gemv_us"]), ("grouped", row["grouped_T16_us"]), key=lambda kv: kv[1])
        row["faster_arm"] = best[0]
        row["grouped_over_gemv"] = round(row["gemv_us"] / row["grouped_T16_us"], 3)
        row["cuda_graphs"] = all(graphed)
        print(json.dumps(row), flush=True)


def run_mlp_sweep(args):
    """Whole SwiGLU expert MLP (tq_moe_mlp_forward) per workload: median time
    per call after an L2 flush, with the lookup count it decodes."""
    import torch
    import trellis_quantized_moe_sort_gb300 as tq
    from trellis_quantized_moe_sort_gb300 import build as b
    b.build()
    torch.cuda.set_device(0)
    tq.tq_init(0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    rate = tq.tq_probe_lut_rate(8)
    for name in moe_inputs.MLP_WORKLOADS:
        prob = moe_inputs.make_mlp_problem(name)
        c = lambda a: _cuda(torch, a)
        x, ids, w = c(prob.x_bits.view(np.int16)), c(prob.topk_ids), c(prob.topk_w)
        pgu, lgu = c(prob.packed_gu), c(prob.lut_gu.view(np.int16))
        pd, ld = c(prob.packed_down), c(prob.lut_down.view(np.int16))
        T = args.tile_m if prob.n <= 1024 else 256
        ws = torch.empty(tq.tq_moe_mlp_workspace_size(prob.n, prob.top_k, prob.E, prob.H, prob.I, T),
                         dtype=torch.uint8, device="cuda")
        y = torch.empty((prob.n, prob.H), dtype=torch.bfloat16, device="cuda")
        for pin in ([tq.ARM_GROUPED, tq.ARM_GEMV] if prob.n <= 128 else [tq.ARM_GROUPED]):
            clocks = ClockSampler(0)
            clocks.start()
            time.sleep(0.3)
            line = _mlp_time(args, tq, torch, flush, rate, name, prob, T, pin,
                             lambda: tq.tq_moe_mlp_forward(x, pgu, lgu, pd, ld, ids, w, tile_m=T, pin=pin,
                                                           workspace=ws, y=y))
            print(json.dumps({**line, "clocks": clocks.stop()}), flush=True)
        del x, pgu, pd, ws, y
        torch.cuda.empty_cache()


def _mlp_time(args, tq, torch, flush, rate, name, prob, T, pin, call):
    """One line of --mlp-sweep (returned): the call's median time after an
    L2 flush; the tensor roofline against the burst peak (each call timed on
    its own)."""
    call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b_.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b_) * 1e3)
    code, where = tq.tq_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where} ({name})")
    counts = np.bincount(prob.topk_ids.reshape(-1), minlength=prob.E)
    tiles = int(np.sum(-(-counts // T)))
    units = tiles if pin == tq.ARM_GROUPED else prob.n * prob.top_k   # decodes per matrix
    lookups = units * (2 * prob.I * prob.H + prob.H * prob.I)
    us = float(np.median(ts))
    ceiling = lookups / (152 * rate * 2.07e9) * 1e6
    flops = 2 * prob.n * prob.top_k * 3 * prob.H * prob.I
    return ({"workload": name, "arm": {tq.ARM_GROUPED: "grouped", tq.ARM_GEMV: "gemv"}[pin],
                      "tile_m": T, "n": prob.n, "pairs": prob.n * prob.top_k, "m_tiles": tiles,
                      "us_per_call": round(us, 1), "tokens_per_s": round(prob.n / (us * 1e-6), 1),
                      "lookups": lookups, "decode_ceiling_us": round(ceiling, 1),
                      "decode_frac": round(ceiling / us, 3),
                      "tensor_roofline_us": round(flops / (measured_peaks()[1] * 1e12) * 1e6, 1)})


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(moe_inputs.WORKLOADS))
    ap.add_argument("--tile-m", type=int, default=16)
    ap.add_argument("--weight-sets", type=int, default=NUM_WEIGHT_SETS,
                    help="independent weight sets cycled over the steps (defeats L2 reuse)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false",
                    help="skip the 8192-token prefill projections timed beside the headline")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--sweep", action="store_true",
                    help="per-workload table of both arms instead of the single bench line")
    ap.add_argument("--sweep-workloads", default="", help="comma-separated subset for --sweep")
    ap.add_argument("--sweep-tiles", default="16,128", help="TILE_M values for --sweep")
    ap.add_argument("--sweep-no-gemv", action="store_true", help="skip the GEMV arm in --sweep")
    ap.add_argument("--sweep-both-layouts", action="store_true",
                    help="time the grouped kernel on token rows (gathered in the kernel) and on the pair-sorted "
                         "copy at every TILE_M (default: the layout the whole-product calls use)")
    ap.add_argument("--sweep-dequant", action="store_true",
                    help="add the dequantize-materialize comparator (dense bf16 experts + the same grouped GEMM) to --sweep")
    ap.add_argument("--gate-study", action="store_true", help="both arms across token counts (V4 up shape)")
    ap.add_argument("--mlp-sweep", action="store_true", help="whole SwiGLU expert MLP per workload")
    ap.add_argument("--step-latency", action="store_true",
                    help="whole decode-step latency through tq_moe_forward across token counts (V4 up shape)")
    ap.add_argument("--gate-ns", default="1,2,4,8,9,16,32,64,128,256,512,682,683,1024")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes (read+write) per grouped launch, if captured for the current kernel source")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl" if args.impl == "ours" else "gloo")
        dist = tdist
    if args.sweep:
        run_sweep(args)
        return
    if args.gate_study:
        run_gate_study(args)
        return
    if args.mlp_sweep:
        run_mlp_sweep(args)
        return
    if args.step_latency:
        run_step_latency(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
