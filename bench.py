#!/usr/bin/env python3
"""Throughput of the multi-LoRA linear layer on GB300; prints one JSON line on rank 0.

Default workload: the 7B-shaped decode stack (32 layers, 128 rows, 100 rank-16
adapters on q and v).  One step is one pass of the batch through the 32 layers;
a layer runs as four projections (fused q|k|v with the adapters, o, fused
gate|up, down), each one mlora_forward call through the C ABI (segment build,
shrink, base projection with the fused expand).  `value` is tokens/s per layer:
128 rows x 32 layers x K steps over the timed K steps.

Timing: inputs resident in HBM; the K timed steps are replayed from CUDA graphs
holding exactly those steps, bracketed by CUDA events on the launching stream,
with a device synchronisation on both sides and the maximum over ranks.  Every
thread block of the library's kernels appends a {start, end} globaltimer record
during the timed region (mlora_profile_stamps); the dominant kernel's launch
duration is the union of its blocks' intervals divided by its launches, so it
never exceeds the step.  The stack's weights (13 GB) exceed L2 many times over;
the smaller workloads rotate over enough copies to exceed twice the L2 size.

The same JSON line carries sub-objects for the decode step, the fragmented
decode batch and the prefill batch (each timed the same way), the merge, the
quantized base and the host-tier prefetch, the end-to-end figure (pinned host
inputs in, result out, every step) and the CPU oracle on a bounded sample.

  --impl ours       (default) the CUDA path through the C ABI
  --impl reference  the fp64 CPU oracle on the host cores, bounded per step
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); rank 0 prints the job total.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "tokens/s per multi-LoRA layer and % of HBM/tensor roofline on 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {"swapab_gemm_kernel": "heterogeneous_lora_gemm_gb300/csrc/tc.cu",
                  "prefill_gemm_kernel": "heterogeneous_lora_gemm_gb300/csrc/tc_prefill.cu"}
STAMP_SHRINK, STAMP_PROJECTION, STAMP_PREFILL = 0, 1, 2
KIND_NAMES = {STAMP_SHRINK: "shrink (swapab_gemm_kernel<true> or shrink_gemv_kernel)", STAMP_PROJECTION: "swapab_gemm_kernel<false>",
              STAMP_PREFILL: "prefill_gemm_kernel"}
SUB_WORKLOADS = {"decode_step": (20480, 64), "fragmented_decode": (8192, 32), "prefill": (256, 8)}
MAX_DECODE_T = 256   # the widest batch the decode kernels (swap-AB projection) take


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stack7b",
                    choices=["stack7b", "decode_step", "fragmented_decode", "prefill"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget of cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="skip the other workloads' sub-objects")
    ap.add_argument("--no-extras", action="store_true", help="skip merge / quantized / prefetch timings")
    ap.add_argument("--layers", type=int, default=wl.STACK7B_LAYERS, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# --------------------------------------------------------------------------- #
# distributed plumbing (host-side timing reduction only)
def dist_env():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_job(dist, elapsed_s: float, tokens: float):
    """Max time over ranks and total tokens over ranks (whole-job throughput)."""
    if dist is None:
        return elapsed_s, tokens
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    n = torch.tensor([tokens], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


# --------------------------------------------------------------------------- #
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """SM clocks, power and throttle reasons sampled every few milliseconds while the
    GPU works: NVML (read-only queries) in a thread, else nvidia-smi."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, uuid: str = "", interval_s: float = 0.002):
        self.dev, self.uuid, self.interval = device_index, uuid, interval_s
        self.rows, self.marks = [], {}
        self.nvml, self.handle, self.proc, self.thread = None, None, None, None
        self.stop = threading.Event()

    def _nvml_open(self):
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        found = False
        if self.uuid:
            n = ctypes.c_uint()
            nv.nvmlDeviceGetCount_v2(ctypes.byref(n))
            for i in range(n.value):
                hi = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(hi)) != 0:
                    continue
                buf = ctypes.create_string_buffer(96)
                if nv.nvmlDeviceGetUUID(hi, buf, 96) == 0 and self.uuid in buf.value.decode():
                    h, found = hi, True
                    break
        if not found and nv.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(h)) != 0:
            return False
        self.nvml, self.handle = nv, h
        return True

    def _loop(self):
        nv, h = self.nvml, self.handle
        mhz, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        while not self.stop.is_set():
            nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz))
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) != 0:
                nv.nvmlDeviceGetCurrentClocksThrottleReasons(h, ctypes.byref(rs))
            self.rows.append((time.perf_counter(), float(mhz.value), float(mx.value), mw.value / 1e3, int(rs.value)))
            time.sleep(self.interval)

    def __enter__(self):
        if self._nvml_open():
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        else:
            self.out = tempfile.NamedTemporaryFile("w+", delete=False, suffix=".csv")
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.dev}", "--query-gpu=clocks.sm,clocks.max.sm,power.draw,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=self.out, stderr=subprocess.DEVNULL)
            except OSError:
                self.proc = None
        time.sleep(0.05)
        return self

    def mark(self, name: str):
        self.marks[name] = time.perf_counter()

    def __exit__(self, *exc):
        self.stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            with open(self.out.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    try:
                        self.rows.append((0.0, float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3], 16)))
                    except (ValueError, IndexError):
                        continue
            os.unlink(self.out.name)

    def summary(self, start: str = "t0", stop: str = "t1"):
        src = "nvml" if self.nvml is not None else ("nvidia-smi" if self.proc is not None else "none")
        rows = self.rows
        if src == "nvml" and start in self.marks and stop in self.marks:
            rows = [r for r in rows if self.marks[start] <= r[0] <= self.marks[stop]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0, "source": src}
        reasons = set()
        for r in rows:
            for bit, name in self.REASONS.items():
                if r[4] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "power_w_max": max(r[3] for r in rows),
                "source": f"{src}, sampled during the timed region"}


def source_hash(rel: str) -> str:
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    return d.get("dram_bytes_per_launch")


def busy_union(rec: np.ndarray, kind: int) -> float:
    """Seconds during which at least one block of kernel `kind` was alive."""
    r = rec[rec[:, 2] == kind]
    if r.shape[0] == 0:
        return 0.0
    r = r[np.argsort(r[:, 0])]
    total, cur0, cur1 = 0, int(r[0, 0]), int(r[0, 1])
    for a, b in zip(r[1:, 0], r[1:, 1]):
        if a > cur1:
            total += cur1 - cur0
            cur0, cur1 = int(a), int(b)
        elif b > cur1:
            cur1 = int(b)
    total += cur1 - cur0
    return total / 1e9


# --------------------------------------------------------------------------- #
# algorithmic work: what the method must move or compute
def call_work(din: int, dout: int, T: int, row_adapter, ranks_of_slot, up_rows_of_slot=None):
    """Bytes and FLOPs of one forward and of its projection kernel.  ranks_of_slot[s] is the
    list of (rank, rows its Up reaches) of slot s's adapters (one per adapted module)."""
    e = 2
    touched = sorted(set(int(a) for a in row_adapter if 0 <= a < len(ranks_of_slot) and ranks_of_slot[a]))
    down_b = sum(r * din * e for s_ in touched for r, _ in ranks_of_slot[s_])
    up_b = sum(r * rows * e for s_ in touched for r, rows in ranks_of_slot[s_])
    lora_f = sum(2 * r * (din + rows) for a in row_adapter if 0 <= a < len(ranks_of_slot)
                 for r, rows in (ranks_of_slot[int(a)] or []))
    lora_up_f = sum(2 * r * rows for a in row_adapter if 0 <= a < len(ranks_of_slot)
                    for r, rows in (ranks_of_slot[int(a)] or []))
    base = dout * din * e + T * din * e + T * dout * e
    return {"step_bytes": base + down_b + up_b + 4 * T, "proj_bytes": base + up_b,
            "step_flops": 2 * T * din * dout + lora_f, "proj_flops": 2 * T * din * dout + lora_up_f,
            "touched": len(touched), "r_touched": sum(r for s_ in touched for r, _ in ranks_of_slot[s_])}


def layer_ranks(L: wl.LayerData):
    return [[(a.rank, L.dout)] if a is not None else [] for a in L.slot_list()]


# --------------------------------------------------------------------------- #
# device-resident workloads: a list of forward calls per step
class Call:
    def __init__(self, pool, X, W, ra, Y, work, launches, kind):
        self.pool, self.X, self.W, self.ra, self.Y = pool, X, W, ra, Y
        self.work, self.launches, self.kind = work, launches, kind

    def __call__(self, stream):
        self.pool.forward(self.X, self.W, self.ra, self.Y, stream=stream)


def build_stack(seed: int, dev, layers: int):
    """32 layers x (q|k|v, o, gate|up, down).  Layer 0 comes from the host generator
    (the oracle checks it); the others are drawn on the device with the same recipe."""
    import torch

    from heterogeneous_lora_gemm_gb300 import Pool
    from heterogeneous_lora_gemm_gb300.torch_io import make_fused_pool, to_device
    calls, host0 = [], []
    base_pools = {}
    for layer in range(layers):
        for g, (gname, din, mods) in enumerate(wl.STACK7B_GROUPS):
            if layer == 0:
                G = wl.stack7b_group(seed, 0, g)
                host0.append(G)
                X, W = to_device(G.X, "bf16"), to_device(G.W, "bf16")
                modules, ra_np = G.modules, G.row_adapter
                tenants = [[(to_device(a.down, "bf16"), to_device(a.up, "bf16"), a.scale) if a is not None else None
                            for a in row] for row in G.tenants]
            else:
                d = wl.stack7b_group_device(seed, layer, g, dev)
                X, W, modules, tenants, ra_np = d["X"], d["W"], d["modules"], d["tenants"], d["row_adapter"]
            dout = sum(n for _, n in modules)
            T = X.shape[0]
            if tenants:
                pool = make_fused_pool(din, modules, tenants, T)
                ra = torch.from_numpy(ra_np.astype(np.int32)).to(dev)
                ranks = [[(16, n) for (_, n), t in zip(modules, row) if t is not None] for row in tenants]
                launches = 2
            else:
                key = (din, dout)
                if key not in base_pools:
                    base_pools[key] = Pool(0, 0, 16, din, dout, "bf16", T)
                pool, ra, ranks, launches = base_pools[key], None, [], 1
            del tenants
            Y = torch.empty((T, dout), dtype=torch.bfloat16, device=dev)
            work = call_work(din, dout, T, ra_np if ra is not None else [], ranks)
            calls.append(Call(pool, X, W, ra, Y, work, launches, STAMP_PROJECTION))
    return calls, host0


def build_single(workload: str, seed: int, dev, l2: int):
    """One forward per step, rotating over enough device copies to exceed twice the L2."""
    import torch

    from heterogeneous_lora_gemm_gb300.torch_io import make_pool, to_device
    L = wl.by_name(workload, seed)
    work = call_work(L.din, L.dout, L.T, L.row_adapter, layer_ranks(L))
    per_copy = work["step_bytes"] + sum(a.down.nbytes + a.up.nbytes for a in L.adapters)
    copies = max(1, math.ceil(2 * l2 / per_copy))
    kind = STAMP_PREFILL if L.T > 256 else STAMP_PROJECTION
    calls = []
    for _ in range(copies):
        pool = make_pool(L)
        X, W = to_device(L.X, L.dtype), to_device(L.W, L.dtype)
        ra = torch.from_numpy(L.row_adapter.astype(np.int32)).to(dev)
        Y = torch.empty((L.T, L.dout), dtype=X.dtype, device=dev)
        calls.append(Call(pool, X, W, ra, Y, work, 2 if L.max_slots > 0 else 1, kind))
    return calls, L, copies


# --------------------------------------------------------------------------- #
def timed_steps(calls, per_step: int, steps: int, warmup: int, stream, dev, clocks=None, group: int = 256):
    """Times exactly `steps` steps (a step = per_step consecutive calls of `calls`, which
    rotate) from CUDA graphs, after `warmup` untimed steps; kernel blocks stamp records."""
    import torch
    pools = {id(c.pool): c.pool for c in calls}
    n = len(calls)
    period = n // per_step                       # steps before the rotation repeats
    big = max(period, (group // period) * period) if per_step == 1 else 1
    cap = 0
    with torch.cuda.stream(stream):
        for c in calls:                          # one eager pass (also checks every call)
            c(stream)
    torch.cuda.synchronize(dev)

    def capture(n_steps, record):
        for p in pools.values():
            if record is not None:
                p.profile_stamps(record, cap)
            else:
                p.profile_stamps(None, 0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps * per_step):
                calls[i % n](stream)
        return g

    # records: one per block; size for the timed steps from a measured eager step
    probe = torch.zeros(4 + 4 * 4, dtype=torch.int64, device=dev)
    for p in pools.values():
        p.profile_stamps(probe, 4)
    with torch.cuda.stream(stream):
        for i in range(per_step):
            calls[i % n](stream)
    torch.cuda.synchronize(dev)
    blocks_per_step = int(probe[0].item())
    cap = int(blocks_per_step * steps * 1.25) + 1024
    rec = torch.zeros(4 + 4 * cap, dtype=torch.int64, device=dev)
    q, r = divmod(steps, big)
    g_big = capture(big, rec) if q > 0 else None
    g_rest = capture(r, rec) if r > 0 else None
    for p in pools.values():
        p.profile_stamps(None, 0)
    # warm-up: the same graphs' shape, W steps (at least 3)
    wq, wr = divmod(max(warmup, 3), big)
    g_wbig = g_big if g_big is not None else capture(big, rec)
    g_wrest = capture(wr, rec) if wr > 0 else None
    for p in pools.values():                     # later eager calls record nothing
        p.profile_stamps(None, 0)
    with torch.cuda.stream(stream):
        for _ in range(wq):
            g_wbig.replay()
        if g_wrest is not None:
            g_wrest.replay()
    torch.cuda.synchronize(dev)
    rec.zero_()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.mark("t0")
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(q):
            g_big.replay()
        if g_rest is not None:
            g_rest.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.mark("t1")
    elapsed = ev0.elapsed_time(ev1) / 1e3
    count = int(rec[0].item())
    records = rec[4:4 + 4 * min(count, cap)].view(-1, 4).cpu().numpy().astype(np.int64) if count else None
    return {"elapsed": elapsed, "records": records, "records_complete": count <= cap, "graph_steps": big,
            "replays": q + (1 if r else 0)}


def kernel_roofline(t, kind, launches, bytes_per_launch, flops_per_launch, peaks, peak_src, bound, workload):
    if t["records"] is None or not t["records_complete"]:
        return None
    busy = busy_union(t["records"], kind)
    if busy <= 0:
        return None
    launch_s = busy / launches
    name = "prefill_gemm_kernel" if kind == STAMP_PREFILL else "swapab_gemm_kernel"
    if bound == "tensor":
        peak = peaks["bf16_tflops"]
        achieved = flops_per_launch / launch_s / 1e12
        unit, pk = "TFLOP/s", "bf16_tflops (burst: the kernel's own blocks are timed)"
    else:
        peak = peaks["hbm_gbs"]
        achieved = bytes_per_launch / launch_s / 1e9
        unit, pk = "GB/s", "hbm_gbs"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": profiled_traffic(name, workload), "kernel": KIND_NAMES[kind], "launch_us": launch_s * 1e6,
            "launches": int(launches), "busy_share_of_timed_region": busy / t["elapsed"],
            "algorithmic_bytes_per_launch": int(bytes_per_launch),
            "algorithmic_flops_per_launch": int(flops_per_launch),
            "peak_source": f"{pk} of {'MEASURED_PEAKS.json' if peak_src == 'measured' else 'the fallback'}",
            "duration": "union of the kernel's block intervals (device globaltimer, every block of every launch "
                        "in the timed region) / launches",
            "frac_of_8tbs": (bytes_per_launch / launch_s / 8e12) if bound == "hbm" else None}


def other_kernels(t, kinds):
    if t["records"] is None:
        return None
    return {KIND_NAMES[k]: {"busy_share_of_timed_region": busy_union(t["records"], k) / t["elapsed"]}
            for k in kinds}


# --------------------------------------------------------------------------- #
def run_stack(args, dist, dev, stream, peaks, peak_src, clocks):
    import torch
    calls, host0 = build_stack(args.seed, dev, args.layers)
    per_step = len(calls)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t = timed_steps(calls, per_step, args.steps, args.warmup, stream, dev, clocks=clocks)
    T = wl.STACK7B_T
    tokens = args.steps * args.layers * T
    job_elapsed, job_tokens = reduce_job(dist, t["elapsed"], tokens)
    layer_calls = calls[:len(wl.STACK7B_GROUPS)]
    layer_step_bytes = sum(c.work["step_bytes"] for c in layer_calls)
    layer_flops = sum(c.work["step_flops"] for c in layer_calls)
    proj_bytes = sum(c.work["proj_bytes"] for c in layer_calls) / len(layer_calls)
    proj_flops = sum(c.work["proj_flops"] for c in layer_calls) / len(layer_calls)
    launches = args.steps * len(calls)           # one projection launch per call
    roof = kernel_roofline(t, STAMP_PROJECTION, launches, proj_bytes, proj_flops, peaks, peak_src, "hbm", "stack7b")
    layer_s = job_elapsed / (args.steps * args.layers)
    step_roof_s = max(layer_step_bytes / (peaks["hbm_gbs"] * 1e9), layer_flops / (peaks["bf16_tflops"] * 1e12))
    gpu_launches = args.steps * sum(c.launches for c in calls)

    # per-projection breakdown: each group's 32 calls (one per layer) back to back
    breakdown = {}
    for g, (gname, din, mods) in enumerate(wl.STACK7B_GROUPS):
        gcalls = calls[g::len(wl.STACK7B_GROUPS)]
        tg = timed_steps(gcalls, 1, 4 * len(gcalls), 2 * len(gcalls), stream, dev, group=len(gcalls))
        w = gcalls[0].work
        us = tg["elapsed"] / (4 * len(gcalls)) * 1e6
        r = kernel_roofline(tg, STAMP_PROJECTION, 4 * len(gcalls), w["proj_bytes"], w["proj_flops"], peaks,
                            peak_src, "hbm", "stack7b")
        breakdown[gname] = {"us_per_forward": us, "step_bytes": w["step_bytes"],
                            "frac_of_hbm": w["step_bytes"] / (us * 1e-6) / (peaks["hbm_gbs"] * 1e9),
                            "projection_launch_us": r["launch_us"] if r else None,
                            "projection_frac": r["frac"] if r else None,
                            "launches_per_forward": gcalls[0].launches}

    e2e = None
    if not args.no_e2e:
        e2e = stack_e2e(calls, args, dist, stream, dev)
    out = {
        "value": job_tokens / job_elapsed, "ms_per_step": job_elapsed / args.steps * 1e3,
        "dtype": "bf16",
        "config": {"workload": "stack7b", "layers": args.layers, "T": T,
                   "projections_per_layer": "q|k|v 4096->12288 (adapters on q and v), o 4096->4096, "
                                            "gate|up 4096->22016, down 11008->4096",
                   "adapters": "100 rank-16 tenants, q and v of a tenant in one slot", "seed": args.seed},
        "timing": {"step": f"one pass of {T} rows through {args.layers} layers ({per_step} mlora_forward calls)",
                   "replay": f"CUDA graph of {t['graph_steps']} step(s), {t['replays']} replays = exactly "
                             f"{args.steps} steps",
                   "l2": "13 GB of weights per step, far beyond the 129 MB L2 (no flush needed)",
                   "us_per_layer": layer_s * 1e6},
        "roofline": roof,
        "other_kernels": other_kernels(t, (STAMP_SHRINK,)),
        "step_roofline": {"frac": step_roof_s / layer_s, "bytes_per_layer": int(layer_step_bytes),
                          "flops_per_layer": int(layer_flops), "peak_hbm_gbs": peaks["hbm_gbs"]},
        "per_projection": breakdown,
        "e2e": e2e, "gpu_launches": int(gpu_launches),
    }
    return out, calls, host0


def stack_e2e(calls, args, dist, stream, dev):
    """The stack through the public API end to end: every step copies the batch's input
    activations (the first projection's X) and the row map in from pinned host memory,
    runs the 32 layers, and reads the last projection's output back."""
    import torch
    first = calls[0]
    last = calls[-1]
    hX = first.X.cpu().pin_memory()
    ra_src = first.ra if first.ra is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    hra = ra_src.cpu().pin_memory()
    hY = torch.empty(last.Y.shape, dtype=last.Y.dtype).pin_memory()

    def step():
        first.X.copy_(hX, non_blocking=True)
        ra_src.copy_(hra, non_blocking=True)
        for c in calls:
            c(stream)
        hY.copy_(last.Y, non_blocking=True)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            g.replay()
    torch.cuda.synchronize(dev)
    barrier(dist)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            g.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    el, tok = reduce_job(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * args.layers * wl.STACK7B_T)
    h2d = hX.numel() * hX.element_size() + hra.numel() * 4
    d2h = hY.numel() * hY.element_size()
    return {"value": tok / el, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": el / args.steps * 1e3, "steps": args.steps,
            "copies": "pinned host X of the first projection and the row map in, the last projection's Y out, "
                      "on the forward stream, inside the timed graph replays"}


def run_sub(name: str, args, stream, dev, l2, peaks, peak_src, steps=None, warmup=None, clocks=None):
    import torch
    calls, L, copies = build_single(name, args.seed, dev, l2)
    steps = steps or SUB_WORKLOADS[name][0]
    warmup = warmup or SUB_WORKLOADS[name][1]
    t = timed_steps(calls, 1, steps, warmup, stream, dev, clocks=clocks)
    w = calls[0].work
    step_s = t["elapsed"] / steps
    bound = "tensor" if calls[0].kind == STAMP_PREFILL else "hbm"
    roof = kernel_roofline(t, calls[0].kind, steps, w["proj_bytes"], w["proj_flops"], peaks, peak_src, bound, name)
    step_roof_s = max(w["step_bytes"] / (peaks["hbm_gbs"] * 1e9), w["step_flops"] / (peaks["bf16_tflops"] * 1e12))
    out = {"value": L.T / step_s, "unit": "tokens/s", "ms_per_step": step_s * 1e3, "steps": steps,
           "warmup": warmup,
           "config": {"workload": name, "T": L.T, "din": L.din, "dout": L.dout, "adapters_touched": w["touched"],
                      "rank_touched_sum": w["r_touched"], "seed": args.seed},
           "timing": {"replay": f"CUDA graph of {t['graph_steps']} forwards, exactly {steps} timed",
                      "l2": f"inputs rotate over {copies} device copies (working set > 2x L2 of {l2 >> 20} MiB), "
                            "no flush"},
           "roofline": roof,
           "other_kernels": other_kernels(t, (STAMP_SHRINK,)),
           "step_roofline": {"frac": step_roof_s / step_s, "bytes": int(w["step_bytes"]),
                             "flops": int(w["step_flops"])},
           "gpu_launches": int(steps * calls[0].launches)}
    return out, calls, L


# --------------------------------------------------------------------------- #
# the next rows, timed on the decode step's shapes: merge / un-merge, quantized base,
# host-tier prefetch
def run_extras(calls, L, stream, dev, peaks):
    import torch

    from heterogeneous_lora_gemm_gb300 import Pool, mlora
    from heterogeneous_lora_gemm_gb300.torch_io import to_device
    out = {}
    c0 = calls[0]
    a0 = L.adapters[0]
    Wm = [c.W.clone() for c in calls[:max(2, min(len(calls), 8))]]
    reps = 20
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def t_us(fn, n):
        with torch.cuda.stream(stream):
            fn(0)
            m0.record(stream)
            for k in range(n):
                fn(k)
            m1.record(stream)
        torch.cuda.synchronize(dev)
        return m0.elapsed_time(m1) * 1e3 / n

    m_us = t_us(lambda k: c0.pool.merge(Wm[k % len(Wm)], a0.slot, stream=stream), reps * len(Wm))
    um_us = t_us(lambda k: c0.pool.unmerge(Wm[k % len(Wm)], a0.slot, stream=stream), reps * len(Wm))
    m_bytes = 2 * L.dout * L.din * 2 + a0.rank * (L.din + L.dout) * 2
    out["merge"] = {"us_per_merge": m_us, "us_per_unmerge": um_us, "rank": a0.rank, "dout": L.dout, "din": L.din,
                    "achieved_gbs": m_bytes / m_us / 1e3, "frac": m_bytes / m_us / 1e3 / peaks["hbm_gbs"],
                    "unmerge_frac": m_bytes / um_us / 1e3 / peaks["hbm_gbs"], "copies": len(Wm)}
    del Wm

    Wf = c0.W.float()
    qscale = (Wf.abs().amax(1) / 127).contiguous()
    Wq0 = torch.round(Wf / qscale[:, None]).clamp(-127, 127).to(torch.int8)
    del Wf
    qn = 16
    Wqs = [Wq0.clone() for _ in range(qn)]
    scs = [qscale.clone() for _ in range(qn)]
    scratch = torch.empty_like(c0.W)
    dq_us = t_us(lambda k: mlora.mlora_dequantize(Wqs[k % qn].data_ptr(), scs[k % qn].data_ptr(), L.dout, L.din,
                                                 mlora.MLORA_BF16, scratch.data_ptr(), stream.cuda_stream), 20 * qn)
    fq_us = t_us(lambda k: c0.pool.forward_quantized(c0.X, Wqs[k % qn], scs[k % qn], scratch, c0.ra, c0.Y,
                                                     stream=stream), 20 * qn)
    mq_us = t_us(lambda k: c0.pool.merge_quantized(Wqs[k % qn], scs[k % qn], a0.slot, stream=stream), 20 * qn)
    n_w = L.dout * L.din
    fwd_us = t_us(lambda k: c0.pool.forward(c0.X, calls[k % len(calls)].W, c0.ra, c0.Y, stream=stream),
                  20 * len(calls))
    fq_bytes = n_w + 4 * L.dout + L.T * (L.din + L.dout) * 2 + sum(a.rank for a in L.adapters) * L.dout * 2
    out["quantized"] = {"dequantize_us": dq_us, "dequantize_gbs": (3 * n_w + 4 * L.dout) / dq_us / 1e3,
                        "forward_quantized_us": fq_us, "forward_bf16_us": fwd_us,
                        "forward_quantized_frac": fq_bytes / fq_us / 1e3 / peaks["hbm_gbs"],
                        "merge_quantized_us": mq_us,
                        "merge_quantized_gbs": (2 * n_w + 8 * L.dout) / mq_us / 1e3,
                        "base": "int8 codes, fp32 scale per output row; the decode projection reads the codes",
                        "copies": qn}
    # the same comparison at wider batches (the decode step's adapters, its row map
    # repeated): the codes path moves half of W's bytes and restores W in every stage
    qpool = Pool(L.max_slots, sum((a.rank + 7) // 8 * 8 for a in L.adapters), L.max_rank, L.din, L.dout, "bf16",
                 MAX_DECODE_T)
    for a in L.adapters:
        qpool.load(a.slot, to_device(a.down, "bf16"), to_device(a.up, "bf16"), a.scale)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    by_t = {}
    for T in (32, 128, 192, MAX_DECODE_T):
        Xt = torch.randn((T, L.din), generator=gen, device=dev).to(torch.bfloat16)
        rat = torch.from_numpy(np.resize(L.row_adapter, T).astype(np.int32)).to(dev)
        Yt = torch.empty((T, L.dout), dtype=torch.bfloat16, device=dev)
        # (NVTX ranges name these launches for a profiler: codes_T<T>, bf16_T<T>)
        torch.cuda.nvtx.range_push(f"codes_T{T}")
        q_us = t_us(lambda k: qpool.forward_quantized(Xt, Wqs[k % qn], scs[k % qn], scratch, rat, Yt, stream=stream),
                    20 * qn)
        torch.cuda.nvtx.range_pop()
        torch.cuda.nvtx.range_push(f"bf16_T{T}")
        b_us = t_us(lambda k: qpool.forward(Xt, calls[k % len(calls)].W, rat, Yt, stream=stream), 20 * len(calls))
        torch.cuda.nvtx.range_pop()
        by_t[str(T)] = {"forward_quantized_us": q_us, "forward_bf16_us": b_us}
    qpool.close()
    out["quantized"]["by_tokens"] = by_t
    out["quantized"]["by_tokens_note"] = ("eager back-to-back forwards over 4096 x 4096, the decode step's three "
                                          "rank-16 adapters with its row map repeated to T rows")
    del Wqs, scs, scratch

    # NF4 base (4-bit codes, fp32 absmax per row and 64 columns, the NormalFloat codebook)
    cb = wl.nf4_codebook()
    packed, absmax = wl.nf4_random_base(0, L.dout, L.din)
    Q4 = [torch.from_numpy(packed).to(dev) for _ in range(qn)]
    A4 = [torch.from_numpy(absmax).to(dev) for _ in range(qn)]
    f4_us = t_us(lambda k: c0.pool.forward_nf4(c0.X, Q4[k % qn], A4[k % qn], cb, None, c0.ra, c0.Y, stream=stream),
                 20 * qn)
    Wr = torch.empty_like(c0.W)
    d4_us = t_us(lambda k: mlora.mlora_dequantize_nf4(Q4[k % qn].data_ptr(), A4[k % qn].data_ptr(), cb, L.dout, L.din,
                                                       mlora.MLORA_BF16, Wr.data_ptr(), stream.cuda_stream), 20 * qn)
    m4_us = t_us(lambda k: c0.pool.merge_nf4(Q4[k % qn], A4[k % qn], cb, a0.slot, stream=stream), 20 * qn)
    f4_bytes = n_w // 2 + n_w // 64 * 4 + L.T * (L.din + L.dout) * 2 + sum(a.rank for a in L.adapters) * L.dout * 2
    out["nf4"] = {"forward_nf4_us": f4_us, "forward_nf4_frac": f4_bytes / f4_us / 1e3 / peaks["hbm_gbs"],
                  "dequantize_nf4_us": d4_us, "dequantize_nf4_gbs": (n_w // 2 + n_w // 16 + 2 * n_w) / d4_us / 1e3,
                  "merge_nf4_us": m4_us, "merge_nf4_gbs": (n_w + n_w // 8) / m4_us / 1e3,
                  "base": "4-bit codes, fp32 absmax per row and 64 columns, NormalFloat codebook; "
                          "the decode projection reads the codes", "copies": qn}
    del Q4, A4, Wr

    src = L.adapters[0]
    ppool = Pool(L.max_slots + 1, sum((a.rank + 7) // 8 * 8 for a in L.adapters) + 3 * 16,
                 max(L.max_rank, 16), L.din, L.dout, "bf16", max(L.T, 1))
    for a in L.adapters:
        ppool.load(a.slot, to_device(a.down, "bf16"), to_device(a.up, "bf16"), a.scale)
    for hid in (0, 1):
        ppool.host_add(hid, to_device(src.down, "bf16", "cpu"), to_device(src.up, "bf16", "cpu"), src.scale)
    spare = L.max_slots
    pf_us = t_us(lambda k: ppool.prefetch(spare, k & 1, stream=stream), 64)
    pf_bytes = (src.rank + 7) // 8 * 8 * (L.din + L.dout) * 2
    plain = t_us(lambda k: ppool.forward(c0.X, c0.W, c0.ra, c0.Y, stream=stream), 64)

    def with_pf(k):
        ppool.prefetch(spare, k & 1, stream=stream)
        ppool.forward(c0.X, c0.W, c0.ra, c0.Y, stream=stream)
    both = t_us(with_pf, 64)
    out["prefetch"] = {"us_per_prefetch": pf_us, "bytes": int(pf_bytes), "h2d_gbs": pf_bytes / pf_us / 1e3,
                       "step_us_eager": plain, "step_us_eager_with_prefetch": both,
                       "note": "eager launches (no graph), one copy of the decode step: not a bench step time"}
    ppool.close()
    return out


# --------------------------------------------------------------------------- #
# the oracle on the host cores (cpu_baseline leg and reference arm)
def oracle_layer0_stack(seed: int, host0=None):
    """Layer 0 of the stack on the host, in the oracle's terms, per input group."""
    import oracle
    groups = host0 if host0 is not None else [wl.stack7b_group(seed, 0, g) for g in range(len(wl.STACK7B_GROUPS))]
    out = []
    f64 = wl.bf16_bits_to_f64
    for G in groups:
        tenants = [[None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in row]
                   for row in G.tenants]
        out.append({"G": G, "X": f64(G.X), "W": f64(G.W), "tenants": tenants})
    return out


def oracle_stack_rows(og, rows):
    import oracle
    if og["tenants"]:
        return oracle.forward_modules(og["X"], og["W"], og["G"].row_adapter, og["G"].modules, og["tenants"],
                                      rows=rows)
    return oracle.forward(og["X"], og["W"], None, [], rows=rows)


def oracle_single(workload: str, seed: int):
    import oracle
    L = wl.by_name(workload, seed)
    ads = [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in L.slot_list()]
    return L, ads


def time_oracle_rows(fn, T: int, budget_s: float, rng, min_rows: int):
    """Rows per second of `fn(rows)` over seeded row samples for about budget_s seconds."""
    t0 = time.perf_counter()
    fn(np.array([0], np.int64))
    row_s = max(time.perf_counter() - t0, 1e-6)
    per_call = int(max(min(T, min_rows), min(T, 2.0 / row_s)))
    done, t0 = 0, time.perf_counter()
    while True:
        rows = np.sort(rng.choice(T, size=per_call, replace=False)).astype(np.int64)
        fn(rows)
        done += per_call
        if time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0, per_call


def cpu_baseline(args, calls, host0, L_single):
    """The oracle as it stands, on the host cores, over a bounded sample of the timed
    workload; it also checks the GPU's output rows it computes (spot check)."""
    import oracle

    from heterogeneous_lora_gemm_gb300.torch_io import to_f64
    rng = np.random.default_rng(args.seed)
    cores = oracle.threads()
    spot = {}
    if args.workload == "stack7b":
        ogs = oracle_layer0_stack(args.seed, host0)
        per_group = []
        for g, og in enumerate(ogs):
            rows = np.array([0, wl.STACK7B_T - 1], np.int64)
            got = to_f64(calls[g].Y)[rows]
            want = oracle_stack_rows(og, rows)
            spot[og["G"].name] = bool(np.all(np.abs(got - want) <= 1e-2 * (1 + np.abs(want))))
            done, el, per = time_oracle_rows(lambda r, og=og: oracle_stack_rows(og, r), wl.STACK7B_T,
                                             args.cpu_seconds / len(ogs), rng, cores)
            per_group.append(el / done)
        value = 1.0 / sum(per_group)    # rows through one layer (its four projections) per second
        sample = (f"seeded row samples of layer 0's four projections ({args.cpu_seconds:.0f} s), fp64 per-row "
                  "loop; tokens/s per layer = 1 / sum of the per-row times")
    else:
        L, ads = L_single
        rows = np.array([0, L.T - 1], np.int64)
        got = to_f64(calls[0].Y)[rows]
        want = oracle.forward(L.X_f64, L.W_f64, L.row_adapter, ads, rows=rows)
        spot[L.name] = bool(np.all(np.abs(got - want) <= 1e-2 * (1 + np.abs(want))))
        done, el, per = time_oracle_rows(lambda r: oracle.forward(L.X_f64, L.W_f64, L.row_adapter, ads, rows=r),
                                         L.T, args.cpu_seconds, rng, cores)
        value = done / el
        sample = f"{done} seeded rows of {L.name} ({per} per call, {el:.1f} s), fp64 per-row loop"
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
            "spot_check": spot}


def config_of(workload: str, seed: int, layers: int = wl.STACK7B_LAYERS):
    if workload == "stack7b":
        return {"workload": "stack7b", "layers": layers, "T": wl.STACK7B_T,
                "projections_per_layer": "q|k|v 4096->12288 (adapters on q and v), o 4096->4096, "
                                         "gate|up 4096->22016, down 11008->4096",
                "adapters": "100 rank-16 tenants, q and v of a tenant in one slot", "seed": seed}
    L = wl.by_name(workload, seed)
    return {"workload": workload, "T": L.T, "din": L.din, "dout": L.dout}


def run_reference(args):
    """The oracle timed as the reference arm: K timed steps of a bounded row sample each."""
    import oracle
    cores = oracle.threads()
    rng = np.random.default_rng(args.seed)
    if args.workload == "stack7b":
        ogs = oracle_layer0_stack(args.seed)
        fns = [lambda r, og=og: oracle_stack_rows(og, r) for og in ogs]
        T = wl.STACK7B_T
        per_step = min(T, cores)
        desc = f"{per_step} seeded rows through layer 0's four projections per step"
    else:
        L, ads = oracle_single(args.workload, args.seed)
        fns = [lambda r: oracle.forward(L.X_f64, L.W_f64, L.row_adapter, ads, rows=r)]
        T = L.T
        per_step = min(T, cores)
        desc = f"{per_step} seeded rows of {L.name} per step"
    samples = [np.sort(rng.choice(T, size=per_step, replace=False)).astype(np.int64)
               for _ in range(min(args.steps, 64))]
    for i in range(args.warmup):
        for fn in fns:
            fn(samples[i % len(samples)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        for fn in fns:
            fn(samples[i % len(samples)])
    el = time.perf_counter() - t0
    value = args.steps * per_step / el      # rows through one layer per second
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(args.workload, args.seed, args.layers),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": desc + ", fp64 per-row loop on the host cores (rank 0 only)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------------- #
def run_ours(args, dist, rank, local):
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    uuid = str(getattr(props, "uuid", "") or "")
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    with ClockSampler(local, uuid) as clk:
        if args.workload == "stack7b":
            head, calls, host0 = run_stack(args, dist, dev, stream, peaks, peak_src, clk)
            L_single = None
        else:
            sub, calls, L = run_sub(args.workload, args, stream, dev, l2, peaks, peak_src, steps=args.steps,
                                    warmup=args.warmup, clocks=clk)
            el, tok = reduce_job(dist, sub["ms_per_step"] * args.steps / 1e3, args.steps * L.T)
            head = dict(sub)
            head["value"], head["ms_per_step"] = tok / el, el / args.steps * 1e3
            if args.workload == "decode_step" and not args.no_extras:
                head.update(run_extras(calls, L, stream, dev, peaks))
            head["dtype"] = L.dtype
            head["e2e"] = None
            host0, L_single = None, (L, None)
    clocks = clk.summary()
    out = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
           "config": dict(config_of(args.workload, args.seed, args.layers), parallelism=f"replicas x{args.gpus}")}
    for k in ("timing", "roofline", "other_kernels", "step_roofline", "per_projection", "e2e", "gpu_launches",
              "merge", "quantized", "nf4", "prefetch"):
        if k in head:
            out[k] = head[k]
    out["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        if L_single is not None:
            import oracle
            L = L_single[0]
            L_single = (L, [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale)
                            for a in L.slot_list()])
        out["cpu_baseline"] = cpu_baseline(args, calls, host0, L_single)
    else:
        out["cpu_baseline"] = None
    del calls
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    if args.workload == "stack7b" and not args.no_sub:
        subs = {}
        for name in SUB_WORKLOADS:
            s, scalls, sL = run_sub(name, args, stream, dev, l2, peaks, peak_src)
            if name == "decode_step" and not args.no_extras:
                out.update(run_extras(scalls, sL, stream, dev, peaks))
            subs[name] = s
            del scalls
            torch.cuda.empty_cache()
        out["sub_workloads"] = subs
    return out


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl ours needs a CUDA GPU")
    dist = init_dist(world, "nccl")
    out = run_ours(args, dist, rank, local)
    out["n_gpus"] = world if world > 1 else args.gpus
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
