#!/usr/bin/env python3
"""Throughput of the multi-LoRA linear layer on GB300; prints one JSON line on rank 0.

A step is one mlora_forward over one batch of the workload (segment build,
shrink, base projection with the fused expand), inputs resident in HBM.  The
default workload is the 32-token decode step (4096 -> 4096, adapters 20/8/4,
rank 16).  Small workloads rotate through enough copies of (W, X, Y, adapter
pool) that the working set is at least twice the L2 size, so every step streams
its weights from HBM.  Steps are replayed from a CUDA graph of at least 256
forwards.  The `e2e` figure adds, every step, the copy of X and the row map from
pinned host memory and the copy of Y back, on two copy streams pipelined with the
forwards (the next step's inputs go in and the previous step's output comes back
while a forward runs).

  --impl ours       (default) the CUDA path through the C ABI
  --impl reference  the fp64 CPU oracle on the host cores, bounded per step
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); rank 0 prints the job total.
"""
from __future__ import annotations

import argparse
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
# the projection kernel of each workload (the dominant kernel) and the file that holds it
KERNEL_SOURCES = {"swapab_gemm_kernel": "heterogeneous_lora_gemm_gb300/csrc/tc.cu",
                  "prefill_gemm_kernel": "heterogeneous_lora_gemm_gb300/csrc/tc_prefill.cu"}


def dominant_kernel(workload: str) -> str:
    return "prefill_gemm_kernel" if workload == "prefill" else "swapab_gemm_kernel"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_step",
                    choices=["decode_step", "fragmented_decode", "prefill", "stack7b", "worked_example"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget of cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------- #
# distributed plumbing (host-side timing reduction only)
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


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
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, interval_ms: int = 20):
        self.dev = device_index
        self.interval = interval_ms
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", delete=False, suffix=".csv")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", f"-lms", str(self.interval)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_load: float):
        if self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                                 "active": parts[4], "hw": parts[5], "hw_th": parts[6], "sw_th": parts[7],
                                 "sw_pc": parts[8]})
                except ValueError:
                    continue
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 0.5 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                              ("sw_th", "sw_thermal_slowdown"), ("sw_pc", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows)}


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


def multi_module_timing(seed: int, dev, stream, reps: int = 64):
    """q and v of one 7B-shaped layer in one launch -- a fused q|v projection whose
    slots each hold a tenant's q and v adapters -- against the two projections
    launched one after the other, on the same rows (the q rows' tenant mapping)."""
    import torch

    from heterogeneous_lora_gemm_gb300 import Pool
    from tests.gpu_harness import make_pool, to_device
    from tests.tolerance import within
    Lq, Lv = wl.stack7b_projection(seed, 0, "q"), wl.stack7b_projection(seed, 0, "v")
    T, din, dout = Lq.T, Lq.din, Lq.dout
    ra = torch.from_numpy(Lq.row_adapter.astype(np.int32)).to(dev)
    X = to_device(Lq.X, "bf16")
    qa, va = {a.slot: a for a in Lq.adapters}, {a.slot: a for a in Lv.adapters}
    budget = sum(-(-a.rank // 16) * 16 for a in Lq.adapters + Lv.adapters)
    fpool = Pool(Lq.max_slots, budget, 64, din, 2 * dout, "bf16", T)
    for s_ in range(Lq.max_slots):
        mods = []
        for off, ad in ((0, qa.get(s_)), (dout, va.get(s_))):
            mods.append((off, dout, to_device(ad.down, "bf16"), to_device(ad.up, "bf16"), ad.scale) if ad
                        else (off, dout, None, None, 0.0))
        fpool.load_modules(s_, mods)
    qpool, vpool = make_pool(Lq), make_pool(Lv)
    copies = 3   # W of the pair: 64 MiB per copy, rotated
    Wq = [to_device(Lq.W, "bf16") for _ in range(copies)]
    Wv = [to_device(Lv.W, "bf16") for _ in range(copies)]
    Wqv = [torch.cat([a, b], 0) for a, b in zip(Wq, Wv)]
    Yqv = torch.empty((T, 2 * dout), dtype=torch.bfloat16, device=dev)
    Yq, Yv = torch.empty((T, dout), dtype=torch.bfloat16, device=dev), torch.empty_like(Yqv[:, :dout])

    def fused(k):
        fpool.forward(X, Wqv[k % copies], ra, Yqv, stream=stream)

    def apart(k):
        qpool.forward(X, Wq[k % copies], ra, Yq, stream=stream)
        vpool.forward(X, Wv[k % copies], ra, Yv, stream=stream)

    out = {}
    for name, fn in (("fused_qv_us", fused), ("separate_q_plus_v_us", apart)):
        with torch.cuda.stream(stream):
            for k in range(8):
                fn(k)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(reps):
                fn(k)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            for _ in range(4):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = e0.elapsed_time(e1) * 1e3 / (4 * reps)
    got = torch.cat([Yq, Yv], 1).to(torch.float64).cpu().numpy()
    out["agree"] = bool(within(Yqv.to(torch.float64).cpu().numpy(), got, "bf16").all())
    out.update({"T": T, "tenants": len(qa), "ranks": "16 (q) + 16 (v) per tenant"})
    for pl in (fpool, qpool, vpool):
        pl.close()
    return out


# --------------------------------------------------------------------------- #
# workload bookkeeping# --------------------------------------------------------------------------- #
# workload bookkeeping
def layer_work(layer: wl.LayerData):
    """Algorithmic bytes and FLOPs of one forward and of its projection kernel."""
    e = 2 if layer.dtype == "bf16" else 4
    T, din, dout = layer.T, layer.din, layer.dout
    slots = layer.slot_list()
    ra = layer.row_adapter
    touched = sorted(set(int(a) for a in ra if 0 <= a < layer.max_slots and slots[a] is not None))
    r_touched = sum(slots[a].rank for a in touched)
    lora_rows_r = sum(slots[int(a)].rank for a in ra if 0 <= a < layer.max_slots and slots[int(a)] is not None)
    w_bytes, x_bytes, y_bytes = dout * din * e, T * din * e, T * dout * e
    step_bytes = w_bytes + x_bytes + y_bytes + r_touched * (din + dout) * e + 4 * T
    proj_bytes = w_bytes + x_bytes + y_bytes + r_touched * dout * e
    step_flops = 2 * T * din * dout + 2 * lora_rows_r * (din + dout)
    proj_flops = 2 * T * din * dout + 2 * lora_rows_r * dout
    return {"step_bytes": step_bytes, "proj_bytes": proj_bytes, "step_flops": step_flops, "proj_flops": proj_flops,
            "touched": len(touched), "r_touched": r_touched}


def layers_for(workload: str, seed: int):
    if workload == "stack7b":
        out = []
        for layer in range(wl.STACK7B_LAYERS):
            for m in wl.STACK7B_MODULES:
                out.append(wl.stack7b_projection(seed, layer, m[0]))
        return out
    return [wl.by_name(workload, seed)]


# --------------------------------------------------------------------------- #
def run_ours(args, dist, rank, local):
    import torch

    from heterogeneous_lora_gemm_gb300 import mlora
    from tests.gpu_harness import make_pool, to_device

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    peaks, peak_src = load_peaks()

    # ---- device-resident copies of the workload
    if args.workload == "stack7b":
        base_layers = None
        t0 = time.time()
        units = []
        for layer in range(wl.STACK7B_LAYERS):
            for m in wl.STACK7B_MODULES:
                L = wl.stack7b_projection(args.seed, layer, m[0])
                units.append(L)
        layers = units
        copies = 1
    else:
        layers = layers_for(args.workload, args.seed)
        per_copy = sum(layer_work(L)["step_bytes"] + sum(a.down.nbytes + a.up.nbytes for a in L.adapters)
                       for L in layers)
        copies = max(1, math.ceil(2 * l2 / per_copy))
    items = []
    for c in range(copies):
        for L in layers:
            pool = make_pool(L)
            X = to_device(L.X, L.dtype)
            W = to_device(L.W, L.dtype)
            ra = torch.from_numpy(L.row_adapter.astype(np.int32)).to(dev)
            Y = torch.empty((L.T, L.dout), dtype=X.dtype, device=dev)
            items.append({"layer": L, "pool": pool, "X": X, "W": W, "ra": ra, "Y": Y})
    if args.workload == "stack7b":
        for it in items:   # the generator's payloads are no longer needed on the host
            it["layer"] = wl.LayerData(it["layer"].name, it["layer"].dtype, it["layer"].din, it["layer"].dout,
                                       it["layer"].X[:1], it["layer"].W[:1], it["layer"].row_adapter,
                                       it["layer"].max_slots, [])
    n_items = len(items)
    works = [layer_work(layers[i % len(layers)]) for i in range(n_items)]
    tokens_per_item = [layers[i % len(layers)].T for i in range(n_items)]
    # one "step" is one layer call; stack7b counts 7 projections as one layer
    per_step_items = 7 if args.workload == "stack7b" else 1
    stream = torch.cuda.Stream(device=dev)

    def fwd(it):
        it["pool"].forward(it["X"], it["W"], it["ra"], it["Y"], stream=stream)

    # ---- warm-up (eager), then one graph per rotation
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3) * per_step_items):
            fwd(items[i % n_items])
    torch.cuda.synchronize(dev)
    # at least 256 forwards per replay, so that the gap between two graph launches
    # is spread over many steps
    passes = max(1, -(-256 // n_items))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(passes):
            for it in items:
                fwd(it)
    steps_per_replay = passes * n_items // per_step_items
    replays, rest = divmod(args.steps, steps_per_replay)
    with torch.cuda.stream(stream):      # a graph replays on the current stream
        graph.replay()
    torch.cuda.synchronize(dev)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(dist)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(replays):
                graph.replay()
            for i in range(rest * per_step_items):
                fwd(items[i % n_items])
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dist)
        elapsed = ev0.elapsed_time(ev1) / 1e3
        clocks = clk.summary(elapsed)
    # a forward is one projection launch, plus the shrink (which also builds the
    # segments) when its pool has adapter slots (every workload here loads them all)
    launches = [2 if it["layer"].max_slots > 0 else 1 for it in items]
    gpu_launches = args.steps * sum(launches[:per_step_items])
    tokens_rank = args.steps * tokens_per_item[0]
    job_elapsed, job_tokens = reduce_job(dist, elapsed, tokens_rank)

    # ---- projection-kernel duration from CUDA events around its launches (no work skipped)
    prof_pairs = []
    for it in items:
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)   # torch creates the CUDA event lazily, at its first record
        e_ev.record(stream)
        it["pool"].profile_events([s_ev], [e_ev])
        prof_pairs.append((s_ev, e_ev))
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph, stream=stream):
        for it in items:
            fwd(it)
    reps = max(1, min(replays, 400 // max(1, n_items) + 1))
    kern_ms = 0.0
    for _ in range(reps):
        with torch.cuda.stream(stream):
            pgraph.replay()
        stream.synchronize()
        kern_ms += sum(s.elapsed_time(e) for s, e in prof_pairs)
    for it in items:
        it["pool"].profile_events([], [])
    kern_avg_s = kern_ms / 1e3 / (reps * n_items)

    # ---- end to end: pinned host X and row map in, Y out, every step.  The copies run
    # on their own streams, pipelined with the forwards over the rotating device
    # copies: step i's inputs go in while step i-1 computes, its output comes back
    # while step i+1 computes.  Events order the reuse of each copy's buffers (its X
    # and row map are overwritten only after its last forward ran, its Y only after it
    # was read out).  Every step's copies are inside the timed region.
    e2e = None
    if not args.no_e2e:
        hosts = []
        for it in items:
            hosts.append({"X": it["X"].cpu().pin_memory(), "ra": it["ra"].cpu().pin_memory(),
                          "Y": torch.empty(it["Y"].shape, dtype=it["Y"].dtype).pin_memory()})
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        e_passes = max(1, -(-256 // n_items))   # at least 256 forwards per replay, as above

        # rounds of half the device copies: a round's inputs go in while the round
        # before computes, its outputs come back while the next one computes; one
        # event edge per round, so the forwards inside a round keep their
        # programmatic launch overlap
        rnd = max(1, n_items // 2)
        n_rounds = -(-n_items // rnd)

        def e2e_steps():
            ev_in, ev_fwd, ev_out = {}, {}, {}
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            for p_ in range(e_passes):
                for r in range(n_rounds):
                    idxs = list(range(r * rnd, min(n_items, (r + 1) * rnd)))
                    key = (p_, r)
                    prev = (p_ - 1, r) if p_ > 0 else None   # the round that last used these copies
                    if prev is not None:
                        s_in.wait_event(ev_fwd[prev])
                    with torch.cuda.stream(s_in):
                        for idx in idxs:
                            items[idx]["X"].copy_(hosts[idx]["X"], non_blocking=True)
                            items[idx]["ra"].copy_(hosts[idx]["ra"], non_blocking=True)
                    ev_in[key] = torch.cuda.Event()
                    ev_in[key].record(s_in)
                    stream.wait_event(ev_in[key])
                    if prev is not None:
                        stream.wait_event(ev_out[prev])
                    for idx in idxs:
                        fwd(items[idx])
                    ev_fwd[key] = torch.cuda.Event()
                    ev_fwd[key].record(stream)
                    s_out.wait_event(ev_fwd[key])
                    with torch.cuda.stream(s_out):
                        for idx in idxs:
                            hosts[idx]["Y"].copy_(items[idx]["Y"], non_blocking=True)
                    ev_out[key] = torch.cuda.Event()
                    ev_out[key].record(s_out)
            # join the copy streams back into the forward stream
            for s_side in (s_in, s_out):
                done = torch.cuda.Event()
                done.record(s_side)
                stream.wait_event(done)

        egraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(egraph, stream=stream):
            e2e_steps()
        with torch.cuda.stream(stream):
            egraph.replay()
        torch.cuda.synchronize(dev)
        barrier(dist)
        torch.cuda.synchronize(dev)
        e_steps_per_replay = e_passes * n_items // per_step_items
        e_replays = max(1, -(-args.steps // e_steps_per_replay))
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(e_replays):
                egraph.replay()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dist)
        e_steps = e_replays * e_steps_per_replay
        e_elapsed, e_tokens = reduce_job(dist, ev0.elapsed_time(ev1) / 1e3, e_steps * tokens_per_item[0])
        it0 = items[0]
        h2d = (it0["X"].numel() * it0["X"].element_size() + it0["ra"].numel() * 4) * per_step_items
        d2h = it0["Y"].numel() * it0["Y"].element_size() * per_step_items
        e2e = {"value": e_tokens / e_elapsed, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_elapsed / e_steps * 1e3, "steps": int(e_steps),
               "copies": "pinned host <-> device on two copy streams, in rounds of half the device copies, "
                         "pipelined with the forwards"}

    # ---- correctness spot check of the timed buffers (one row, oracle)
    spot = None
    if rank == 0 and args.workload != "stack7b":
        import oracle
        from tests.gpu_harness import to_f64
        L = items[0]["layer"]
        torch.cuda.synchronize(dev)
        fwd(items[0])
        torch.cuda.synchronize(dev)
        got = to_f64(items[0]["Y"])
        rows = np.array([0, L.T - 1], np.int64)
        ads = [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in L.slot_list()]
        want = oracle.forward(L.X_f64, L.W_f64, L.row_adapter, ads, rows=rows)
        from tests.tolerance import within
        spot = bool(within(got[rows], want, L.dtype).all())

    # ---- merge (W <- W + s Up Down) of the first adapter, on scratch copies of W: one
    # launch per merge, read + write of W plus the adapter's Up and Down
    merge = None
    L0m = items[0]["layer"]
    if L0m.max_slots > 0 and L0m.dtype == "bf16" and args.workload != "stack7b":
        a0 = layers[0].adapters[0]
        Wm = [torch.empty_like(items[i % n_items]["W"]).copy_(items[i % n_items]["W"]) for i in range(max(2, copies))]
        pool0 = items[0]["pool"]
        for w in Wm:
            pool0.merge(w, a0.slot, stream=stream)
        torch.cuda.synchronize(dev)
        mreps = 20
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for _ in range(mreps):
            for w in Wm:
                pool0.merge(w, a0.slot, stream=stream)
        m1.record(stream)
        torch.cuda.synchronize(dev)
        m_us = m0.elapsed_time(m1) * 1e3 / (mreps * len(Wm))
        # the un-merge (W <- W - s Up Down) on the same copies: the same kernel, sign flipped
        m0.record(stream)
        for _ in range(mreps):
            for w in Wm:
                pool0.unmerge(w, a0.slot, stream=stream)
        m1.record(stream)
        torch.cuda.synchronize(dev)
        um_us = m0.elapsed_time(m1) * 1e3 / (mreps * len(Wm))
        m_bytes = 2 * L0m.dout * L0m.din * 2 + a0.rank * (L0m.din + L0m.dout) * 2
        merge = {"us_per_merge": m_us, "rank": a0.rank, "dout": L0m.dout, "din": L0m.din,
                 "achieved_gbs": m_bytes / m_us / 1e3, "frac": m_bytes / m_us / 1e3 / peaks["hbm_gbs"],
                 "us_per_unmerge": um_us, "unmerge_frac": m_bytes / um_us / 1e3 / peaks["hbm_gbs"],
                 "copies": len(Wm)}
        del Wm

    # ---- quantized base (int8 codes x per-row scale): restoring W, the dynamic branch
    # over it (restore + forward), and the merge that re-quantizes (M031 §05)
    quantized = None
    if L0m.max_slots > 0 and L0m.dtype == "bf16" and args.workload not in ("stack7b", "prefill"):
        it0 = items[0]
        Wf = it0["W"].float()
        qscale = (Wf.abs().amax(1) / 127).contiguous()
        Wq0 = torch.round(Wf / qscale[:, None]).clamp(-127, 127).to(torch.int8)
        qcopies = 16   # 16 MiB of codes each: more than twice the L2
        Wqs = [Wq0.clone() for _ in range(qcopies)]
        scs = [qscale.clone() for _ in range(qcopies)]
        scratch = torch.empty_like(it0["W"])
        qreps = 20

        def q_time(fn):
            with torch.cuda.stream(stream):
                fn(0)
                p0.record(stream)
                for k in range(qreps * qcopies):
                    fn(k)
                p1.record(stream)
            torch.cuda.synchronize(dev)
            return p0.elapsed_time(p1) * 1e3 / (qreps * qcopies)

        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dq_us = q_time(lambda k: mlora.mlora_dequantize(Wqs[k % qcopies].data_ptr(), scs[k % qcopies].data_ptr(),
                                                       L0m.dout, L0m.din, mlora.MLORA_BF16, scratch.data_ptr(),
                                                       stream.cuda_stream))
        fq_us = q_time(lambda k: it0["pool"].forward_quantized(it0["X"], Wqs[k % qcopies], scs[k % qcopies], scratch,
                                                               it0["ra"], it0["Y"], stream=stream))
        mq_us = q_time(lambda k: it0["pool"].merge_quantized(Wqs[k % qcopies], scs[k % qcopies], 0, stream=stream))
        n_w = L0m.dout * L0m.din
        quantized = {"dequantize_us": dq_us, "dequantize_gbs": (3 * n_w + 4 * L0m.dout) / dq_us / 1e3,
                     "forward_quantized_us": fq_us, "merge_quantized_us": mq_us,
                     "merge_quantized_gbs": (2 * n_w + 8 * L0m.dout) / mq_us / 1e3,
                     "base": "int8 codes, fp32 scale per output row; the forward restores W (bf16) then runs"}

    # ---- q and v of a layer in one launch (fused projection) against two launches
    multi_module = None
    if args.workload == "stack7b" and rank == 0:
        multi_module = multi_module_timing(args.seed, dev, stream)

    # ---- host tier: a rank-16 adapter prefetched from pinned host memory into a spare
    # slot (M031 §06).  Cost of a prefetch alone (its H2D copies and the table update,
    # on the forward's stream), and the step time with one prefetch per step beside
    # the forwards of the timed workload's first copy.
    prefetch = None
    if L0m.max_slots > 0 and L0m.dtype == "bf16" and args.workload != "stack7b":
        from heterogeneous_lora_gemm_gb300 import Pool
        src = layers[0].adapters[0]
        ppool = Pool(L0m.max_slots + 1, sum((a.rank + 7) // 8 * 8 for a in layers[0].adapters) + 3 * 16,
                     max(L0m.max_rank, 16), L0m.din, L0m.dout, "bf16", max(L0m.T, 1))
        for a in layers[0].adapters:
            ppool.load(a.slot, to_device(a.down, "bf16"), to_device(a.up, "bf16"), a.scale)
        for hid in (0, 1):
            ppool.host_add(hid, to_device(src.down, "bf16", "cpu"), to_device(src.up, "bf16", "cpu"), src.scale)
        spare = L0m.max_slots
        it0 = items[0]
        reps = 64
        torch.cuda.synchronize(dev)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ppool.prefetch(spare, 0, stream=stream)
            p0.record(stream)
            for k in range(reps):
                ppool.prefetch(spare, k & 1, stream=stream)
            p1.record(stream)
        torch.cuda.synchronize(dev)
        pf_us = p0.elapsed_time(p1) * 1e3 / reps
        pf_bytes = (src.rank + 7) // 8 * 8 * (L0m.din + L0m.dout) * 2

        def steps_us(with_prefetch):
            with torch.cuda.stream(stream):
                for _ in range(8):
                    ppool.forward(it0["X"], it0["W"], it0["ra"], it0["Y"], stream=stream)
                p0.record(stream)
                for k in range(reps):
                    if with_prefetch:
                        ppool.prefetch(spare, k & 1, stream=stream)
                    ppool.forward(it0["X"], it0["W"], it0["ra"], it0["Y"], stream=stream)
                p1.record(stream)
            torch.cuda.synchronize(dev)
            return p0.elapsed_time(p1) * 1e3 / reps

        plain_us, with_us = steps_us(False), steps_us(True)
        prefetch = {"us_per_prefetch": pf_us, "bytes": int(pf_bytes), "h2d_gbs": pf_bytes / pf_us / 1e3,
                    "step_us_eager": plain_us, "step_us_eager_with_prefetch": with_us,
                    "note": "eager launches (no graph), one copy of the workload: not the bench's step time"}
        ppool.close()

    w0 = works[0]
    if per_step_items == 7:
        layer_bytes = sum(w["proj_bytes"] for w in works[:7])
        layer_step_bytes = sum(w["step_bytes"] for w in works[:7])
        layer_flops = sum(w["step_flops"] for w in works[:7])
        kernel_bytes = layer_bytes / 7
        kernel_flops = sum(w["proj_flops"] for w in works[:7]) / 7
    else:
        layer_step_bytes, layer_flops = w0["step_bytes"], w0["step_flops"]
        kernel_bytes, kernel_flops = w0["proj_bytes"], w0["proj_flops"]
    step_s = job_elapsed / args.steps
    tensor_bound = args.workload == "prefill"
    if tensor_bound:
        peak = peaks["bf16_tflops_sustained"]
        achieved = kernel_flops / kern_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak}
    else:
        peak = peaks["hbm_gbs"]
        achieved = kernel_bytes / kern_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak}
    roof.update({"peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                 "kernel": dominant_kernel(args.workload), "launch_us": kern_avg_s * 1e6,
                 "algorithmic_bytes_per_launch": int(kernel_bytes), "algorithmic_flops_per_launch": int(kernel_flops),
                 "traffic": profiled_traffic(dominant_kernel(args.workload), args.workload)})
    step_roof_s = max(layer_step_bytes / (peaks["hbm_gbs"] * 1e9), layer_flops / (peaks["bf16_tflops"] * 1e12))
    L0 = layers[0]
    out = {
        "metric": METRIC, "value": job_tokens / job_elapsed, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": L0.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "T": L0.T, "din": L0.din, "dout": L0.dout,
                   "adapters_touched": w0["touched"], "rank_touched_sum": w0["r_touched"],
                   "l2": f"inputs rotate over {copies} device copies (working set > 2x L2 of {l2 >> 20} MiB), no flush",
                   "replay": f"CUDA graph of {passes * n_items} forwards", "parallelism": f"replicas x{args.gpus}",
                   "seed": args.seed},
        "roofline": roof,
        "step_roofline": {"frac": step_roof_s / step_s, "bytes": int(layer_step_bytes), "flops": int(layer_flops)},
        "e2e": e2e, "gpu_launches": int(gpu_launches), "clocks": clocks, "spot_check": spot, "merge": merge, "prefetch": prefetch, "multi_module": multi_module,
        "quantized": quantized,
    }
    return out, L0


def cpu_baseline(workload: str, seed: int, budget_s: float, rows_cap: int = None):
    """The oracle as it stands, on the host cores, over a bounded sample of the workload."""
    import oracle
    if workload == "stack7b":
        L = wl.stack7b_projection(seed, 0, "q")
    else:
        L = wl.by_name(workload, seed)
    ads = [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in L.slot_list()]
    X, W = L.X_f64, L.W_f64
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    oracle.forward(X, W, L.row_adapter, ads, rows=np.array([0], np.int64))   # warm
    row_s = time.perf_counter() - t0
    per_call = int(max(1, min(L.T, 2.0 / max(row_s, 1e-6) * oracle.threads())))
    if rows_cap:
        per_call = min(per_call, rows_cap)
    done, t0 = 0, time.perf_counter()
    while True:
        rows = np.sort(rng.choice(L.T, size=per_call, replace=False)).astype(np.int64)
        oracle.forward(X, W, L.row_adapter, ads, rows=rows)
        done += per_call
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{done} rows of {L.name} ({per_call} seeded rows per call, {el:.1f} s, fp64 per-row loop)"}


def run_reference(args, rank):
    """The oracle timed as the reference arm: K timed steps of a bounded sample each."""
    import oracle
    L = wl.stack7b_projection(args.seed, 0, "q") if args.workload == "stack7b" else wl.by_name(args.workload, args.seed)
    ads = [None if a is None else oracle.OracleAdapter(a.down_f64, a.up_f64, a.scale) for a in L.slot_list()]
    X, W = L.X_f64, L.W_f64
    t0 = time.perf_counter()
    oracle.forward(X, W, L.row_adapter, ads, rows=np.array([0], np.int64))
    row_s = max(time.perf_counter() - t0, 1e-6)
    budget = 90.0       # whole timed run, seconds
    # at least one row per host core: the oracle's row loop runs them in parallel, so
    # a step costs about the same up to that many rows
    per_step = int(max(min(L.T, oracle.threads()),
                       min(L.T, budget / (args.steps + args.warmup) / row_s * oracle.threads())))
    rng = np.random.default_rng(args.seed)
    samples = [np.sort(rng.choice(L.T, size=per_step, replace=False)).astype(np.int64)
               for _ in range(min(args.steps, 64))]
    for i in range(args.warmup):
        oracle.forward(X, W, L.row_adapter, ads, rows=samples[i % len(samples)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.forward(X, W, L.row_adapter, ads, rows=samples[i % len(samples)])
    el = time.perf_counter() - t0
    value = args.steps * per_step / el
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "T": L.T, "din": L.din, "dout": L.dout,
                   "sample_rows_per_step": per_step, "parallelism": "rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{per_step} seeded rows of {L.name} per step, fp64 per-row loop"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank)), flush=True)
        return 0
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl ours needs a CUDA GPU")
    dist = init_dist(world, "nccl")
    out, L0 = run_ours(args, dist, rank, local)
    out["n_gpus"] = world if world > 1 else args.gpus
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(args.workload, args.seed, args.cpu_seconds)
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
