"""Multi-process (gloo, CPU) checks of bench.py's replica plumbing.

Rows are independent, so N GPUs run N replicas with no collective on the data
path; the only cross-rank step is the host-side reduction of the timing (max of
the elapsed times, sum of the tokens).  These run world-size-2 process groups
on the CPU.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    t, n = bench.reduce_job(dist, elapsed_s=1.0 + rank, tokens=100.0 * (rank + 1))
    q.put((rank, t, n))
    dist.destroy_process_group()


def test_reduce_job_max_time_sum_tokens_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reduce_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    for _, t, n in got:
        assert t == 2.0 and n == 300.0


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_job(None, 0.5, 32.0) == (0.5, 32.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "1"]) == 0
    assert capsys.readouterr().out == ""


def test_call_work_counts_touched_adapters_once():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    L = wl.decode_step(0)
    w = bench.call_work(L.din, L.dout, L.T, L.row_adapter, bench.layer_ranks(L))
    e = 2
    assert w["touched"] == 3 and w["r_touched"] == 48
    assert w["step_bytes"] == (4096 * 4096 + 32 * 4096 * 2 + 48 * 8192) * e + 4 * 32
    assert w["proj_bytes"] == (4096 * 4096 + 32 * 4096 * 2 + 48 * 4096) * e
    assert w["step_flops"] == 2 * 32 * 4096 * 4096 + 2 * 32 * 16 * 8192


def test_call_work_of_the_fused_qkv_group():
    """q|k|v of a 7B-shaped layer: 100 tenants, each with a rank-16 q and a rank-16 v
    adapter whose Up reaches 4096 rows; every tenant is used."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    G = wl.stack7b_group(0, 0, 0)
    ranks = [[(a.rank, n) for (_, n), a in zip(G.modules, row) if a is not None] for row in G.tenants]
    w = bench.call_work(G.din, G.dout, G.T, G.row_adapter, ranks)
    e = 2
    assert w["touched"] == 100 and w["r_touched"] == 3200
    adapters = 100 * 2 * 16 * (4096 + 4096) * e
    assert w["step_bytes"] == (12288 * 4096 + 128 * 4096 + 128 * 12288) * e + adapters + 4 * 128
    assert w["proj_bytes"] == (12288 * 4096 + 128 * 4096 + 128 * 12288) * e + 100 * 2 * 16 * 4096 * e
    assert w["step_flops"] == 2 * 128 * 4096 * 12288 + 128 * 2 * 2 * 16 * (4096 + 4096)


def test_busy_union_of_block_records():
    """The kernel's busy time is the measure of the union of its blocks' intervals:
    overlapping blocks count once, gaps not at all, other kinds are ignored."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    rec = np.array([[100, 200, 1, 0], [150, 260, 1, 1], [300, 350, 1, 2], [310, 320, 1, 3],
                    [0, 1000, 0, 0], [400, 400, 1, 4]], np.int64)
    assert abs(bench.busy_union(rec, 1) - 210e-9) < 1e-15
    assert abs(bench.busy_union(rec, 0) - 1000e-9) < 1e-15
    assert bench.busy_union(rec, 2) == 0.0
