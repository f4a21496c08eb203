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


def test_layer_work_counts_touched_adapters_once():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    L = wl.decode_step(0)
    w = bench.layer_work(L)
    e = 2
    assert w["touched"] == 3 and w["r_touched"] == 48
    assert w["step_bytes"] == (4096 * 4096 + 32 * 4096 * 2 + 48 * 8192) * e + 4 * 32
    assert w["step_flops"] == 2 * 32 * 4096 * 4096 + 2 * 32 * 16 * 8192
