"""Multi-rank logic of bench.py on the CPU (gloo, world size 2).

bench.py runs one replica batch per GPU; the job's time is the slowest rank's
and its throughput counts every rank's bytes.  Under torchrun only rank 0 of
the reference arm does work.  These tests exercise that logic with two CPU
processes; no GPU is touched.
"""

import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms_per_rank, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(ms_per_rank[rank], dist, torch.device("cpu"))
        q.put((rank, slowest, bench.job_throughput(world, 1e9, slowest)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ms = [0.110, 0.125]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, gbs in got:
        assert slowest == pytest.approx(0.125)
        # two ranks x 1 GB in the slowest rank's 0.125 ms
        assert gbs == pytest.approx(2 * 1e9 / 0.125e-3 / 1e9)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(0.5, None, None) == 0.5
    assert bench.job_throughput(1, 2e9, 1.0) == pytest.approx(2000.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) == 0
