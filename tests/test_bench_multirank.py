"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1 (the
GPU run uses the same functions over NCCL).  Every rank ends with the slowest
rank's time, the job rate counts every rank's units, and the reference arm
runs on rank 0 only."""
import argparse
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        local_ms = [3.0, 5.0][rank]  # rank 1 is the slower one
        ms = b.max_over_ranks(local_ms, dist, torch.device("cpu"))
        q.put((rank, ms, b.job_rate(32768, world, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == 5.0, (rank, ms)
        assert rate == pytest.approx(2 * 32768 / 5e-3)


def test_single_process_needs_no_group():
    b = _bench()
    assert b.max_over_ranks(4.0, None, torch.device("cpu")) == 4.0
    assert b.job_rate(100, 1, 2.0) == pytest.approx(5e4)


def test_reference_arm_other_ranks_exit_without_work():
    b = _bench()
    args = argparse.Namespace(warmup=3, steps=1, gpus=2)
    assert b.run_reference(args, 2, 1) == 0
