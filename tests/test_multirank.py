"""Multi-rank path of bench.py (one replica of the workload per rank, no
data-path collective), exercised with two gloo ranks on the CPU: the job time
is the slowest rank's, the job throughput counts every replica, and the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, _ = bench.dist_env()
        ms = 1.0 + 0.5 * rank                       # rank 1 is the slow replica
        ms_max = bench.max_over_ranks(ms, got_ws, torch.device("cpu"))
        value = bench.job_throughput(1e12, got_ws, ms_max)
        ref_ret = bench.run_reference(None) if got_rank != 0 else None
        q.put((got_rank, got_ws, ms_max, value, ref_ret))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got_ws, ms_max, value, ref_ret in out:
        assert got_ws == 2
        assert ms_max == pytest.approx(1.5)          # max over ranks, on every rank
        assert value == pytest.approx(2 * 1e12 / 1.5e-3 / 1e12)
        if rank == 1:
            assert ref_ret == 0                       # non-zero ranks do no reference work


def test_single_rank_is_identity():
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5
    assert bench.job_throughput(2e12, 1, 2.0) == pytest.approx(1000.0)
