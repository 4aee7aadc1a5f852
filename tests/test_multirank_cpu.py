"""The host logic of bench.py's multi-GPU (replica) mode on two gloo ranks on
the CPU: the slowest rank's time is the step time, throughput counts every
rank's tokens, the timing barrier holds, and ranks route different batches."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        assert env == (ws, rank, rank)
        bench.barrier(ws)
        ms_local = 2.0 + rank  # rank 1 is the slow one
        ms, value = bench.aggregate(ms_local, 4096, ws, "cpu")
        out[rank] = (ms, value, bench.rank_batch_seed(rank))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        ms, value, seed = res[r]
        assert ms == 3.0  # max over ranks
        assert value == pytest.approx(2 * 4096 / 3.0e-3)
    assert res[0][2] != res[1][2]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.aggregate(2.5, 100, 1, "cpu") == (2.5, 100 / 2.5e-3)
