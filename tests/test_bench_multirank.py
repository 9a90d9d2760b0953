"""bench.py's multi-GPU logic on CPU: world-size-2 gloo ranks, no GPU.

The decode path does not shard (replicas only), so the only multi-rank logic is the
whole-job timing: the maximum of the ranks' timed regions, and the throughput of all
ranks' bytes over it."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [3.0, 5.0][rank]                      # rank 1 is the slow replica
    ms = bench.job_time_ms(local, world, "cpu")
    out[rank] = ms
    dist.barrier()
    dist.destroy_process_group()


def test_job_time_is_max_over_ranks_and_throughput_sums_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 5.0
    import bench
    # 1 GB per rank in 5 ms on each of 2 ranks: 400 GB/s for the job
    assert bench.job_throughput(1e9, 5.0, 2) == pytest.approx(400.0)
    assert bench.job_time_ms(7.0, 1, "cpu") == 7.0
