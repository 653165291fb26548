"""The bench's multi-GPU path (independent replicas, one per GPU) on the CPU: two gloo ranks
run the same reduction the bench runs over NCCL (the slowest rank's times) and the whole-job
throughput rule.  No GPU and no data-path collective: replicas share only these scalars."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 + r ms for the blend, 30 - r for the full prefill, r for the e2e wall
        mx = bench.max_over_ranks([10.0 + rank, 30.0 - rank, float(rank), 1.0 + 0.5 * rank], world)
        dist.barrier()
        out[rank] = mx
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_with_gloo(world):
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    expect = [10.0 + world - 1, 30.0, float(world - 1), 1.0 + 0.5 * (world - 1)]
    assert [out[r] for r in range(world)] == [expect] * world


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]


def test_job_throughput_is_weak_scaling():
    # 3200 tokens per rank, slowest rank 11.4 ms: the job's rate counts every rank's tokens
    assert bench.job_throughput(3200, 1, 11.4) == pytest.approx(3200 / 0.0114)
    assert bench.job_throughput(3200, 8, 11.4) == pytest.approx(8 * 3200 / 0.0114)
