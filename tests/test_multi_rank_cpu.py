"""The bench's multi-GPU path on the CPU: requests are independent units, so a batch is
partitioned over the ranks with no collective on the data path.  Two and three gloo ranks
take their share of the Llama-70B-shaped batch (4 requests over a pool of 64 chunks),
and reduce the same scalars the bench reduces over NCCL: the slowest rank's times and the
tokens of every rank, which give the whole-job TTFT and tokens/s."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import harness as hz


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = hz.workload("llama70b")
        mine, partitioned = bench.shard_requests(len(spec.requests), world, rank)
        tokens = sum(spec.n_tokens(r) for r in mine)
        chunks = sorted({s.chunk for r in mine for s in spec.requests[r] if s.chunk >= 0})
        # rank r "took" 400 + 10 r ms for its blend, 3000 - r for its full prefill
        blend_ms, full_ms = bench.max_over_ranks([400.0 + 10 * rank, 3000.0 - rank], world)
        total = bench.sum_over_ranks(tokens, world)
        dist.barrier()
        out[rank] = {"mine": mine, "partitioned": partitioned, "tokens": tokens, "chunks": chunks,
                     "blend_ms": blend_ms, "full_ms": full_ms, "total": total}
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_requests_partitioned_over_gloo_ranks(world):
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    res = [out[r] for r in range(world)]
    spec = hz.workload("llama70b")
    # every request exactly once, none twice
    owned = sorted(q for r in res for q in r["mine"])
    assert owned == list(range(len(spec.requests)))
    assert all(r["partitioned"] for r in res)
    # each rank holds only the pooled chunks its own requests use
    for r in res:
        need = {s.chunk for q in r["mine"] for s in spec.requests[q] if s.chunk >= 0}
        assert set(r["chunks"]) == need
    # whole-job figures: the slowest rank's times, every rank's tokens
    T = sum(spec.n_tokens(q) for q in range(len(spec.requests)))
    for r in res:
        assert r["blend_ms"] == 400.0 + 10 * (world - 1) and r["full_ms"] == 3000.0
        assert r["total"] == T
    ttft = res[0]["blend_ms"]
    assert bench.job_throughput(res[0]["total"], ttft) == pytest.approx(T / (ttft * 1e-3))


def test_single_request_workload_runs_one_copy_per_rank():
    for rank in range(4):
        assert bench.shard_requests(1, 4, rank) == ([0], False)
    assert bench.shard_requests(4, 1, 0) == ([0, 1, 2, 3], False)


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.sum_over_ranks(8320, 1) == 8320
