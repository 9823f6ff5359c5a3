"""The multi-GPU bench path is independent replicas (the layer is not sharded across
GPUs here): each rank times its own layer, the job's step time is the slowest
rank's, and throughput counts every rank's tokens.  Checked with two gloo ranks on
the CPU."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    bench.barrier(world)
    step_ms = 1.5 + rank                      # rank 1 is the slower replica
    slowest = bench.max_over_ranks(world, step_ms)
    out.put((rank, slowest, bench.job_tokens_per_s(world, 512, slowest)))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_take_slowest_rank_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == 2.5
        assert value == pytest.approx(2 * 512 / 2.5e-3)
