"""The N>1 benchmark path on CPU: world-size-2 gloo ranks.  The rasterizer
does not shard (every rank renders its own independent image), so the only
cross-rank step is the timing aggregation: the job time is the slowest
rank's and the throughput counts every rank's steps.  The reference arm runs
on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [40.0, 55.0][rank]
    value, job_ms = bench.aggregate_replicas(local_ms, steps=10, world=world)
    q.put((rank, value, job_ms))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, value, job_ms in out:
        assert job_ms == 55.0                       # the slowest rank
        assert value == pytest.approx(2 * 10 / 0.055)  # all ranks' steps


def test_single_rank_needs_no_process_group():
    import bench
    value, job_ms = bench.aggregate_replicas(20.0, steps=4, world=1)
    assert job_ms == 20.0 and value == pytest.approx(200.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload = "small_64x64_1k"
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(Args()) == 0
