"""The benchmark's multi-rank path on CPU (gloo, world size 2): each rank
runs an independent replica; the only exchange is the max of the per-rank
step times, and whole-job throughput counts every rank's bytes."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                       # rank 1 is the slow one
    got = bench.max_over_ranks(ms, world, torch.device("cpu"))
    gbs = bench.aggregate_throughput(1e9, got, world)
    q.put((rank, got, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    # 2 ranks x 1 GB in 5 ms
    assert res[0][2] == pytest.approx(400.0)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    assert bench.aggregate_throughput(2e9, 1.0, 1) == pytest.approx(2000.0)


def test_child_env_runs_a_single_process_on_the_ranks_gpu(monkeypatch):
    """The extra workloads' child runs drop the launcher's rank variables and
    see only this rank's GPU (the rank's entry of CUDA_VISIBLE_DEVICES, else
    its local rank)."""
    import bench
    for k, v in (("RANK", "3"), ("WORLD_SIZE", "4"), ("LOCAL_RANK", "3"),
                 ("MASTER_ADDR", "127.0.0.1"), ("MASTER_PORT", "29500")):
        monkeypatch.setenv(k, v)
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    env = bench._child_env(3)
    assert not {"RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"} & set(env)
    assert env["CUDA_VISIBLE_DEVICES"] == "3"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "4,5,6,7")
    assert bench._child_env(1)["CUDA_VISIBLE_DEVICES"] == "5"
