"""Replica plumbing of bench.py (the path has no exchange step: N GPUs run N
independent replicas).  World-size-2 gloo ranks on the CPU check the barrier
and the max-over-ranks timing that the whole-job rate is computed from."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_defaults(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_algorithmic_bytes_of_the_headline_step():
    import bench
    import workloads
    host = workloads.make("drama3", 0)
    assert workloads.logit_bytes(host) == 128 * (4096 + 9 * 1024) * 2
    assert bench.algorithmic_bytes(host) == 3407872 + 1280 * 73
