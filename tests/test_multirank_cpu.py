"""The benchmark's multi-process plumbing on CPU ranks (gloo, world size 2).

The block's shards all live on one GPU, so several GPUs run independent
replicas (weak scaling) and the only cross-rank steps are the barrier around
the timed region and the max over ranks of its duration.  Those host-side
steps are checked here with two CPU processes.
"""
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


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    try:
        assert bench.dist_env() == (ws, rank, rank)
        bench.barrier(ws)
        got = bench.max_over_ranks(10.0 + 5.0 * rank, ws)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ws = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(ws))
    assert res == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    import bench
    import synthetic_inputs as si
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 3, 3, 2

    assert bench.run_reference(A, si.WORKLOADS["C1"]) == 0
    assert capsys.readouterr().out == ""
