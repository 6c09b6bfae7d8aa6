"""Replicas across ranks (the benchmark's multi-GPU mode) on CPU with gloo,
world size 2: no data exchange, timing reduced with a max over ranks."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 1.0 + rank                     # rank 1 is the slower replica
    m = bench.reduce_max_over_ranks(ms)
    v = bench.replica_throughput(61385, world, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_timing_is_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == 2.0 and out[1][0] == 2.0
    assert out[0][1] == pytest.approx(2 * 61385 / 2e-3)


def test_single_process_identity():
    import bench
    assert bench.reduce_max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(100, 1, 1.0) == pytest.approx(1e5)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    bench.reference_arm(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert capsys.readouterr().out == ""
