"""The multi-rank path of bench.py on CPU with world_size 2 over gloo: each rank runs its own
replica (weak scaling, no data-path collective); the job time is the slowest rank's, the value
counts every rank's units, and only rank 0 of the reference arm does any work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank                       # rank 1 is the slower replica
    total = bench.max_over_ranks(local_ms, world, "cpu")
    value = bench.job_throughput(2.0e12, 4, world, total, 1e12)
    out[rank] = (total, value)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 15.0               # every rank reports the slowest time
    # 2 ranks x 4 steps x 2 TFLOP in 15 ms
    assert out[0][1] == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_is_plain():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_throughput(1e9, 10, 1, 10.0, 1e9) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    class A:
        steps, warmup, workload = 1, 0, "dense"
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "_oracle_sample", lambda *a: called.append(a))
    bench.run_reference(A())
    assert not called and capsys.readouterr().out == ""
