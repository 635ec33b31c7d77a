"""The multi-GPU path of the benchmark, on CPU with gloo (world size 2).

The attention path has no exchange step (every (batch, head) is independent),
so N GPUs run N replicas and the benchmark only reduces its numbers across
ranks: the slowest rank's time (max) and the total work (sum). These tests
run that reduction in two real processes over gloo.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, ws = bench.dist_init("gloo")
    assert (r, ws) == (rank, world)
    times, units = bench.aggregate({"fwd_ms": 1.0 + rank, "dec_ms": 5.0 - rank},
                                   {"fwd_flops": 100.0 * (rank + 1)})
    bench.barrier()
    out[rank] = (times, units)
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_total_work():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        results = dict(out)
    for rank in range(world):
        times, units = results[rank]
        assert times == {"fwd_ms": 2.0, "dec_ms": 5.0}
        assert units == {"fwd_flops": 300.0}


def test_single_rank_is_identity():
    import bench

    times, units = bench.aggregate({"a": 1.5}, {"u": 7.0})
    assert times == {"a": 1.5} and units == {"u": 7.0}


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    """Under torchrun only rank 0 times the oracle; other ranks print nothing."""
    import bench

    monkeypatch.setattr(bench, "dist_init", lambda backend: (1, 2))
    bench.run_reference(type("A", (), {"steps": 1, "warmup": 3})())
    assert capsys.readouterr().out == ""
