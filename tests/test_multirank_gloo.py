"""CPU (gloo, world size 2) checks of the multi-rank host logic of bench.py.

Each rank runs an independent replica of the workload (the indexer's rows
are independent; there is no collective on the data path).  The only
cross-rank step is the timing reduction: whole-job units are summed and the
slowest rank's time is taken.
"""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units, secs = bench.aggregate(1000.0 * (rank + 1), 0.5 + rank)
    results[rank] = (units, secs)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_sums_units_and_takes_slowest_rank():
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    for r in range(world):
        assert results[r] == (3000.0, 1.5)


def test_aggregate_without_process_group_is_identity():
    import bench
    assert bench.aggregate(7.0, 2.0) == (7.0, 2.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1"])) == 0
    assert capsys.readouterr().out == ""
