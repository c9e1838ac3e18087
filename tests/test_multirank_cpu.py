"""The N-rank aggregation of bench.py on CPU: two gloo ranks, each timing its own replica.

Every rank processes the same number of units; the whole-job rate counts all ranks'
units against the slowest rank's time (the max over ranks), as bench.py reports it."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 * (rank + 1) + 0.25          # rank 1 is the slowest
        ms = bench.slowest_rank_ms(ms_local, world, "cpu")
        rate = bench.whole_job_rate(32, ms, world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_slowest_time_and_whole_job_rate(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for rank in range(world):
        got = json.load(open(tmp_path / f"rank{rank}.json"))
        assert got["ms"] == pytest.approx(20.25)
        assert got["rate"] == pytest.approx(32 * 2 / 0.02025)


def test_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(7.5, 1, "cpu") == 7.5
    assert bench.whole_job_rate(32, 7.5, 1) == pytest.approx(32 / 0.0075)
