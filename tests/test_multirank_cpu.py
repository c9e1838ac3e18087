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


# ------------------------------------------------------------ sharded calibration
def _calib_rank_main(rank, world, port, out_dir):
    """Each rank calibrates its share of the batches; the ranges are all-gathered
    and merged.  The library's two kernels are replaced by CPU stand-ins built from
    the oracle, so this checks the exchange and the merge order, not the kernels
    (those are checked on the GPU)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import workloads as W
    from int8_head_kv_gb300 import fa3 as F
    from oracle import fa3_oracle as O

    def fake_calibrate(x, ratio, mn, mx, workspace=None, stream=None):
        lo, hi = O.calibrate_batch(x.float().numpy(), ratio)
        O.accumulate(mn.numpy(), mx.numpy(), lo, hi)

    def fake_merge(mins, maxs, mn, mx, stream=None):
        for r in range(mins.shape[0]):
            O.accumulate(mn.numpy(), mx.numpy(), mins[r].numpy(), maxs[r].numpy())

    F.calibrate_perhead = fake_calibrate
    F.range_merge = fake_merge
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.mla_tiny()
        batches = W.mla_inputs(w).calib_q                       # 3 batches over 2 ranks: 2 + 1
        mine = [torch.from_numpy(b).to(torch.bfloat16) for k, b in enumerate(batches) if k % world == rank]
        mn = torch.full((w.H,), float("inf"))
        mx = torch.full((w.H,), float("-inf"))
        F.calibrate_perhead_sharded(mine, w.ratio, mn, mx)
        np.save(os.path.join(out_dir, f"calib{rank}.npy"), np.stack([mn.numpy(), mx.numpy()]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sharded_calibration_equals_one_process(tmp_path):
    import numpy as np
    sys.path.insert(0, ROOT)
    import workloads as W
    from oracle import fa3_oracle as O
    world = 2
    mp.spawn(_calib_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    w = W.mla_tiny()
    omn, omx = O.calibrate(W.mla_inputs(w).calib_q, w.ratio)
    for rank in range(world):
        got = np.load(tmp_path / f"calib{rank}.npy")
        assert np.array_equal(got[0].view(np.uint32), omn.view(np.uint32))
        assert np.array_equal(got[1].view(np.uint32), omx.view(np.uint32))
