"""Host-side logic of bench.py on CPU: the multi-rank reduction (max of the
per-rank step times, sum of the units) over a world-size-2 gloo group, and
the reference arm's rank handling. No GPU is touched."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # rank r: a step of (r + 1) ms over 100 * (r + 1) units
    ms, units = bench.aggregate(float(rank + 1), float(100 * (rank + 1)), world)
    bench._barrier(world)
    out[rank] = (ms, units)
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    for rank in range(world):
        ms, units = res[rank]
        assert ms == 2.0          # slowest rank's step time
        assert units == 300.0     # units of all ranks


def test_aggregate_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate(3.5, 42.0, 1) == (3.5, 42.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args(), 2, 1) is None


@pytest.mark.parametrize("argv", [["--warmup", "2"]])
def test_bench_rejects_fewer_than_three_warmup_steps(argv):
    sys.path.insert(0, ROOT)
    import bench

    with pytest.raises(SystemExit):
        bench.main(argv)


def test_bench_rejects_gpus_without_matching_world(monkeypatch):
    """--gpus N must match the launcher's WORLD_SIZE (one process per GPU)."""
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.delenv("WORLD_SIZE", raising=False)
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2", "--no-cpu-baseline"])
