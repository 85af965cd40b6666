"""The replica path of bench.py on CPU: two gloo ranks (no GPU).

One process per GPU runs an independent replica of the blend (it does not shard); the ranks
meet only to take the slowest rank's time, and the whole-job figure counts every rank's work.
"""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(times[rank], "cpu", world)
    dist.barrier()
    out[rank] = slowest
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [3.5, 7.25]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        assert dict(out) == {0: 7.25, 1: 7.25}
    # whole job: both ranks' units over the slowest time
    assert bench.whole_job_rate(1000, world, 7.25) == pytest.approx(2000 / 7.25e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.0, "cpu", 1) == 4.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""
