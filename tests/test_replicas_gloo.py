"""The multi-GPU bench path is replicas only: each rank runs its own copy of
the stack and the only cross-rank step is the max of the timed regions.  Its
host logic runs here on CPU ranks over gloo (world size 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (t, bench.job_throughput(t, world, 1, 40, 200))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world, times = 2, [80.0, 125.0]
    with mp.get_context("spawn").Manager() as m:  # no fork of a threaded process
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    # every rank sees the slowest rank's time; the job rate counts both replicas' work
    assert res[0] == res[1]
    t, v = res[0]
    assert t == 125.0
    assert v == pytest.approx(2 * 1 * 40 * 200 / 0.125)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(2.0, 1, 4, 10, 5) == pytest.approx(4 * 10 * 5 / 0.002)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the other ranks exit without work or output."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.argparse.Namespace(layers=None, steps=3, warmup=3)
    assert bench.run_reference(args, bench.synth.WORKLOADS[1]) is None
    assert capsys.readouterr().out == ""
