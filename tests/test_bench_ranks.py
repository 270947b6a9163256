"""The multi-GPU path of bench.py (independent replicas, weak scaling) on CPU ranks.

Two gloo ranks stand in for two GPUs: each reports its own timed-region length; every
rank must see the slowest rank's time, and the whole-job value must count the work of
both replicas over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank])
        v = bench.whole_job_tflops(world, 1e12, 10, t)
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    times = [80.0, 95.5]
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, times, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 95.5
    # 2 replicas x 10 steps x 1e12 flop in 95.5 ms
    assert res[0][1] == pytest.approx(2 * 10 * 1e12 / 0.0955 / 1e12)


def test_single_process_is_unchanged():
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_tflops(1, 2e12, 5, 1000.0) == pytest.approx(10.0)


def test_clock_summary_keys_with_and_without_samples():
    """The clock record always carries the keys the bench line reads, also when the timed
    region was too short for any nvidia-smi sample."""
    keys = {"sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w"}
    c = bench.ClockSampler(0)
    c.out = ""
    empty = c.summary()
    assert keys <= set(empty) and empty["samples"] == 0 and empty["sm_mhz"] is None
    c.out = ("0, 1980, 2070, 1215.37, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
             "0, 1990, 2070, 1200.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")
    full = c.summary()
    assert keys <= set(full) and full["samples"] == 2
    assert full["sm_mhz"] == 1985.0 and full["sm_max_mhz"] == 2070.0 and full["reasons"] == ["sw_power_cap"]
    assert abs(full["power_w"] - 1207.685) < 1e-9
