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
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` runs on host cores alone (the CPU oracle on a bounded sample)
    and prints one JSON line with the keys of the bench contract, for the same metric and
    workload as the GPU arm."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "0", "--ref-rows", "4"], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1 and "4 query rows" in d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("wan")
