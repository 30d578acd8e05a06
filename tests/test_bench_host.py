"""Host logic of bench.py: max-over-ranks aggregation on world-size-2 gloo ranks, the reference
arm's rank behaviour, clock-sample parsing and the roofline peak choice (CPU only)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own step time; the job's step is the slowest rank's
        v = bench.aggregate_max(1.5 + rank, world)
        dist.barrier()
        out[rank] = v
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_only_rank0_prints(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        ref_sample, steps, warmup, gpus = 1, 1, 0, 2
    bench.run_reference(A(), bench.WORKLOADS["tiny_f32"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(monkeypatch, capsys):
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class A:
        ref_sample, steps, warmup, gpus = 2, 2, 1, 1
    bench.run_reference(A(), bench.WORKLOADS["tiny_f32"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_clock_summary_window_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [
        "2026/12/02 10:00:00.000, 0, 1900, 2032, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.200, 0, 1300, 2032, 1099.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.400, 0, 1200, 2032, 1099.0, 0x4, Not Active, Not Active, Not Active, Active",
    ]
    import datetime
    t = datetime.datetime(2026, 12, 2, 10, 0, 0).timestamp()
    s = c.summary(t + 0.1, t + 0.5, t - 1, t + 1)
    assert s["sm_mhz"] == 1250 and s["reasons"] == ["sw_power_cap"] and s["samples"] == 2
    s = c.summary(t + 5, t + 6, t - 1, t + 1)  # no sample inside: fall back to the busy window
    assert s["samples"] == 3 and "busy" in s["window"]


def test_peak_choice():
    pk = {"bf16_tflops": 1815.6, "bf16_tflops_sustained": 1413.1, "source": "measured"}
    assert bench.choose_peak(pk, {"reasons": [], "sm_mhz": 2032, "sm_max_mhz": 2032})[0] == 1815.6
    assert bench.choose_peak(pk, {"reasons": ["sw_power_cap"], "sm_mhz": 1300, "sm_max_mhz": 2032})[0] == 1413.1
    assert bench.choose_peak(pk, {"reasons": [], "sm_mhz": 1000, "sm_max_mhz": 2032})[0] == 1413.1
