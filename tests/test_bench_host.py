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


def test_gemm_bytes_by_hand():
    s = bench.WORKLOADS["mixtral_bf16"]
    kept = s.T_units * s.K
    w = 3 * 8 * 4096 * 14336 * 2                   # W1, W3, W2 of every expert, bf16
    a = kept * (4096 + 14336 + 14336 + 4096) * 2     # x_packed, H written and read, y_packed
    assert bench.gemm_bytes(s, kept, 8) == w + a
    assert bench.gemm_bytes(s, kept, 3) - bench.gemm_bytes(s, kept, 2) == 3 * 4096 * 14336 * 2


def test_layer_roofline_dense_workload_is_tensor_bound():
    s = bench.WORKLOADS["mixtral_bf16"]
    kept = s.T_units * s.K
    stage = {"route": 0.02, "dispatch": 0.03, "expert_ffn": 2.2, "combine": 0.04}
    lr = bench.layer_roofline(s, kept, 8, stage, 2.35, 7000.0, 1413.0)
    assert lr["gemm_bound"] == "tensor"
    t_ffn = 6.0 * 4096 * 14336 * kept / 1413e12
    assert lr["expert_ffn_ms_at_roofline"] == pytest.approx(1e3 * t_ffn)
    # dispatch: x read, x_packed written, 8 B of slot bookkeeping per kept row
    assert lr["dispatch_ms_at_roofline"] == pytest.approx(1e3 * (4096 * 4096 * 2 * 3 + kept * 8) / 7e12)
    parts = [lr[f"{k}_ms_at_roofline"] for k in ("route", "dispatch", "expert_ffn", "combine")]
    assert lr["sum_ms_at_roofline"] == pytest.approx(sum(parts))
    assert lr["frac_of_forward"] == pytest.approx(lr["sum_ms_at_roofline"] / 2.35)
    assert lr["stage_frac"]["expert_ffn"] == pytest.approx(1e3 * t_ffn / 2.2)
    assert 0.8 < lr["frac_of_forward"] < 1.0


def test_layer_roofline_with_the_combine_folded_into_the_down_gemm():
    """Folded: the expert_ffn stage's time holds the combine too, so it is graded against both
    rooflines; the combine has no stage fraction of its own; the sum is unchanged."""
    s = bench.WORKLOADS["multihead_bf16"]
    kept = s.T_units * s.K
    stage = {"route": 0.02, "dispatch": 0.04, "expert_ffn": 0.4, "combine": 0.001}
    plain = bench.layer_roofline(s, kept, 64, stage, 0.5, 7000.0, 1413.0)
    fold = bench.layer_roofline(s, kept, 64, stage, 0.5, 7000.0, 1413.0, folded=True)
    assert "combine" not in fold["stage_frac"]
    both = fold["expert_ffn_ms_at_roofline"] + fold["combine_ms_at_roofline"]
    assert fold["stage_frac"]["expert_ffn"] == pytest.approx(both / 0.4)
    assert fold["sum_ms_at_roofline"] == pytest.approx(plain["sum_ms_at_roofline"])
    assert fold["stage_frac"]["route"] == plain["stage_frac"]["route"]


def test_layer_roofline_fine_grained_workload_streams_weights():
    """256 experts of d_ff 2048 at T = 4096: each expert's weights are read for ~128 rows, so the
    GEMMs take longer to stream their weights from HBM than to do their FLOP."""
    s = bench.WORKLOADS["finegrained_bf16"]
    kept = s.T_units * s.K
    stage = {"route": 0.03, "dispatch": 0.1, "expert_ffn": 4.8, "combine": 0.1}
    lr = bench.layer_roofline(s, kept, 256, stage, 5.03, 7000.0, 1413.0)
    assert lr["gemm_bound"] == "hbm"
    assert lr["expert_ffn_ms_at_roofline"] == pytest.approx(1e3 * bench.gemm_bytes(s, kept, 256) / 7e12)
    # with few experts active the weight stream shrinks below the FLOP time
    assert bench.layer_roofline(s, kept, 16, stage, 5.03, 7000.0, 1413.0)["gemm_bound"] == "tensor"


def test_median_of_step_times():
    assert bench.median([3.0, 1.0, 2.0]) == 2.0
    assert bench.median([4.0, 1.0, 2.0, 3.0]) == 2.5
    assert bench.median([]) == 0.0


def test_cpu_baseline_adds_a_single_core_time_for_the_f32_layer():
    cb = bench.cpu_baseline_leg(bench.WORKLOADS["tiny_f32"], 8)
    assert cb["kind"] == "oracle" and cb["value"] > 0
    assert cb["single_core_value"] is not None and cb["single_core_value"] > 0


def test_nvml_sampler_reads_reason_bits():
    """NVML samples (timestamp, SM MHz, max MHz, clock-event reason bits) summarise like the
    nvidia-smi record: median clock inside the window and the active slowdown reasons."""
    c = bench.NvmlClockSampler(0)
    c._thread = object()  # as if the sampling thread had run
    t = 1000.0
    c.samples = [(t, 1900.0, 2032.0, 0x0), (t + 0.01, 1300.0, 2032.0, 0x4), (t + 0.02, 1200.0, 2032.0, 0x4 | 0x40),
                 (t + 5.0, 500.0, 2032.0, 0x8)]
    s = c.summary(t - 0.001, t + 0.03, t - 1, t + 10)
    assert s["samples"] == 3 and s["sm_mhz"] == 1300
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_reference_arm_times_a_real_sub_batch(monkeypatch, capsys):
    """No scaling: value × the step time is the number of tokens each step runs."""
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class A:
        ref_sample, steps, warmup, gpus = 64, 2, 1, 1
    bench.run_reference(A(), bench.WORKLOADS["tiny_f32"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["config"]["tokens_per_step"] == 64
    assert line["value"] * line["ms_per_step"] / 1000.0 == pytest.approx(64, rel=1e-9)


def test_oracle_sub_batch_sizes():
    # whole batch for the small layer; a bounded sub-batch for the benchmark layer
    assert bench.default_oracle_tokens(bench.WORKLOADS["tiny_f32"]) == 256
    n = bench.default_oracle_tokens(bench.WORKLOADS["mixtral_bf16"])
    assert 64 <= n < 4096
