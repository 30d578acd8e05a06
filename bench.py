#!/usr/bin/env python3
"""Benchmark of the MoE FFN layer forward (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one forward of the whole layer (router → Top-K → capacity/dispatch → expert SwiGLU
grouped GEMMs → combine, plus the aux loss) over one batch of the workload, inputs resident in
HBM. Default workload: the Mixtral-shaped layer (T=4096, h=4096, E=8, K=2, d_ff=14336, bf16,
softmax Top-2, no drop). `value` is tokens/s of the whole job (N replicas, one per GPU, each with
its own batch: weak scaling). Between timed steps L2 holds nothing useful: each forward streams
more expert weight than L2 holds (2.8 GB here); layers whose weights fit in L2 get a 512 MiB
write between steps, outside the timed events.

--impl reference times the CPU oracle (float64 numpy) on the host cores on a bounded sample of
the same workload, scaled to tokens/s.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, Generator, bf16_bits_to_f32, scaled  # noqa: E402

METRIC = "MoE-layer fwd tokens/s"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


GEMM_SOURCES = ("mixture_experts_layer_96_b300/csrc/expert_tc.cu", "mixture_experts_layer_96_b300/csrc/moe_device.cuh")


def gemm_source_sha() -> str:
    import hashlib
    h = hashlib.sha1()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(workload: str):
    """DRAM bytes of one forward's expert GEMM launches from a committed ncu capture
    (profiles/traffic.json), or None when the GEMM sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("source_sha1") != gemm_source_sha():
        return None
    return rec["dram_bytes_per_forward"]


def choose_peak(pk: dict, clocks: dict):
    """Burst peak for a kernel running at full clocks; the sustained (power-capped) peak when the
    clock samples of the timed region show the power cap or clocks well below maximum."""
    capped = "sw_power_cap" in clocks.get("reasons", []) or (
        clocks.get("sm_mhz") and clocks.get("sm_max_mhz") and clocks["sm_mhz"] < 0.9 * clocks["sm_max_mhz"])
    if capped and "bf16_tflops_sustained" in pk:
        return float(pk["bf16_tflops_sustained"]), f"bf16 sustained ({pk['source']}): power-capped clocks in the timed region"
    return float(pk["bf16_tflops"]), f"bf16 burst ({pk['source']})"


SPEC_BF16_TFLOPS = 2250.0  # B300 dense bf16, nominal


def gemm_bytes(shape, kept: int, e_active: int) -> float:
    """HBM bytes of the expert GEMMs of one forward: the active experts' weights once, plus the
    activations (x_packed read, H written and read back, y_packed written)."""
    s = 2 if shape.dtype == "bf16" else 4
    weights = 3.0 * e_active * shape.h_unit * shape.d_ff * s
    acts = kept * (shape.h_unit + 2 * shape.d_ff + shape.h_unit) * s
    return weights + acts


def layer_roofline(shape, kept: int, e_active: int, stage_ms: dict, ms_per_forward: float, hbm_gbs: float,
                   gemm_peak_tf: float, folded: bool = False) -> dict:
    """Each stage's time at its roofline and the forward's fraction of their sum.

    route: x, W_g and the picks at HBM rate, or the router FLOP at the tensor peak if that is
    longer; dispatch and combine: their bytes at HBM rate; expert GEMMs: the longer of FLOP at the
    tensor peak and weight + activation bytes at HBM rate (that choice names the GEMMs' bound).
    folded: the combine runs inside the down GEMM, so the expert_ffn stage is graded against the
    sum of both rooflines and the combine stage has no time of its own.
    """
    s = 2 if shape.dtype == "bf16" else 4
    Tu, hu, E, K = shape.T_units, shape.h_unit, shape.E, shape.K
    bw = hbm_gbs * 1e9
    pk = gemm_peak_tf * 1e12
    route = max((Tu * hu * s + hu * E * s + Tu * K * 8) / bw, 2.0 * Tu * hu * E / pk)
    dispatch = (Tu * hu * s + kept * hu * s + kept * 8) / bw
    combine = (kept * hu * s + Tu * hu * s + Tu * K * 8) / bw
    t_flop = 6.0 * hu * shape.d_ff * kept / pk
    t_bytes = gemm_bytes(shape, kept, e_active) / bw
    ffn = max(t_flop, t_bytes)
    roof = {"route": route, "dispatch": dispatch, "expert_ffn": ffn, "combine": combine}
    total = sum(roof.values())
    out = {f"{k}_ms_at_roofline": 1e3 * v for k, v in roof.items()}
    out.update({
        "sum_ms_at_roofline": 1e3 * total,
        "forward_ms": ms_per_forward,
        "frac_of_forward": 1e3 * total / ms_per_forward if ms_per_forward > 0 else None,
        "gemm_bound": "tensor" if t_flop >= t_bytes else "hbm",
        "stage_frac": ({k: 1e3 * roof[k] / stage_ms[k] for k in roof if stage_ms.get(k) and k != "combine"}
                       | {"expert_ffn": 1e3 * (ffn + combine) / stage_ms["expert_ffn"]}) if folded else
                      {k: 1e3 * roof[k] / stage_ms[k] for k in roof if stage_ms.get(k)},
        "peaks": {"hbm_gbs": hbm_gbs, "bf16_tflops": gemm_peak_tf},
    })
    return out


def median(values) -> float:
    return float(statistics.median(values)) if values else 0.0


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank value over all ranks (the slowest rank sets the step)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms with host timestamps; summary() keeps the samples inside
    a wall-clock window (the timed region), or, when that region is shorter than the sampling
    period, the samples of the surrounding busy window (warm-up, timed loop, stage loop)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def _rows(self):
        import datetime
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        return rows

    def summary(self, t0, t1, busy0, busy1):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = self._rows()
        sel = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not sel:
            sel = [r for r in rows if busy0 <= r[0] <= busy1]
            window = "busy window around the timed region (shorter than the sampling period)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = sorted({n for r in sel for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": sel[-1][2], "reasons": reasons,
                "samples": len(sel), "window": window}


class NvmlClockSampler(ClockSampler):
    """The same record from NVML in a sampling thread every 5 ms (a 40 ms timed region then holds
    several samples); falls back to nvidia-smi when NVML cannot be opened."""
    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
                   0x4: "sw_power_cap"}

    def __init__(self, device_index: int, period_s: float = 0.005):
        super().__init__(device_index)
        self.period = period_s
        self.samples = []  # (timestamp, sm_mhz, max_mhz, reason bitmask)
        self._thread = None
        self._stop = None
        self._nvml = None

    def start(self):
        import threading
        try:
            import pynvml as nv
            nv.nvmlInit()
            h = nv.nvmlDeviceGetHandleByIndex(self.dev)
            reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            max_mhz = float(nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM))
        except Exception:
            return super().start()
        self._nvml = nv
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                try:
                    self.samples.append((time.time(), float(nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM)),
                                         max_mhz, int(reasons(h))))
                except Exception:
                    pass
                self._stop.wait(self.period)

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        return self

    def stop(self):
        if self._thread is None:
            return super().stop()
        self._stop.set()
        self._thread.join(timeout=5)
        try:
            self._nvml.nvmlShutdown()
        except Exception:
            pass

    def _rows(self):
        if self._thread is None:
            return super()._rows()
        order = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        bit = {v: k for k, v in self.REASON_BITS.items()}
        return [(ts, mhz, mx, ["Active" if (mask & bit[n]) else "Not Active" for n in order])
                for ts, mhz, mx, mask in self.samples]


# ------------------------------------------------------------------------------------ inputs
def device_inputs(shape, device):
    from mixture_experts_layer_96_b300 import LayerWeights
    g = Generator(shape, seed=0)
    bf = shape.dtype == "bf16"

    def dev(a):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if bf else torch.from_numpy(a)
        return t.to(device)

    x_host = g.x()
    w1, w3, w2 = g.experts()
    lb, sb = g.logit_bias(), g.select_bias()
    lw = LayerWeights(dev(g.w_router()), dev(w1), dev(w3), dev(w2),
                      None if lb is None else torch.from_numpy(lb).to(device),
                      None if sb is None else torch.from_numpy(sb).to(device))
    del w1, w3, w2
    return dev(x_host), lw


def kept_rows(shape):
    if shape.capacity_factor is None:
        return shape.T_units * shape.K
    return None  # data-dependent; read back after a run


# ------------------------------------------------------------------------------------ CPU oracle
def default_oracle_tokens(shape) -> int:
    """Tokens per oracle step: the whole batch for small layers, else a sub-batch of about 3e11
    expert FLOP (about half a second of float64 BLAS on a GPU server's host cores)."""
    per_token = 6.0 * shape.h_unit * shape.d_ff * shape.K * shape.n_heads
    return int(max(16, min(shape.T, 3e11 // per_token)))


class OracleSubBatch:
    """The oracle's whole layer forward on a sub-batch: the workload's first `n_tokens` tokens taken
    as a batch of their own (routing, capacity and aux loss over those tokens), with the workload's
    weights. Inputs are widened to float64 before timing, like inputs resident on the GPU; expert
    weights too, unless the experts the sub-batch routes to exceed `widen_budget_gb`, in which case
    the oracle widens each expert when it needs it, inside the timed step."""

    def __init__(self, shape, n_tokens: int, seed: int = 0, widen_budget_gb: float = 24.0):
        import oracle.moe_oracle as O
        self.O = O
        self.shape = shape
        self.n = int(min(n_tokens, shape.T))
        g = Generator(shape, seed)
        self.g = g
        bf = shape.dtype == "bf16"
        self.f64 = (lambda a: bf16_bits_to_f32(a).astype(np.float64)) if bf else (lambda a: np.asarray(a, np.float64))
        self.x = self.f64(g.x()[: self.n])
        self.wg = self.f64(g.w_router())
        self.kw = dict(E=shape.E, K=shape.K, score=shape.score, n_heads=shape.n_heads, n_groups=shape.n_groups,
                       topk_groups=shape.topk_groups, capacity_factor=shape.capacity_factor,
                       aux_alpha=shape.aux_alpha, logit_bias=g.logit_bias(), select_bias=g.select_bias())
        r = O.forward(self.x, self.wg, lambda e: None, sample_units=np.zeros(0, np.int64), **self.kw)
        need = sorted(int(e) for e in np.unique(r.idx))
        per_expert = 3.0 * shape.d_ff * shape.h_unit * 8
        self.cache = {}
        self.prewidened = len(need) * per_expert <= widen_budget_gb * 1e9
        if self.prewidened:
            for e in need:
                self.cache[e] = tuple(self.f64(w) for w in g.expert(e))

    def _expert(self, e):
        if e in self.cache:
            return self.cache[e]
        return tuple(self.f64(w) for w in self.g.expert(e))

    def step(self) -> float:
        """Seconds of one oracle forward over the sub-batch."""
        t0 = time.perf_counter()
        self.O.forward(self.x, self.wg, self._expert, **self.kw)
        return time.perf_counter() - t0

    def describe(self) -> str:
        s = self.shape
        how = "weights widened before timing" if self.prewidened else "expert weights widened inside the step"
        return (f"float64 numpy oracle: the whole layer forward on the first {self.n} of the {s.T} tokens as "
                f"their own batch ({s.T_units // s.T * self.n} routed units), {how}")


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else 1
    except Exception:
        # without threadpoolctl: an explicit BLAS thread setting, else the cores this process may use
        for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(k, "").isdigit():
                return int(os.environ[k])
        return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline_leg(shape, n_tokens):
    """The oracle timed like the reference arm: one untimed and two timed sub-batch steps."""
    run = OracleSubBatch(shape, n_tokens)
    run.step()
    t = min(run.step(), run.step())
    out = {"value": run.n / t, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
           "sample": run.describe() + "; best of 2 steps"}
    if shape.dtype == "f32":  # the small layer: also the oracle on one core
        try:
            out["single_core_value"] = single_core_oracle(shape.name, n_tokens)
        except Exception as ex:  # a report extra: never lose the line for it
            out["single_core_value"] = None
            out["single_core_error"] = repr(ex)
    return out


def oracle_tokens_per_s(name: str, n_tokens: int) -> float:
    run = OracleSubBatch(WORKLOADS[name], n_tokens)
    run.step()
    return run.n / min(run.step(), run.step())


def single_core_oracle(name: str, n_tokens: int, timeout_s: float = 300.0) -> float:
    """The oracle's tokens/s with its BLAS held to one thread: a fresh interpreter (the thread
    count is fixed when numpy loads) that sees no GPU."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        env.pop(k, None)
    code = f"import bench; print(bench.oracle_tokens_per_s({name!r}, {int(n_tokens)}))"
    r = subprocess.run([sys.executable, "-c", code], cwd=os.path.dirname(os.path.abspath(__file__)), env=env,
                       capture_output=True, text=True, timeout=timeout_s, check=True)
    return float(r.stdout.strip().splitlines()[-1])


# ------------------------------------------------------------------------------------ reference arm
def run_reference(args, shape):
    """The oracle as the reference arm: W untimed and K timed steps, each the oracle's forward on the
    same sub-batch; value = its tokens / the mean step time (no scaling to the full batch)."""
    _, rank, _ = dist_env()
    if rank != 0:
        return
    n = args.ref_sample if getattr(args, "ref_sample", None) else default_oracle_tokens(shape)
    run = OracleSubBatch(shape, n)
    times = []
    for i in range(args.warmup + args.steps):
        t = run.step()
        if i >= args.warmup:
            times.append(t)
    ms = 1000.0 * statistics.mean(times)
    v = run.n / (ms / 1000.0)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator, the workload's recipe)",
            "config": {"workload": shape.describe(), "tokens_per_step": run.n, "global_batch": shape.T,
                       "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": run.describe()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------ train leg
def train_supported(shape) -> bool:
    return shape.dtype == "bf16" and shape.h_unit % 64 == 0 and shape.d_ff % 64 == 0


def train_leg(args, shape, cfg, x, lw, device, flush, stream):
    """One training step of the layer = moe_forward_train + moe_backward (routing held fixed), timed
    with CUDA events per part, inputs and the upstream gradient resident. Reported beside the
    forward metric, not in place of it."""
    from mixture_experts_layer_96_b300 import (BackwardWorkspace, ForwardOutputs, Grads, Workspace, launch_count,
                                               moe_backward, moe_forward_train)
    ws = Workspace(cfg, device=device)
    outs = ForwardOutputs.allocate(cfg, device)
    rows = shape.T_units * shape.K
    gu = torch.empty((rows, 2 * shape.d_ff), dtype=x.dtype, device=device)
    bws = BackwardWorkspace(cfg, device=device)
    grads = Grads.allocate(cfg, device, extras=False)
    dy_bits = Generator(shape).dy()
    dy = torch.from_numpy(dy_bits.view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.empty_like(x)

    def step():
        moe_forward_train(cfg, x, lw, outs, ws=ws, gu=gu, y=y)
        moe_backward(cfg, x, lw, dy, outs, gu, ws=ws, bws=bws, d_aux=1.0, grads=grads)

    clk = NvmlClockSampler(device.index or 0).start()
    b0 = time.time()
    n_warm = 0
    while n_warm < max(3, args.warmup) or time.time() - b0 < min(args.min_warmup_s, 1.0):
        step()
        n_warm += 1
    ws.check()
    kept = int(outs.offsets[-1].item())
    c0 = launch_count()
    step()
    per_step = launch_count() - c0
    n = max(3, args.steps // 2)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    torch.cuda.synchronize(device)
    t0 = time.time()
    for i in range(n):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        moe_forward_train(cfg, x, lw, outs, ws=ws, gu=gu, y=y)
        ev[i][1].record(stream)
        moe_backward(cfg, x, lw, dy, outs, gu, ws=ws, bws=bws, d_aux=1.0, grads=grads)
        ev[i][2].record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    clk.stop()
    ws.check()
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    bwd_flop = 12.0 * shape.h_unit * shape.d_ff * kept   # dH, dX (2x), dW2, dW1|dW3 (2x)
    return {
        "what": "forward_train (saves G|U) + backward (dx, dW_g, dW1, dW3, dW2; routing held fixed), d_aux=1",
        "steps": n, "ms_per_step": fwd_ms + bwd_ms, "forward_train_ms": fwd_ms, "backward_ms": bwd_ms,
        "tokens_per_s": shape.T / ((fwd_ms + bwd_ms) * 1e-3), "unit": "tokens/s",
        "backward_algorithmic_flop": bwd_flop,
        "backward_tflops_whole": bwd_flop / (bwd_ms * 1e-3) / 1e12,
        "gpu_launches_per_step": per_step,
        "clocks": clk.summary(t0, t1, b0, t1),
    }


# ------------------------------------------------------------------------------------ our arm
def run_ours(args, shape):
    from mixture_experts_layer_96_b300 import ForwardOutputs, Workspace, launch_count, moe_forward, moe_forward_profiled
    from mixture_experts_layer_96_b300.moe import FORWARD_STAGES
    from mixture_experts_layer_96_b300.moe import make_config

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = make_config(shape.T, shape.h, shape.E, shape.K, shape.d_ff, n_heads=shape.n_heads,
                      n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                      capacity_factor=shape.capacity_factor, aux_alpha=shape.aux_alpha,
                      score=shape.score, dtype=shape.dtype)
    x, lw = device_inputs(shape, device)
    ws = Workspace(cfg, device=device)
    outs = ForwardOutputs(aux=torch.empty(1, dtype=torch.float32, device=device),
                          counts=torch.empty(shape.E, dtype=torch.int32, device=device),
                          offsets=torch.empty(shape.E + 1, dtype=torch.int32, device=device))
    y = torch.empty_like(x)
    # L2 between timed steps: every bf16 workload streams more expert weight per forward than the
    # 126 MB L2 holds, which evicts it; smaller layers get a 512 MiB write between steps instead.
    weight_bytes = 3 * shape.E * shape.d_ff * shape.h_unit * (2 if shape.dtype == "bf16" else 4)
    l2_bytes = 126 * 1024 * 1024
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device) if weight_bytes <= l2_bytes else None
    l2_note = (f"inputs larger than L2: {weight_bytes / 1e9:.2f} GB of expert weights streamed per forward"
               if flush is None else "flushed between timed steps (512 MiB write, outside the events)")
    stream = torch.cuda.current_stream(device)

    def barrier():
        torch.cuda.synchronize(device)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(device)

    clk = NvmlClockSampler(local).start()
    busy0 = time.time()
    n_warm = 0
    while n_warm < max(3, args.warmup) or time.time() - busy0 < args.min_warmup_s:
        moe_forward(cfg, x, lw, ws=ws, y=y, outputs=outs)
        n_warm += 1
        if n_warm % 50 == 0:
            torch.cuda.synchronize(device)
    ws.check()
    kept = int(outs.offsets[-1].item())
    aux = float(outs.aux.item())
    counts = outs.counts.cpu().tolist()

    # kernels one forward launches (counted by the library)
    c0 = launch_count()
    moe_forward(cfg, x, lw, ws=ws, y=y, outputs=outs)
    per_forward = launch_count() - c0
    graph = None
    if args.graph:
        # the forward allocates and synchronises nothing, so it can be captured once and replayed
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            moe_forward(cfg, x, lw, ws=ws, y=y, outputs=outs)
        graph.replay()
        torch.cuda.synchronize(device)
        ws.check()

    # ---- timed: whole forward, one event pair per step, L2 flushed between steps (untimed)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    n0 = launch_count()
    t0 = time.time()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            moe_forward(cfg, x, lw, ws=ws, y=y, outputs=outs)
        ev[i][1].record(stream)
    barrier()
    t1 = time.time()
    n_launch = (per_forward * args.steps) if graph is not None else (launch_count() - n0)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = aggregate_max(sum(step_ms) / args.steps, world, device)
    ms_median = aggregate_max(median(step_ms), world, device)
    ws.check()

    # ---- per-stage events: the same forward with an event at each stage boundary (moe_forward_profiled;
    # programmatic dependent launch is off between stages there, so the stages' sum exceeds a step)
    st = {k: [] for k in FORWARD_STAGES}
    prof = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        moe_forward_profiled(cfg, x, lw, prof, ws=ws, y=y, outputs=outs)
        torch.cuda.synchronize(device)
        for j, k in enumerate(FORWARD_STAGES):
            st[k].append(prof[j].elapsed_time(prof[j + 1]))
    ws.check()
    busy1 = time.time()
    clk.stop()
    clocks = clk.summary(t0, t1, busy0, busy1)
    busy_clocks = clk.summary(busy0, busy1, busy0, busy1)  # warm-up + timed + stage loops
    stage_ms = {k: statistics.mean(v) for k, v in st.items()}

    # ---- e2e: every step copies its input x from pinned host memory to the device, runs the
    # forward through the public API and copies y (and the aux loss) back to pinned host memory.
    # Like a serving loop, the copies of neighbouring steps run on their own streams while this
    # step computes (device x and y double-buffered, ordered by events).
    x_host = x.cpu().pin_memory()
    y_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    aux_host = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    yd = [torch.empty_like(x) for _ in range(2)]
    auxd = [torch.empty(1, dtype=torch.float32, device=device) for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    n_e2e = args.steps
    ev_in = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_done = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_out = [torch.cuda.Event() for _ in range(n_e2e)]
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(n_e2e):
        b = i & 1
        if i >= 2:
            s_h2d.wait_event(ev_done[i - 2])        # xd[b] no longer read by step i-2
        with torch.cuda.stream(s_h2d):
            xd[b].copy_(x_host, non_blocking=True)
        ev_in[i].record(s_h2d)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])        # yd[b] already copied out by step i-2
        outs_i = ForwardOutputs(aux=auxd[b], counts=outs.counts, offsets=outs.offsets)
        moe_forward(cfg, xd[b], lw, ws=ws, y=yd[b], outputs=outs_i, stream=stream)
        ev_done[i].record(stream)
        s_d2h.wait_event(ev_done[i])
        with torch.cuda.stream(s_d2h):
            y_host[b].copy_(yd[b], non_blocking=True)
            aux_host[b].copy_(auxd[b], non_blocking=True)
        ev_out[i].record(s_d2h)
    s_d2h.wait_event(ev_done[n_e2e - 1])
    e1.record(s_d2h)
    barrier()
    e2e_ms = aggregate_max(e0.elapsed_time(e1) / n_e2e, world, device)
    h2d = x_host.numel() * x_host.element_size()
    d2h = y_host[0].numel() * y_host[0].element_size() + 4
    train = None
    if args.train and train_supported(shape):
        del xd, yd, x_host, y_host
        train = train_leg(args, shape, cfg, x, lw, device, flush, stream)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel group (the expert grouped GEMMs). Its time inside a timed
    # forward is the step time times the GEMMs' share of the profiled forward's stages (the stages
    # run without overlap there), so achieved never exceeds what the timed step allows.
    pk = peaks()
    flops = 6.0 * shape.h_unit * shape.d_ff * kept
    stage_sum = sum(stage_ms.values())
    gemm_share = stage_ms["expert_ffn"] / stage_sum if stage_sum > 0 else 1.0
    gemm_ms_in_step = ms * gemm_share
    achieved_tf = flops / (gemm_ms_in_step * 1e-3) / 1e12
    achieved_profiled_tf = flops / (stage_ms["expert_ffn"] * 1e-3) / 1e12
    # the regime (power-capped or not) is read from the whole busy window: the timed region alone
    # can be shorter than a few samples and catch the clock between power-cap adjustments
    peak_tf, peak_kind = choose_peak(pk, busy_clocks)
    elt = 2 if shape.dtype == "bf16" else 4
    # dispatch: x read, x_packed written, per pick its index and place read and slot written, per
    # packed row its source unit written
    d_bytes = shape.T_units * shape.h_unit * elt + kept * shape.h_unit * elt + shape.T_units * shape.K * 12 + \
        shape.T_units * shape.K * 4
    c_bytes = kept * shape.h_unit * elt + shape.T_units * shape.h_unit * elt + shape.T_units * shape.K * 8
    # top-1 bf16 layers fold the combine into the down GEMM's epilogue (the library's automatic choice)
    folded = shape.dtype == "bf16" and shape.K == 1
    hbm = float(pk["hbm_gbs"])
    disp_ms = stage_ms["scan"] + stage_ms["pack"]
    stages = {f"{k}_ms": v for k, v in stage_ms.items()}
    stages.update({
        "dispatch_ms": disp_ms, "expert_ffn_tflops_profiled": achieved_profiled_tf,
        "expert_ffn_share_of_step": gemm_share,
        "pack_gbs": d_bytes / (stage_ms["pack"] * 1e-3) / 1e9,
        "dispatch_gbs": d_bytes / (disp_ms * 1e-3) / 1e9,
        "how": "moe_forward_profiled: the forward's own kernels with a CUDA event at each stage boundary",
    })
    stages["pack_frac_hbm"] = stages["pack_gbs"] / hbm
    stages["dispatch_frac_hbm"] = stages["dispatch_gbs"] / hbm
    if folded:
        stages["combine"] = "folded into the down GEMM's epilogue: expert_ffn_ms includes it"
    else:
        stages["combine_gbs"] = c_bytes / (stage_ms["combine"] * 1e-3) / 1e9
        stages["combine_frac_hbm"] = stages["combine_gbs"] / hbm
    value = world * shape.T / (ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": n_warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if shape.dtype == "bf16" else "f32",
        "data": "synthetic (seeded generator; x~N(0,1), W~N(0,1/fan_in), bf16)",
        "config": {"workload": shape.describe(), "global_batch": shape.T * world, "units_per_gpu": shape.T_units,
                   "parallelism": f"replicas x{world} (data parallel, no collective on the data path)",
                   "l2": l2_note,
                   "kept_rows": kept, "aux_loss": aux,
                   "cuda_graph": bool(args.graph), "kernels_per_forward": per_forward, "max_over_mean_load": max(counts) / (sum(counts) / len(counts))},
        "roofline": {"bound": "tensor", "kernel": "expert grouped GEMMs (gate/up+SwiGLU and down, 2 launches per forward)"
                     + (", the down GEMM with the combine folded in" if folded else ""),
                     "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved_tf / peak_tf,
                     "how": "6·h'·d_ff·kept FLOP per forward ÷ (ms_per_step × the GEMMs' share of the profiled "
                            "forward's stage times)",
                     "gemm_ms_in_step": gemm_ms_in_step, "achieved_profiled": achieved_profiled_tf,
                     "peak_kind": peak_kind,
                     "frac_of_burst": achieved_tf / float(pk["bf16_tflops"]),
                     "frac_of_sustained": achieved_tf / float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                     "algorithmic_flop": flops,
                     "traffic": recorded_traffic(args.workload) if args.d_ff is None else None,
                     "traffic_unit": "DRAM bytes per forward (both GEMM launches), ncu",
                     "gemm_source_sha1": gemm_source_sha()},
        "stages": stages,
        "clocks": clocks,
        "clocks_busy_window": busy_clocks,
        "e2e": {"value": shape.T * world / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "pinned host x -> device, moe_forward, y and aux -> pinned host every step; copies of "
                       "neighbouring steps overlap this step's compute on two copy streams"},
        "gpu_launches": n_launch,
    }
    line["ms_per_step_median"] = ms_median
    line["roofline"]["frac_of_spec"] = achieved_tf / SPEC_BF16_TFLOPS
    try:  # report extras: on any error the line keeps everything above and says why
        e_active = sum(1 for c in counts if c > 0)
        lr_stage = {"route": stage_ms["route"], "dispatch": disp_ms, "expert_ffn": stage_ms["expert_ffn"],
                    "combine": stage_ms["combine"]}
        lr = layer_roofline(shape, kept, e_active, lr_stage, ms, hbm, peak_tf, folded)
        line["layer_roofline"] = lr
        if lr["gemm_bound"] == "hbm":
            # the GEMMs stream more weight bytes than their FLOP take at the tensor peak: the HBM
            # roofline grades them; the tensor view stays in the line
            gb = gemm_bytes(shape, kept, e_active)
            ach = gb / (gemm_ms_in_step * 1e-3) / 1e9
            tensor_view = dict(line["roofline"])
            line["roofline"] = {"bound": "hbm", "kernel": tensor_view["kernel"], "achieved": ach, "peak": hbm,
                                "unit": "GB/s", "frac": ach / hbm, "algorithmic_bytes": gb,
                                "traffic": tensor_view["traffic"], "traffic_unit": tensor_view["traffic_unit"],
                                "gemm_source_sha1": tensor_view["gemm_source_sha1"], "tensor_view": tensor_view}
    except Exception as ex:
        line["layer_roofline"] = {"error": repr(ex)}
    if train is not None:
        bw_peak = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
        train["backward_frac_of_sustained_whole"] = train["backward_tflops_whole"] / bw_peak
        line["train"] = train
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_leg(shape, args.cpu_sample or default_oracle_tokens(shape))
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral_bf16", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-sample", type=int, default=None,
                    help="tokens per CPU-baseline oracle step (default: the whole batch, or ~1e11 expert FLOP)")
    ap.add_argument("--ref-sample", type=int, default=None,
                    help="tokens per reference-arm step (default as --cpu-sample)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", dest="graph", action="store_true", default=True,
                    help="replay the forward from a CUDA graph in the timed loop (default)")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--train", dest="train", action="store_true", default=True,
                    help="also time a training step (forward_train + backward) and report it under 'train'")
    ap.add_argument("--no-train", dest="train", action="store_false")
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up at least this long (steady clocks); 0 for profiling runs")
    ap.add_argument("--d-ff", type=int, default=None,
                    help="replace the workload's d_ff (small cases for profiler captures of the kernels that "
                         "do not depend on it; the line then names the changed workload)")
    args = ap.parse_args()
    shape = WORKLOADS[args.workload]
    if args.d_ff is not None:
        shape = scaled(shape, d_ff=args.d_ff)
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_ours(args, shape)


if __name__ == "__main__":
    main()
