"""End-to-end parity of moe_forward against the oracle (GPU).

Routing is checked bit for bit: the GPU's fp32 router logits (written by moe_forward, logit bias
included) must lie within the fp32 error bound of the exact logits, and the oracle, routing on
those same fp32 logits, must pick exactly the GPU's experts for every unit. Counts, offsets and
packed slots must then equal the oracle's dispatch of those picks, the gates the oracle's gates
on those logits, and y must meet the layer's float tolerance against the oracle's float64 layer
at those picks.
"""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from harness import TILE_MODES, Inputs, as_f64, bits_of, config_of, expert_tiles, route_on_gpu_logits, tol_ok
from mixture_experts_layer_96_b300 import (ForwardOutputs, Workspace, moe_combine, moe_dispatch,
                                           moe_expert_ffn, moe_forward, moe_route)
from workloads import WORKLOADS, MoEShape, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


SMALL = [
    WORKLOADS["tiny_f32"],
    scaled(WORKLOADS["mixtral_bf16"], T=700, h=512, d_ff=1024),
    scaled(WORKLOADS["finegrained_bf16"], T=300, h=512, d_ff=256),
    scaled(WORKLOADS["skewed_bf16"], T=3000, h=256, d_ff=384),
    scaled(WORKLOADS["multihead_bf16"], T=600, h=1024, d_ff=512),
    MoEShape("drop_heavy", T=500, h=128, E=4, K=2, d_ff=128, capacity_factor=0.3, logit_bias="zipf1.2"),
    MoEShape("one_unit", T=1, h=64, E=8, K=2, d_ff=64),
    # Switch-style top-1 routing with HAI-LLM's training / validation capacity factors
    MoEShape("switch_top1_cf1.2", T=1000, h=256, E=16, K=1, d_ff=256, capacity_factor=1.2, logit_bias="zipf1.2"),
    MoEShape("switch_top1_cf1.5", T=1000, h=256, E=16, K=1, d_ff=256, capacity_factor=1.5, logit_bias="zipf1.2"),
    MoEShape("dense_e1", T=200, h=64, E=1, K=1, d_ff=96),
]


def run_forward(inp: Inputs):
    cfg = config_of(inp.shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    outs = ForwardOutputs.allocate(cfg, "cuda")
    y = moe_forward(cfg, x, lw, ws=ws, outputs=outs)
    ws.check()
    return y, outs


def check_forward(inp: Inputs, y, outs, sample=None):
    """`sample`: None (every unit), an array of units, or a callable that picks the units from
    the oracle's dispatch of the GPU's picks."""
    s = inp.shape
    gidx, gate_ref, gl = route_on_gpu_logits(inp, outs)
    if callable(sample):
        sample = sample(O.dispatch(gidx, s.E, O.capacity(s.capacity_factor, s.K, s.T_units, s.E)))
    # the oracle's layer at the GPU's picks (float64 logits, gates and experts)
    ref = inp.oracle_forward(sample_units=sample, idx_override=gidx)
    d = ref.dispatch
    np.testing.assert_array_equal(bits_of(outs.counts), d.counts)
    np.testing.assert_array_equal(bits_of(outs.offsets), d.offsets)
    np.testing.assert_array_equal(bits_of(outs.slot_of), d.slot_of)
    # gates from the same fp32 logits: fp32 softmax / sigmoid normalisation against float64
    np.testing.assert_allclose(as_f64(outs.topk_gate), gate_ref, atol=2e-6, rtol=0)
    aux_ref = O.aux_loss(gl, gidx, s.E, s.K, s.aux_alpha, s.score)
    aux = float(outs.aux.item())
    assert abs(aux - aux_ref) <= 1e-4 * abs(aux_ref) + 1e-7, (aux, aux_ref)
    yg = as_f64(y)
    if sample is None:
        ok, err, tb = tol_ok(yg, ref.y, s.dtype)
    else:
        yu = yg.reshape(s.T_units, s.h_unit)
        got = np.stack([yu[u] for u in sample])
        want = np.stack([ref.y_units[int(u)] for u in sample])
        ok, err, tb = tol_ok(got, want, s.dtype)
    assert ok, f"max |y - y_ref| = {err} > {tb}"
    return gidx


@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_forward_parity_small(shape):
    inp = Inputs.make(shape)
    y, outs = run_forward(inp)
    check_forward(inp, y, outs)


def test_forward_is_deterministic_and_equals_the_stages():
    shape = scaled(WORKLOADS["skewed_bf16"], T=2000, h=256, d_ff=384)
    inp = Inputs.make(shape)
    cfg = config_of(shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    y1 = moe_forward(cfg, x, lw, ws=ws)
    y2 = moe_forward(cfg, x, lw, ws=ws)
    ws.check()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    idx, gate, _, _ = moe_route(cfg, x, lw.w_router, lw.logit_bias, lw.select_bias, ws=ws)
    counts, offsets, slot_of, row_token, xp = moe_dispatch(cfg, x, idx, ws=ws)
    yp = moe_expert_ffn(cfg, xp, offsets, lw.w_gate, lw.w_up, lw.w_down, ws=ws)
    y3 = moe_combine(cfg, yp, slot_of, gate, ws=ws)
    ws.check()
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))


def test_forward_replays_from_a_cuda_graph():
    """moe_forward allocates and synchronises nothing, so a captured forward replays to the same
    bits as a direct call (the benchmark times graph replays)."""
    shape = scaled(WORKLOADS["multihead_bf16"], T=600, h=1024, d_ff=512)
    inp = Inputs.make(shape)
    cfg = config_of(shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    y_direct = moe_forward(cfg, x, lw, ws=ws)
    y = torch.empty_like(y_direct)
    outs = ForwardOutputs.allocate(cfg, "cuda")
    moe_forward(cfg, x, lw, ws=ws, y=y, outputs=outs)  # first use outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe_forward(cfg, x, lw, ws=ws, y=y, outputs=outs)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(y.view(torch.int16), y_direct.view(torch.int16))


def test_forward_empty_batch():
    shape = MoEShape("empty", T=0, h=128, E=8, K=2, d_ff=128)
    cfg = config_of(shape)
    ws = Workspace(cfg)
    inp = Inputs.make(scaled(shape, T=1))
    _, lw = inp.device()
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    outs = ForwardOutputs.allocate(cfg, "cuda")
    y = moe_forward(cfg, x, lw, ws=ws, outputs=outs)
    ws.check()
    assert y.shape == (0, 128)
    assert bits_of(outs.counts).tolist() == [0] * 8
    assert bits_of(outs.offsets).tolist() == [0] * 9
    assert float(outs.aux.item()) == 0.0


# ------------------------------------------------------------------------- full-size, sampled
FULL = ["mixtral_bf16", "skewed_bf16", "multihead_bf16", "tiny_f32", "finegrained_bf16"]


def tile_covering_sample(n_min: int, seed: int = 123):
    """Units whose outputs the full-size check computes: for every expert with rows, the units
    of its first and last packed row (so each expert's first and last m-tile is looked at,
    ragged tails included), plus random units up to n_min."""
    def pick(d):
        units = set()
        for e in range(len(d.offsets) - 1):
            r0, r1 = int(d.offsets[e]), int(d.offsets[e + 1])
            if r1 > r0:
                units.add(int(d.row_token[r0]))
                units.add(int(d.row_token[r1 - 1]))
        rng = np.random.default_rng(seed)
        T = d.slot_of.shape[0]
        while len(units) < min(n_min, T):
            units.add(int(rng.integers(T)))
        return np.array(sorted(units), dtype=np.int64)
    return pick


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_forward_parity_full_size_sampled(name):
    shape = WORKLOADS[name]
    inp = Inputs.make(shape)
    y, outs = run_forward(inp)
    check_forward(inp, y, outs, sample=tile_covering_sample(256))


def test_forward_parity_when_the_route_grid_exceeds_two_ctas_per_sm():
    """More 128-unit tiles than two per SM (T' = 40000, h' = 512: 313 single-CTA tiles), so the
    routing kernel runs in more than one wave: routing stays bit-exact on the GPU's logits for every
    unit, and y is checked on a tile-covering sample."""
    shape = scaled(WORKLOADS["multihead_bf16"], T=10000, d_ff=256)
    inp = Inputs.make(shape)
    y, outs = run_forward(inp)
    check_forward(inp, y, outs, sample=tile_covering_sample(256))


def test_profiled_forward_gives_the_same_bits_and_ordered_stage_events():
    """moe_forward_profiled runs the forward's own kernels with an event at each stage boundary: y
    and the outputs equal moe_forward's bit for bit, and the events bracket five stages."""
    from mixture_experts_layer_96_b300 import moe_forward_profiled
    shape = scaled(WORKLOADS["skewed_bf16"], T=2000, h=256, d_ff=384)
    inp = Inputs.make(shape)
    cfg = config_of(shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    o1, o2 = ForwardOutputs.allocate(cfg, "cuda"), ForwardOutputs.allocate(cfg, "cuda")
    y1 = moe_forward(cfg, x, lw, ws=ws, outputs=o1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    y2 = moe_forward_profiled(cfg, x, lw, ev, ws=ws, outputs=o2)
    torch.cuda.synchronize()
    ws.check()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    for t1, t2 in zip(o1.tensors(), o2.tensors()):
        assert torch.equal(t1, t2)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times) and sum(times) > 0


# ---------------------------------------------------------- combine folded into the down GEMM
FOLD_CASES = [
    scaled(WORKLOADS["skewed_bf16"], T=2000, h=256, d_ff=384),             # K = 2, capacity drops
    MoEShape("switch_top1_cf1.2", T=1000, h=256, E=16, K=1, d_ff=256, capacity_factor=1.2,
             logit_bias="zipf1.2"),                                       # K = 1: g·Y written directly
    MoEShape("drop_heavy", T=500, h=128, E=4, K=2, d_ff=128, capacity_factor=0.3,
             logit_bias="zipf1.2"),                                       # units with no kept pick
    scaled(WORKLOADS["finegrained_bf16"], T=300, h=512, d_ff=256),        # K = 8, sigmoid, groups
    MoEShape("e33k5", T=700, h=96, E=33, K=5, d_ff=160),                  # K = 5, ragged widths
    scaled(WORKLOADS["multihead_bf16"], T=600, h=1024, d_ff=1024),        # H = 4, many 256-row tiles
    scaled(WORKLOADS["mixtral_bf16"], T=900, h=512, d_ff=1024),
]


@pytest.mark.parametrize("mode", list(TILE_MODES))
@pytest.mark.parametrize("shape", FOLD_CASES, ids=[s.name for s in FOLD_CASES])
def test_folded_combine_equals_the_separate_combine(shape, mode):
    """moe_forward with the combine folded into the down GEMM (forced on for every K: with K >= 2
    the last row of each unit sums it) must give the bits of the separate stages
    route → dispatch → expert_ffn → combine, for every tile shape of the down GEMM (plain rows and
    transposed tails), with every y element written (y starts as NaN)."""
    inp = Inputs.make(shape)
    cfg = config_of(shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    with expert_tiles(mode, fold_combine=1):
        y = torch.full((shape.T, shape.h), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe_forward(cfg, x, lw, ws=ws, y=y)
        y_again = torch.full_like(y, float("nan"))
        moe_forward(cfg, x, lw, ws=ws, y=y_again)
        idx, gate, _, _ = moe_route(cfg, x, lw.w_router, lw.logit_bias, lw.select_bias, ws=ws)
        counts, offsets, slot_of, row_token, xp = moe_dispatch(cfg, x, idx, ws=ws)
        yp = moe_expert_ffn(cfg, xp, offsets, lw.w_gate, lw.w_up, lw.w_down, ws=ws)
        y_sep = moe_combine(cfg, yp, slot_of, gate, ws=ws)
        ws.check()
    assert not torch.isnan(y.float()).any()
    assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16))
    assert torch.equal(y.view(torch.int16), y_again.view(torch.int16))
    # units none of whose picks was kept are zero
    dropped = (bits_of(slot_of) < 0).all(axis=1)
    if dropped.any():
        yu = y.view(shape.T_units, shape.h_unit)
        assert not yu[torch.from_numpy(np.nonzero(dropped)[0]).cuda()].any()


@pytest.mark.parametrize("K", [1, 2])
def test_combine_is_folded_automatically_for_top1_only(K):
    """Automatic choice: a top-1 forward folds the combine into the down GEMM (one launch fewer),
    a top-2 forward keeps the separate combine launch; both equal the separate stages' bits."""
    from mixture_experts_layer_96_b300 import launch_count
    shape = MoEShape(f"top{K}", T=800, h=256, E=16, K=K, d_ff=256, capacity_factor=1.25)
    inp = Inputs.make(shape)
    cfg = config_of(shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    counts = {}
    ys = {}
    for fold in (-1, 0):
        with expert_tiles("single", fold_combine=fold):
            moe_forward(cfg, x, lw, ws=ws)  # first call outside the count (one-time setup)
            torch.cuda.synchronize()
            n0 = launch_count()
            ys[fold] = moe_forward(cfg, x, lw, ws=ws)
            counts[fold] = launch_count() - n0
    ws.check()
    assert counts[-1] == counts[0] - (1 if K == 1 else 0), counts
    assert torch.equal(ys[-1].view(torch.int16), ys[0].view(torch.int16))
