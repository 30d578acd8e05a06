"""Parity of moe_forward_train + moe_backward against the backward oracle (GPU).

The GPU's routing is first checked bit for bit against the oracle's routing of the GPU's own fp32
logits; the oracle's gradient is then taken at the GPU's picks, which is what the backward
differentiates (routing held fixed).

Tolerance, from the rounding points of the bf16 path: dY_packed, dG|dU, dX_packed, G|U and H are
each rounded to bf16 once (unit roundoff u = 2^-8 relative per element), and every gradient is a
sum of products of such values in fp32. A gradient element therefore carries a few u relative to
the sum of |terms|, which for sums of mixed-sign random terms is a modest multiple of the largest
result. The bar, per gradient tensor: max|got − ref| <= 2e-2·max|ref| and
||got − ref||_F <= 1e-2·||ref||_F (about 2.5 u).
"""
import numpy as np
import pytest
import torch

import oracle.moe_backward as B
from harness import Inputs, as_f64, bits_of, config_of, expert_tiles, route_on_gpu_logits, to_device, widen
from mixture_experts_layer_96_b300 import (BackwardWorkspace, ForwardOutputs, Workspace, moe_backward,
                                           moe_forward, moe_forward_train)
from workloads import WORKLOADS, Generator, MoEShape, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


D_AUX = 0.7

SMALL = [
    scaled(WORKLOADS["mixtral_bf16"], T=700, h=512, d_ff=1024),
    scaled(WORKLOADS["skewed_bf16"], T=1500, h=256, d_ff=384, E=16),                       # drops, Zipf bias
    scaled(WORKLOADS["finegrained_bf16"], T=300, h=512, d_ff=256),                         # sigmoid, groups, K=8
    scaled(WORKLOADS["multihead_bf16"], T=400, h=1024, d_ff=512, E=16),                    # 4 heads, h'=256
    MoEShape("odd_tiles", T=300, h=192, E=5, K=2, d_ff=192, capacity_factor=0.9),           # partial M/N tiles
    MoEShape("sparse_experts", T=20, h=128, E=16, K=1, d_ff=128),                           # empty experts
    MoEShape("switch_top1", T=600, h=128, E=8, K=1, d_ff=256, capacity_factor=1.2, logit_bias="zipf1.2"),
    MoEShape("drop_heavy", T=500, h=128, E=4, K=2, d_ff=128, capacity_factor=0.3, logit_bias="zipf1.2"),
]


def grad_ok(got, ref):
    err = np.abs(got - ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    fro_ref = float(np.linalg.norm(ref))
    ok_max = float(err.max(initial=0.0)) <= 2e-2 * scale + 1e-6
    ok_fro = float(np.linalg.norm(got - ref)) <= 1e-2 * fro_ref + 1e-6
    return ok_max and ok_fro, float(err.max(initial=0.0)), scale, float(np.linalg.norm(got - ref)) / max(fro_ref, 1e-30)


def run_train(inp: Inputs):
    s = inp.shape
    cfg = config_of(s)
    x, lw = inp.device()
    ws = Workspace(cfg)
    outs = ForwardOutputs.allocate(cfg, "cuda")
    y, gu = moe_forward_train(cfg, x, lw, outs, ws=ws)
    dy = to_device(Generator(s).dy(), True)
    bws = BackwardWorkspace(cfg)
    g = moe_backward(cfg, x, lw, dy, outs, gu, ws=ws, bws=bws, d_aux=D_AUX)
    ws.check()
    return cfg, x, lw, ws, outs, y, gu, dy, bws, g


def gpu_picks_checked(inp: Inputs, outs):
    """The GPU's picks, after checking them bit for bit against the oracle's routing of the same
    fp32 logits."""
    gidx, _, _ = route_on_gpu_logits(inp, outs)
    return gidx


def oracle_grads(inp: Inputs, dy_bits, idx):
    s = inp.shape
    W1, W3, W2 = inp.w1, inp.w3, inp.w2
    return B.backward(widen(inp.x, True), widen(inp.w_g, True), lambda e: (widen(W1[e], True), widen(W3[e], True),
                      widen(W2[e], True)), widen(dy_bits, True), D_AUX, E=s.E, K=s.K, d_ff=s.d_ff, score=s.score,
                      n_heads=s.n_heads, n_groups=s.n_groups, topk_groups=s.topk_groups,
                      capacity_factor=s.capacity_factor, aux_alpha=s.aux_alpha, logit_bias=inp.logit_bias,
                      select_bias=inp.select_bias, idx_override=idx)


def check_all(inp, g, ref):
    pairs = [("dgate", g.dgate, ref.dgate), ("dlogits", g.dlogits, ref.dlogits), ("dw_down", g.dw_down, ref.dw2),
             ("dw_gate", g.dw_gate, ref.dw1), ("dw_up", g.dw_up, ref.dw3), ("dw_router", g.dw_router, ref.dw_g),
             ("dx", g.dx, ref.dx)]
    for name, got, want in pairs:
        ok, err, scale, rel = grad_ok(as_f64(got), want)
        assert ok, f"{name}: max err {err:.3e} vs max|ref| {scale:.3e}, relative Frobenius {rel:.3e}"


@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_backward_parity_small(shape):
    inp = Inputs.make(shape)
    cfg, x, lw, ws, outs, y, gu, dy, bws, g = run_train(inp)
    idx = gpu_picks_checked(inp, outs)
    ref = oracle_grads(inp, Generator(shape).dy(), idx)
    np.testing.assert_array_equal(bits_of(outs.slot_of), ref.slot_of)
    check_all(inp, g, ref)


@pytest.mark.parametrize("mode", ["single_tails_transposed", "single_tails_plain", "pair_tails_transposed",
                                  "pair_tails_plain"])
def test_backward_parity_with_each_forward_tile_mode(mode):
    """G|U are saved by every forward epilogue: single-CTA tiles, pair tiles, transposed tails."""
    shape = scaled(WORKLOADS["mixtral_bf16"], T=900, h=256, d_ff=512)
    inp = Inputs.make(shape)
    with expert_tiles(mode):
        cfg, x, lw, ws, outs, y, gu, dy, bws, g = run_train(inp)
    idx = gpu_picks_checked(inp, outs)
    check_all(inp, g, oracle_grads(inp, Generator(shape).dy(), idx))


def test_forward_train_equals_forward_and_saves_the_swiglu_inputs():
    shape = scaled(WORKLOADS["skewed_bf16"], T=1200, h=256, d_ff=384, E=16)
    inp = Inputs.make(shape)
    cfg = config_of(shape)
    x, lw = inp.device()
    ws = Workspace(cfg)
    y0 = moe_forward(cfg, x, lw, ws=ws)
    outs = ForwardOutputs.allocate(cfg, "cuda")
    y1, gu = moe_forward_train(cfg, x, lw, outs, ws=ws)
    ws.check()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    # G|U of each kept packed row against X_e·W1ᵀ, X_e·W3ᵀ (bf16 rounding of the fp32 result)
    off = bits_of(outs.offsets).astype(np.int64)
    slot = bits_of(outs.slot_of).astype(np.int64)
    xu = widen(inp.x, True)
    gu64 = as_f64(gu)
    idx = bits_of(outs.topk_idx)
    for t in range(0, shape.T_units, 37):
        for k in range(shape.K):
            r = slot[t, k]
            if r < 0:
                continue
            e = int(idx[t, k])
            assert off[e] <= r < off[e + 1]
            G = widen(inp.w1[e], True) @ xu[t]
            U = widen(inp.w3[e], True) @ xu[t]
            want = np.concatenate([G, U])
            assert np.max(np.abs(gu64[r] - want)) <= 2 ** -8 * np.max(np.abs(want)) + 1e-3


def test_backward_empty_batch():
    """T = 0: nothing to route; the weight gradients are zero and every call succeeds."""
    shape = MoEShape("empty", T=0, h=128, E=8, K=2, d_ff=128)
    cfg = config_of(shape)
    inp = Inputs.make(scaled(shape, T=1))
    _, lw = inp.device()
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    ws = Workspace(cfg)
    outs = ForwardOutputs.allocate(cfg, "cuda")
    y, gu = moe_forward_train(cfg, x, lw, outs, ws=ws)
    g = moe_backward(cfg, x, lw, torch.empty_like(x), outs, gu, ws=ws, bws=BackwardWorkspace(cfg), d_aux=1.0)
    ws.check()
    assert g.dx.shape == (0, 128)
    for name in ("dw_router", "dw_gate", "dw_up", "dw_down"):
        assert int(torch.count_nonzero(getattr(g, name))) == 0, name


def test_backward_is_deterministic():
    shape = scaled(WORKLOADS["multihead_bf16"], T=400, h=1024, d_ff=512, E=16)
    inp = Inputs.make(shape)
    cfg, x, lw, ws, outs, y, gu, dy, bws, g1 = run_train(inp)
    g2 = moe_backward(cfg, x, lw, dy, outs, gu, ws=ws, bws=bws, d_aux=D_AUX)
    ws.check()
    for name in ("dx", "dw_router", "dw_gate", "dw_up", "dw_down", "dlogits", "dgate"):
        a, b = getattr(g1, name), getattr(g2, name)
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), name


# ------------------------------------------------------------------------- full-size, sampled
FULL = ["mixtral_bf16", "skewed_bf16", "multihead_bf16", "finegrained_bf16"]


def sampled_ok(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    scale = float(np.max(np.abs(want)))
    err = float(np.max(np.abs(got - want)))
    assert err <= 2e-2 * scale + 1e-6, f"{what}: max err {err:.3e} vs max|ref| {scale:.3e}"


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_backward_parity_full_size_sampled(name):
    """The benchmark's layers at full size, in the benchmark's launch configuration. Sampled units
    (dgate, dlogits, whole dx rows) and sampled weight-gradient entries against the oracle's
    entry-by-entry gradients; then a second backward with dy = 0, where dl is the aux term alone
    and the oracle differentiates the router path whole (dW_g, dx, dlogits; expert grads exactly 0)."""
    shape = WORKLOADS[name]
    inp = Inputs.make(shape)
    cfg, x, lw, ws, outs, y, gu, dy, bws, g = run_train(inp)
    ref = inp.oracle_forward(sample_units=np.array([0]))   # routing of all units; y of one
    gidx, _, _ = route_on_gpu_logits(inp, outs, exact_logits=ref.logits)
    counts = np.bincount(gidx.reshape(-1), minlength=shape.E)
    slot = bits_of(outs.slot_of)
    rng = np.random.default_rng(321)
    units = np.sort(rng.choice(shape.T_units, size=6, replace=False))
    live = [e for e in range(shape.E) if counts[e] > 0 and np.any(gidx[slot >= 0] == e)]
    def at(n, d0, d1):
        return [(int(rng.choice(live)), int(rng.integers(d0)), int(rng.integers(d1))) for _ in range(n)]
    hu, F = shape.h_unit, shape.d_ff
    at2, at1, at3 = at(10, hu, F), at(10, F, hu), at(10, F, hu)
    W1, W3, W2 = inp.w1, inp.w3, inp.w2
    ex = lambda e: (widen(W1[e], True), widen(W3[e], True), widen(W2[e], True))
    dy_bits = Generator(shape).dy()
    ent = B.backward_entries(widen(inp.x, True), widen(inp.w_g, True), ex, widen(dy_bits, True), D_AUX, gidx,
                             E=shape.E, K=shape.K, score=shape.score, n_heads=shape.n_heads,
                             capacity_factor=shape.capacity_factor, aux_alpha=shape.aux_alpha,
                             logit_bias=inp.logit_bias, units=units, dw2_at=at2, dw1_at=at1, dw3_at=at3)
    H = shape.n_heads
    dx_units = g.dx.view(shape.T_units, hu)
    sampled_ok([float(g.dgate[u, k]) for u in units for k in range(shape.K)],
               [ent["dgate"][(u, k)] for u in units for k in range(shape.K)], "dgate")
    sampled_ok(np.stack([as_f64(g.dlogits[u]) for u in units]), np.stack([ent["dlogits"][u] for u in units]), "dlogits")
    for u in units:
        sampled_ok(as_f64(dx_units[u]), ent["dx"][u], f"dx[{u}]")
    for key, ats, t in (("dw2", at2, g.dw_down), ("dw1", at1, g.dw_gate), ("dw3", at3, g.dw_up)):
        sampled_ok([float(t[a]) for a in ats], [ent[key][a] for a in ats], key)

    # dy = 0: dl = d_aux·(aux gradient) for every unit; the router path is checked whole
    zero = torch.zeros_like(dy)
    g0 = moe_backward(cfg, x, lw, zero, outs, gu, ws=ws, bws=bws, d_aux=1.0, grads=g)  # reuses g's buffers
    ws.check()
    l = ref.logits
    dl = B.aux_backward(l, gidx, shape.E, shape.K, shape.aux_alpha, shape.score, 1.0)
    xu = O_split(widen(inp.x, True), H)
    sampled_ok(as_f64(g0.dlogits), dl, "dlogits (aux only)")
    sampled_ok(as_f64(g0.dw_router), xu.T @ dl, "dW_g (aux only)")
    sampled_ok(as_f64(g0.dx.view(shape.T_units, hu)), dl @ widen(inp.w_g, True).T, "dx (aux only)")
    for name_, t in (("dw_down", g0.dw_down), ("dw_gate", g0.dw_gate), ("dw_up", g0.dw_up)):
        assert int(torch.count_nonzero(t)) == 0, name_


def O_split(x, H):
    import oracle.moe_oracle as O
    return O.split_heads(x, H)
