"""Stage-by-stage parity of the CUDA library against the oracle, through the C ABI (GPU).

Each stage gets seeded inputs from the shared generator (never from another CUDA stage), and is
compared with the oracle on the same inputs: routing decisions, counts, queues and packed rows
bit-exactly; floats within the layer's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from harness import TILE_MODES, as_f64, bits_of, config_of, expert_tiles, to_device, tol_ok, widen
from mixture_experts_layer_96_b300 import (Workspace, moe_combine, moe_dispatch, moe_expert_ffn,
                                           moe_route_logits)
from workloads import Generator, MoEShape, WORKLOADS, f32_to_bf16_bits, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


# ------------------------------------------------------------------------------------- routing
ROUTE_CASES = [
    scaled(WORKLOADS["mixtral_bf16"], T=1000),
    scaled(WORKLOADS["finegrained_bf16"], T=600),
    scaled(WORKLOADS["skewed_bf16"], T=3000),
    scaled(WORKLOADS["multihead_bf16"], T=300),
    scaled(WORKLOADS["tiny_f32"], T=256),
    MoEShape("e1k1", T=77, h=64, E=1, K=1, d_ff=64),
    MoEShape("k_eq_e", T=130, h=64, E=4, K=4, d_ff=64),
    MoEShape("e3k2", T=300, h=64, E=3, K=2, d_ff=64),
    MoEShape("e33k5", T=300, h=64, E=33, K=5, d_ff=64),
    MoEShape("e128k8_groups", T=257, h=64, E=128, K=8, d_ff=64, n_groups=16, topk_groups=3),
    MoEShape("sigmoid_nobias", T=200, h=64, E=64, K=6, d_ff=64, score="sigmoid"),
    MoEShape("groups_gs1", T=200, h=64, E=16, K=3, d_ff=64, n_groups=16, topk_groups=4),
]


def _route_inputs(shape, ties):
    g = Generator(shape)
    l = g.logits()
    if ties:  # a coarse grid makes many exact ties in keys and group scores
        l = (np.round(l * 2.0) / 2.0).astype(np.float32)
    return l, g.logit_bias(), g.select_bias()


@pytest.mark.parametrize("ties", [False, True], ids=["random", "ties"])
@pytest.mark.parametrize("shape", ROUTE_CASES, ids=[s.name for s in ROUTE_CASES])
def test_route_logits_bit_exact(shape, ties):
    cfg = config_of(shape)
    l, lb, sb = _route_inputs(shape, ties)
    ws = Workspace(cfg)
    dl = torch.from_numpy(l).cuda()
    dlb = None if lb is None else torch.from_numpy(lb).cuda()
    dsb = None if sb is None else torch.from_numpy(sb).cuda()
    idx, gate, aux = moe_route_logits(cfg, dl, dlb, dsb, ws=ws, want_aux=True)
    ws.check()
    lf = O.logits_with_bias_f32(l, lb).astype(np.float64)
    r_idx, r_gate, _ = O.route(lf, shape.score, shape.K, sb, shape.n_groups, shape.topk_groups)
    np.testing.assert_array_equal(bits_of(idx), r_idx)
    np.testing.assert_allclose(as_f64(gate), r_gate, rtol=2e-6, atol=2e-7)
    r_aux = O.aux_loss(lf, r_idx, shape.E, shape.K, shape.aux_alpha, shape.score)
    assert abs(float(aux.item()) - r_aux) <= 1e-5 * abs(r_aux) + 1e-9


# ------------------------------------------------------------------------------------ dispatch
DISPATCH_CASES = [
    (scaled(WORKLOADS["mixtral_bf16"], T=1000, h=256), None),
    (scaled(WORKLOADS["skewed_bf16"], T=3000, h=256), 1.25),
    (scaled(WORKLOADS["finegrained_bf16"], T=700, h=256), None),
    (scaled(WORKLOADS["finegrained_bf16"], T=700, h=256), 0.5),
    (scaled(WORKLOADS["multihead_bf16"], T=150, h=1024), 1.0),
    (scaled(WORKLOADS["tiny_f32"], T=256), 1.25),
    (scaled(WORKLOADS["tiny_f32"], T=257, h=36), 0.05),  # nearly everything dropped; 144-byte rows
    (MoEShape("f32_oddrow", T=100, h=6, E=4, K=2, d_ff=8, dtype="f32"), 1.0),  # 24-byte rows
]


@pytest.mark.parametrize("shape,cf", DISPATCH_CASES, ids=[f"{s.name}-cf{cf}" for s, cf in DISPATCH_CASES])
def test_dispatch_bit_exact(shape, cf):
    shape = scaled(shape, capacity_factor=cf, name=shape.name)
    cfg = config_of(shape)
    g = Generator(shape)
    idx = g.topk_idx()
    x = g.x()
    b = shape.dtype == "bf16"
    ws = Workspace(cfg)
    counts, offsets, slot_of, row_token, x_packed = moe_dispatch(cfg, to_device(x, b), torch.from_numpy(idx).cuda(), ws=ws)
    ws.check()
    C = O.capacity(cf, shape.K, shape.T_units, shape.E)
    d = O.dispatch(idx, shape.E, C)
    np.testing.assert_array_equal(bits_of(counts), d.counts)
    np.testing.assert_array_equal(bits_of(offsets), d.offsets)
    np.testing.assert_array_equal(bits_of(slot_of), d.slot_of)
    np.testing.assert_array_equal(bits_of(row_token), d.row_token)
    kept = int(d.offsets[-1])
    xu = x.reshape(shape.T_units, shape.h_unit)
    np.testing.assert_array_equal(bits_of(x_packed)[:kept], xu[d.row_token[:kept]])


def test_dispatch_flags_bad_index():
    shape = MoEShape("bad", T=64, h=64, E=8, K=2, d_ff=64)
    cfg = config_of(shape)
    idx = Generator(shape).topk_idx()
    idx[5, 1] = 8          # out of range
    idx[9, 1] = idx[9, 0]  # repeated pick
    ws = Workspace(cfg)
    moe_dispatch(cfg, to_device(Generator(shape).x(), True), torch.from_numpy(idx).cuda(), ws=ws)
    assert ws.status() == 5  # MOE_ERR_DEVICE_STATUS
    assert ws.status() == 0  # read clears it


# ---------------------------------------------------------------------------------- expert FFN
FFN_CASES = [
    scaled(WORKLOADS["mixtral_bf16"], T=700, h=512, d_ff=1024),        # 2 m-tiles per expert, ragged
    scaled(WORKLOADS["finegrained_bf16"], T=200, h=256, d_ff=256),      # 256 experts, partial tiles
    scaled(WORKLOADS["skewed_bf16"], T=2000, h=512, d_ff=384, capacity_factor=1.25),
    scaled(WORKLOADS["multihead_bf16"], T=256, h=1024, d_ff=512),       # h' = 256
    MoEShape("odd_widths", T=300, h=96, E=5, K=2, d_ff=160),            # N and K tails
    MoEShape("narrow", T=100, h=32, E=3, K=1, d_ff=32),
    scaled(WORKLOADS["tiny_f32"], T=256),
    MoEShape("f32_odd", T=90, h=20, E=3, K=2, d_ff=36, dtype="f32"),
]


@pytest.fixture(params=list(TILE_MODES))
def tile_mode(request):
    """Run an expert-FFN case with the single-CTA 128-row tiles and with the CTA-pair 256-row tiles,
    each with the automatic choice for experts' last m-tiles and with every tail (up to 112 rows
    single, 224 pair) forced to the transposed tile or to the plain tile."""
    with expert_tiles(request.param):
        yield request.param


@pytest.mark.parametrize("shape", FFN_CASES, ids=[s.name for s in FFN_CASES])
def test_expert_ffn_parity(shape, tile_mode):
    cfg = config_of(shape)
    g = Generator(shape)
    b = shape.dtype == "bf16"
    idx = g.topk_idx()
    C = O.capacity(shape.capacity_factor, shape.K, shape.T_units, shape.E)
    d = O.dispatch(idx, shape.E, C)
    kept = int(d.offsets[-1])
    rows = shape.T_units * shape.K
    # packed rows: seeded values (the rows of x the queue selects, then filler past kept)
    xu = g.x().reshape(shape.T_units, shape.h_unit)
    xp = np.zeros((rows, shape.h_unit), dtype=xu.dtype)
    xp[:kept] = xu[d.row_token[:kept]]
    w1, w3, w2 = g.experts()
    ws = Workspace(cfg)
    yp = moe_expert_ffn(cfg, to_device(xp, b), torch.from_numpy(d.offsets.astype(np.int32)).cuda(),
                        to_device(w1, b), to_device(w3, b), to_device(w2, b), ws=ws)
    ws.check()
    got = as_f64(yp)[:kept]
    ref = np.zeros_like(got)
    for e in range(shape.E):
        r0, r1 = int(d.offsets[e]), int(d.offsets[e + 1])
        if r1 > r0:
            ref[r0:r1] = O.expert_ffn(widen(xp[r0:r1], b), widen(w1[e], b), widen(w3[e], b), widen(w2[e], b))
    ok, err, bound = tol_ok(got, ref, shape.dtype)
    assert ok, f"max err {err} > {bound}"


def test_expert_ffn_empty_and_skewed_experts(tile_mode):
    """Offsets with empty experts, one expert holding most rows, and unused rows at the end."""
    shape = MoEShape("skew_offsets", T=400, h=128, E=6, K=2, d_ff=256)
    cfg = config_of(shape)
    g = Generator(shape)
    rows = shape.T_units * shape.K
    offsets = np.array([0, 0, 517, 517, 530, 531, 700], dtype=np.int32)
    xu = Generator(scaled(shape, T=rows)).x()
    w1, w3, w2 = g.experts()
    ws = Workspace(cfg)
    yp = moe_expert_ffn(cfg, to_device(xu, True), torch.from_numpy(offsets).cuda(), to_device(w1, True),
                        to_device(w3, True), to_device(w2, True), ws=ws)
    ws.check()
    got = as_f64(yp)[:700]
    ref = np.zeros_like(got)
    for e in range(6):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = O.expert_ffn(widen(xu[r0:r1], True), widen(w1[e], True), widen(w3[e], True), widen(w2[e], True))
    ok, err, bound = tol_ok(got, ref, "bf16")
    assert ok, f"max err {err} > {bound}"


@pytest.mark.parametrize("h,d_ff", [(128, 256), (96, 160)], ids=["aligned", "ragged_widths"])
def test_expert_ffn_ragged_tails(tile_mode, h, d_ff):
    """Experts whose row counts put every kind of last m-tile in the batch: tails of 1, 16 and 17
    rows, at and just past the largest transposed tail (224, 225), just short of and at a full pair
    tile (255, 256), one row into the next (257), an expert of one full tile plus a tail (480)."""
    sizes = [1, 16, 17, 224, 225, 255, 256, 257, 480, 0, 33]
    E = len(sizes)
    shape = MoEShape("tails", T=900, h=h, E=E, K=2, d_ff=d_ff)
    cfg = config_of(shape)
    g = Generator(shape)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    kept = int(offsets[-1])
    xu = Generator(scaled(shape, T=shape.T_units * shape.K)).x()
    w1, w3, w2 = g.experts()
    ws = Workspace(cfg)
    yp = moe_expert_ffn(cfg, to_device(xu, True), torch.from_numpy(offsets).cuda(), to_device(w1, True),
                        to_device(w3, True), to_device(w2, True), ws=ws)
    ws.check()
    got = as_f64(yp)[:kept]
    ref = np.zeros_like(got)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            ref[r0:r1] = O.expert_ffn(widen(xu[r0:r1], True), widen(w1[e], True), widen(w3[e], True), widen(w2[e], True))
    for e in range(E):  # per expert, so that a wrong tail shows which one
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        ok, err, bound = tol_ok(got[r0:r1], ref[r0:r1], "bf16")
        assert ok, f"expert {e} ({sizes[e]} rows): max err {err} > {bound}"


def test_expert_ffn_flags_bad_offsets():
    shape = MoEShape("bad_off", T=64, h=64, E=4, K=2, d_ff=64)
    cfg = config_of(shape)
    g = Generator(shape)
    w1, w3, w2 = g.experts()
    ws = Workspace(cfg)
    bad = torch.tensor([0, 10, 5, 20, 30], dtype=torch.int32, device="cuda")  # decreasing
    xp = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    moe_expert_ffn(cfg, xp, bad, to_device(w1, True), to_device(w3, True), to_device(w2, True), ws=ws)
    assert ws.status() == 5


# ------------------------------------------------------------------------------------- combine
COMBINE_CASES = [
    (scaled(WORKLOADS["mixtral_bf16"], T=500, h=512), None),
    (scaled(WORKLOADS["skewed_bf16"], T=2000, h=256), 1.25),
    (scaled(WORKLOADS["multihead_bf16"], T=100, h=1024), 0.3),
    (scaled(WORKLOADS["tiny_f32"], T=256), 1.25),
    (MoEShape("f32_odd", T=50, h=10, E=3, K=2, d_ff=8, dtype="f32"), 1.0),
    # the bulk-copy combine: K = 8 rows of 14 KB in four segments, many items per block (the
    # stage ring wraps several times); K = 5 with drops and a shorter last segment; a long batch
    # of short rows, 24 units per stage
    (scaled(WORKLOADS["finegrained_bf16"], T=400), None),
    (MoEShape("k5_three_segments", T=300, h=4160, E=12, K=5, d_ff=64), 1.0),
    (MoEShape("many_units", T=40000, h=256, E=16, K=2, d_ff=64), 1.25),
]


@pytest.mark.parametrize("shape,cf", COMBINE_CASES, ids=[f"{s.name}-cf{cf}" for s, cf in COMBINE_CASES])
def test_combine_parity(shape, cf):
    shape = scaled(shape, capacity_factor=cf, name=shape.name)
    cfg = config_of(shape)
    g = Generator(shape)
    b = shape.dtype == "bf16"
    idx = g.topk_idx()
    d = O.dispatch(idx, shape.E, O.capacity(cf, shape.K, shape.T_units, shape.E))
    rows = shape.T_units * shape.K
    yp = np.random.default_rng(11).standard_normal((rows, shape.h_unit), dtype=np.float32)
    if b:
        yp = f32_to_bf16_bits(yp)
    gate = np.random.default_rng(7).random((shape.T_units, shape.K)).astype(np.float32)
    ws = Workspace(cfg)
    y = moe_combine(cfg, to_device(yp, b), torch.from_numpy(d.slot_of.astype(np.int32)).cuda(),
                    torch.from_numpy(gate).cuda(), ws=ws)
    ws.check()
    ref = O.merge_heads(O.combine(widen(yp, b), d.slot_of, gate.astype(np.float64)), shape.n_heads)
    got = as_f64(y)
    if b:  # only the final bf16 rounding differs
        np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-6)
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6)
    dropped_all = (d.slot_of < 0).all(axis=1)
    assert (O.split_heads(got, shape.n_heads)[dropped_all] == 0).all()
