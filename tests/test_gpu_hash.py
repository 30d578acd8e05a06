"""The hash gate on the GPU (HAI-LLM's HashGate, top-1): routing bit for bit against the oracle's
fmix32(token id) mod E, and the whole layer against the oracle's hash-gated forward (counts,
offsets and slots bit for bit, y within the layer's float bar)."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from harness import Inputs, as_f64, bits_of, config_of, tol_ok, widen
from mixture_experts_layer_96_b300 import ForwardOutputs, MoEError, Workspace, moe_forward_hash, moe_route_hash
from workloads import WORKLOADS, Generator, MoEShape, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


CASES = [
    MoEShape("hash_e16_cf1.2", T=1000, h=256, E=16, K=1, d_ff=256, capacity_factor=1.2),
    MoEShape("hash_e64_nodrop", T=3000, h=512, E=64, K=1, d_ff=384),
    MoEShape("hash_heads2", T=700, h=512, E=32, K=1, d_ff=256, n_heads=2, capacity_factor=1.0),
    MoEShape("hash_e5_odd", T=300, h=128, E=5, K=1, d_ff=192, capacity_factor=0.8),
    MoEShape("hash_f32", T=256, h=128, E=8, K=1, d_ff=256, dtype="f32", capacity_factor=1.25),
]


@pytest.mark.parametrize("shape", CASES, ids=[c.name for c in CASES])
def test_hash_gate_forward_parity(shape):
    inp = Inputs.make(shape)
    ids = Generator(shape).token_ids()
    cfg = config_of(shape)
    x, lw = inp.device()
    ids_d = torch.from_numpy(ids).cuda()
    ws = Workspace(cfg)
    outs = ForwardOutputs.allocate(cfg, "cuda")
    y = moe_forward_hash(cfg, x, ids_d, lw.w_gate, lw.w_up, lw.w_down, ws=ws, outputs=outs)
    ws.check()
    b = inp.bf16
    ref = O.forward_hashed(widen(inp.x, b), ids, lambda e: (widen(inp.w1[e], b), widen(inp.w3[e], b),
                                                           widen(inp.w2[e], b)),
                           E=shape.E, n_heads=shape.n_heads, capacity_factor=shape.capacity_factor)
    np.testing.assert_array_equal(bits_of(outs.topk_idx), ref.idx)
    assert (bits_of(outs.topk_gate) == 1.0).all()
    np.testing.assert_array_equal(bits_of(outs.counts), ref.dispatch.counts)
    np.testing.assert_array_equal(bits_of(outs.offsets), ref.dispatch.offsets)
    np.testing.assert_array_equal(bits_of(outs.slot_of), ref.dispatch.slot_of)
    assert float(outs.aux.item()) == 0.0
    ok, err, bound = tol_ok(as_f64(y), ref.y, shape.dtype)
    assert ok, f"max |y - y_ref| = {err} > {bound}"


def test_hash_route_alone_and_negative_ids():
    shape = MoEShape("hash_route", T=513, h=64, E=48, K=1, d_ff=64)
    cfg = config_of(shape)
    ids = np.concatenate([np.array([-1, 0, 1, 2 ** 31 - 1, -2 ** 31], np.int32),
                          Generator(shape).token_ids()[:508]])
    ws = Workspace(cfg)
    idx, gate = moe_route_hash(cfg, torch.from_numpy(ids).cuda(), ws=ws)
    ws.check()
    np.testing.assert_array_equal(bits_of(idx), O.hash_route(ids, shape.E)[0])
    assert (bits_of(gate) == 1.0).all()


def test_hash_gate_needs_top1():
    shape = scaled(WORKLOADS["mixtral_bf16"], T=64, h=256, d_ff=256)  # K = 2
    cfg = config_of(shape)
    ws = Workspace(cfg)
    with pytest.raises(MoEError):
        moe_route_hash(cfg, torch.zeros(64, dtype=torch.int32, device="cuda"), ws=ws,
                       topk_idx=torch.empty((64, 2), dtype=torch.int32, device="cuda"),
                       topk_gate=torch.empty((64, 2), dtype=torch.float32, device="cuda"))
