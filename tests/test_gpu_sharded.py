"""moe_dispatch_sharded on the GPU, its ranks emulated one after another on one device (no
collectives, nothing waits on another launch): a batch split into consecutive token shards, each
dispatched with the picks of the earlier shards as its queue bases and the whole batch's capacity.
The shards' keep decisions, concatenated, must equal the single-device dispatch of the whole batch
bit for bit; each shard's counts, offsets and packed rows are its own."""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from harness import bits_of, config_of, to_device
from mixture_experts_layer_96_b300 import Workspace, moe_dispatch_sharded
from workloads import WORKLOADS, Generator, MoEShape, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


CASES = [
    (scaled(WORKLOADS["skewed_bf16"], T=3000, h=256), [1000, 700, 1300]),
    (MoEShape("sharded_k3", T=900, h=128, E=16, K=3, d_ff=64, capacity_factor=0.6), [300, 1, 299, 300]),
    (MoEShape("sharded_nodrop", T=512, h=64, E=8, K=2, d_ff=64), [256, 256]),
]


@pytest.mark.parametrize("shape,shards", CASES, ids=[c[0].name for c in CASES])
def test_sharded_dispatch_equals_whole_batch(shape, shards):
    assert sum(shards) == shape.T
    g = Generator(shape)
    x = g.x()
    idx = g.topk_idx()
    E, K = shape.E, shape.K
    ref = O.dispatch(idx, E, O.capacity(shape.capacity_factor, K, shape.T_units, E))
    kept, t0 = [], 0
    for n in shards:
        sub = scaled(shape, T=n, name=f"{shape.name}_shard")
        cfg = config_of(sub)
        loc_idx = idx[t0:t0 + n]
        base = np.bincount(idx[:t0].reshape(-1), minlength=E).astype(np.int32)   # picks on earlier shards
        ws = Workspace(cfg)
        counts, offsets, slot_of, row_token, xp = moe_dispatch_sharded(
            cfg, to_device(x[t0:t0 + n], True), torch.from_numpy(np.ascontiguousarray(loc_idx)).cuda(),
            torch.from_numpy(base).cuda(), shape.T, ws=ws)
        ws.check()
        so = bits_of(slot_of)
        kept.append(so >= 0)
        # the shard's own bookkeeping: local counts, local offsets of its kept rows, rows in unit order
        np.testing.assert_array_equal(bits_of(counts), np.bincount(loc_idx.reshape(-1), minlength=E))
        kept_e = np.bincount(loc_idx[so >= 0], minlength=E)
        np.testing.assert_array_equal(bits_of(offsets), np.concatenate([[0], np.cumsum(kept_e)]))
        rt = bits_of(row_token)
        xb = bits_of(xp)
        for e in range(E):
            r0, r1 = int(bits_of(offsets)[e]), int(bits_of(offsets)[e + 1])
            want = [u for u in range(n) if any(loc_idx[u, k] == e and so[u, k] >= 0 for k in range(K))]
            np.testing.assert_array_equal(rt[r0:r1], want)
            np.testing.assert_array_equal(xb[r0:r1], x[t0:t0 + n][want])
        t0 += n
    np.testing.assert_array_equal(np.concatenate(kept), ref.slot_of >= 0)
