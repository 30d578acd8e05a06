"""The token-sharded layer's exchange step on world-size 2 and 4 gloo ranks (CPU).

Each rank routes its own consecutive token range with the oracle, counts its picks per expert and
exchanges them (mixture_experts_layer_96_b300.sharded.queue_bases); a pick is kept iff its queue
base plus its place in the rank's own queue is below the whole batch's capacity. The ranks' keep
masks, concatenated in rank order, must equal the single-device oracle dispatch of the whole batch
bit for bit, and the all-reduced aux loss the single-device oracle's to 1e-12."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import oracle.moe_oracle as O  # noqa: E402
from mixture_experts_layer_96_b300 import sharded  # noqa: E402

CASES = {
    # T, h, E, K, CF, shard sizes, score, logit bias skew
    "softmax_drop": (240, 16, 8, 2, 0.9, [100, 140], "softmax"),
    "sigmoid_drop_4": (300, 16, 16, 3, 0.7, [37, 100, 63, 100], "sigmoid"),
    "nodrop_4": (200, 16, 8, 2, None, [50, 50, 50, 50], "softmax"),
}


def _problem(name):
    T, h, E, K, cf, shards, score = CASES[name]
    rng = np.random.default_rng(11)
    x = rng.normal(size=(T, h))
    wg = rng.normal(size=(h, E)) / np.sqrt(h)
    bias = -0.6 * np.log(np.arange(1, E + 1))  # skew towards low experts so capacity binds
    logits = O.router_logits(x, wg, bias)
    return T, E, K, cf, shards, score, logits


def _rank_main(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, E, K, cf, shards, score, logits = _problem(name)
        t0 = sum(shards[:rank])
        loc = logits[t0:t0 + shards[rank]]
        idx, _, _ = O.route(loc, score, K)
        d = O.dispatch(idx, E, None)                       # the rank's own queues, no capacity
        place = d.slot_of - d.offsets[idx]                 # place of each pick in its local queue
        counts = torch.tensor(d.counts, dtype=torch.int32)
        base, total = sharded.queue_bases(counts)
        C = O.capacity(cf, K, T, E)
        g = base.numpy().astype(np.int64)[idx] + place
        kept = np.ones_like(g, dtype=bool) if C is None else g < C
        psum = torch.tensor(O.routing_probs(loc, score).sum(axis=0))
        aux = sharded.aux_loss(counts, psum, T, K, 0.01)
        out[rank] = (kept, aux, total.numpy())
    finally:
        dist.destroy_process_group()


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("name", sorted(CASES))
def test_sharded_keep_masks_and_aux_equal_the_single_device_layer(name):
    T, E, K, cf, shards, score, logits = _problem(name)
    world = len(shards)
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _port(), name, out), nprocs=world, join=True)
    idx, _, _ = O.route(logits, score, K)
    ref = O.dispatch(idx, E, O.capacity(cf, K, T, E))
    kept = np.concatenate([out[r][0] for r in range(world)])
    np.testing.assert_array_equal(kept, ref.slot_of >= 0)
    if cf is not None:
        assert not kept.all()  # the capacity binds in these cases
    aux_ref = O.aux_loss(logits, idx, E, K, 0.01, score)
    for r in range(world):
        assert abs(out[r][1] - aux_ref) <= 1e-12 * abs(aux_ref)
        np.testing.assert_array_equal(out[r][2], ref.counts)
