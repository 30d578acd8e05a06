"""Shared helpers of the parity tests: seeded workloads on the device and for the oracle, the
tolerances, and the near-tie analysis of routing decisions made on differently rounded logits."""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import oracle.moe_oracle as O
from workloads import Generator, MoEShape, bf16_bits_to_f32

U32 = 2.0 ** -24  # unit roundoff of fp32


def config_of(shape: MoEShape):
    from mixture_experts_layer_96_b300 import make_config
    return make_config(shape.T, shape.h, shape.E, shape.K, shape.d_ff, n_heads=shape.n_heads,
                       n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                       capacity_factor=shape.capacity_factor, aux_alpha=shape.aux_alpha,
                       score=shape.score, dtype=shape.dtype)


def to_device(a: np.ndarray, bf16: bool, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if bf16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def widen(a: np.ndarray, bf16: bool) -> np.ndarray:
    return bf16_bits_to_f32(a).astype(np.float64) if bf16 else np.asarray(a, np.float64)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """Device tensor → numpy (bf16 as uint16 bits, else its own dtype)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


@dataclass
class Inputs:
    shape: MoEShape
    x: np.ndarray
    w_g: np.ndarray
    w1: np.ndarray
    w3: np.ndarray
    w2: np.ndarray
    logit_bias: Optional[np.ndarray]
    select_bias: Optional[np.ndarray]

    @staticmethod
    def make(shape: MoEShape, seed: int = 0) -> "Inputs":
        g = Generator(shape, seed)
        w1, w3, w2 = g.experts()
        return Inputs(shape, g.x(), g.w_router(), w1, w3, w2, g.logit_bias(), g.select_bias())

    @property
    def bf16(self) -> bool:
        return self.shape.dtype == "bf16"

    def device(self):
        from mixture_experts_layer_96_b300 import LayerWeights
        b = self.bf16
        x = to_device(self.x, b)
        lw = LayerWeights(to_device(self.w_g, b), to_device(self.w1, b), to_device(self.w3, b),
                          to_device(self.w2, b),
                          None if self.logit_bias is None else torch.from_numpy(self.logit_bias).cuda(),
                          None if self.select_bias is None else torch.from_numpy(self.select_bias).cuda())
        return x, lw

    def oracle_forward(self, sample_units=None, idx_override=None):
        s = self.shape
        b = self.bf16
        W1, W3, W2 = self.w1, self.w3, self.w2
        return O.forward(widen(self.x, b), widen(self.w_g, b),
                         lambda e: (widen(W1[e], b), widen(W3[e], b), widen(W2[e], b)),
                         E=s.E, K=s.K, score=s.score, n_heads=s.n_heads, n_groups=s.n_groups,
                         topk_groups=s.topk_groups, capacity_factor=s.capacity_factor,
                         aux_alpha=s.aux_alpha, logit_bias=self.logit_bias, select_bias=self.select_bias,
                         sample_units=sample_units, idx_override=idx_override)

    def logit_error_bound(self) -> np.ndarray:
        """Per (unit, expert) bound on |fp32 logit − exact|: first-order error of an fp32 sum of
        h' products in any order (bf16 products are exact; tensor-core adds are allowed twice the
        round-to-nearest error), plus the rounding of the bias add and of the result."""
        b = self.bf16
        s = self.shape
        xa = np.abs(O.split_heads(widen(self.x, b), s.n_heads))
        wa = np.abs(widen(self.w_g, b))
        dot = xa @ wa
        l = O.router_logits(O.split_heads(widen(self.x, b), s.n_heads), widen(self.w_g, b), self.logit_bias)
        if b:  # tensor-core accumulation: allow two roundings' worth per add (truncating adders)
            return 2 * (s.h_unit + 2) * U32 * dot + 2 * U32 * np.abs(l)
        # fp32 FMA chains: one rounding per add (products are fused)
        return (s.h_unit + 2) * U32 * dot + 2 * U32 * np.abs(l)


def tol_ok(got: np.ndarray, ref: np.ndarray, dtype: str):
    """The layer's float bar: bf16 max|y−ref| <= 1e-2·max|ref| + 1e-3; fp32 <= 1e-5·max|ref|."""
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    bound = 1e-2 * scale + 1e-3 if dtype == "bf16" else 1e-5 * scale
    return err <= bound, err, bound


def routing_margins(keys: np.ndarray, idx: np.ndarray, n_groups: int, topk_groups: int) -> np.ndarray:
    """Per unit, the smallest gap between a decision's winner and loser in the oracle's keys:
    the K-th vs (K+1)-th eligible key, and (group limit) the last kept vs first dropped group score."""
    T, E = keys.shape
    K = idx.shape[1]
    elig = O.group_limit(keys, n_groups, topk_groups)
    kk = np.where(elig, keys, -np.inf)
    srt = -np.sort(-kk, axis=1)
    m = srt[:, K - 1] - (srt[:, K] if K < E else -np.inf)
    if n_groups > 1:
        gs = E // n_groups
        top = -np.sort(-keys.reshape(T, n_groups, gs), axis=2)
        score = top[:, :, 0] + (top[:, :, 1] if gs > 1 else 0)
        gsrt = -np.sort(-score, axis=1)
        gm = gsrt[:, topk_groups - 1] - (gsrt[:, topk_groups] if topk_groups < n_groups else -np.inf)
        m = np.minimum(m, gm)
    return m


def check_routing(gpu_idx: np.ndarray, ref_idx: np.ndarray, keys: np.ndarray, key_err: np.ndarray,
                  shape: MoEShape):
    """Exact where the oracle's decision margin exceeds twice the key error (per unit, twice for
    group scores); elsewhere the GPU's picks must be a valid near-optimal choice.
    Returns (n_ambiguous, n_differ)."""
    E, K = shape.E, shape.K
    margin = routing_margins(keys, ref_idx, shape.n_groups, shape.topk_groups)
    slack = 4.0 * key_err.max(axis=1)
    amb = margin <= slack
    same = (gpu_idx == ref_idx).all(axis=1)
    bad_robust = np.nonzero(~amb & ~same)[0]
    assert bad_robust.size == 0, f"routing differs on units with a clear margin: {bad_robust[:10]}"
    n_differ = int((~same).sum())
    for u in np.nonzero(~same)[0]:
        g = gpu_idx[u]
        assert len(set(g.tolist())) == K and g.min() >= 0 and g.max() < E
        if shape.n_groups > 1:
            assert len({int(e) // (E // shape.n_groups) for e in g}) <= shape.topk_groups
        assert keys[u, g].sum() >= keys[u, ref_idx[u]].sum() - 2 * K * slack[u]
    return int(amb.sum()), n_differ
