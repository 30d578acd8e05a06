"""Shared helpers of the parity tests: seeded workloads on the device and for the oracle, the
tolerances, and the bit-exact routing check on the GPU's own fp32 logits."""
from __future__ import annotations

import math
from contextlib import contextmanager
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import oracle.moe_oracle as O
from workloads import Generator, MoEShape, bf16_bits_to_f32

U32 = 2.0 ** -24  # unit roundoff of fp32


TILE_MODES = {  # name -> (pair_tiles, transposed_tails) for set_expert_gemm
    "single": (0, -1),
    "single_tails_transposed": (0, 1),
    "single_tails_plain": (0, 0),
    "pair": (1, -1),
    "pair_tails_transposed": (1, 1),
    "pair_tails_plain": (1, 0),
}


@contextmanager
def expert_tiles(mode: str, fold_combine: int = -1):
    """Force the expert GEMMs' tile shape (and the combine fold) for the duration (automatic again
    afterwards)."""
    from mixture_experts_layer_96_b300 import set_expert_gemm
    set_expert_gemm(*TILE_MODES[mode], fold_combine)
    try:
        yield mode
    finally:
        set_expert_gemm(-1, -1, -1)


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


def route_on_gpu_logits(inp: "Inputs", outs, exact_logits: Optional[np.ndarray] = None):
    """The routing check of a forward, bit for bit.

    1. The GPU's fp32 logits (logit bias included) lie within the rigorous fp32 error bound of the
       exact float64 logits.
    2. The oracle routes on those same fp32 logits: its picks must equal the GPU's for every unit
       (softmax keys are the logits themselves; sigmoid keys σ(l) + b are formed in float64 on
       both sides).

    Returns (gpu picks [T'][K] int64, oracle gates at those logits, the GPU logits as float64).
    """
    s = inp.shape
    gl = as_f64(outs.logits)
    if exact_logits is None:
        b = inp.bf16
        exact_logits = O.router_logits(O.split_heads(widen(inp.x, b), s.n_heads), widen(inp.w_g, b),
                                       inp.logit_bias)
    bound = inp.logit_error_bound()
    over = np.abs(gl - exact_logits) - bound
    assert (over <= 0).all(), f"GPU logits outside the fp32 error bound by {float(over.max()):.3e}"
    idx, gate, _ = O.route(gl, s.score, s.K, inp.select_bias, s.n_groups, s.topk_groups)
    gidx = bits_of(outs.topk_idx).astype(np.int64)
    bad = np.nonzero((gidx != idx).any(axis=1))[0]
    assert bad.size == 0, (f"{bad.size} of {s.T_units} units routed differently from the oracle on the same "
                           f"fp32 logits, e.g. unit {bad[0]}: GPU {gidx[bad[0]].tolist()} oracle {idx[bad[0]].tolist()}")
    return gidx, gate, gl
