"""Seeded synthetic inputs for the MoE FFN layer forward.

This module is shared by the tests, the benchmark and the smoke check. It holds the five workload
shapes and a seeded generator for their tensors, and nothing of the layer's arithmetic: no
routing, no scoring, no expert math. Both the CUDA path and the CPU oracle take their inputs from
here, so both see identical bits.

Recipe (every workload, seed 0 unless stated):
  x       ~ N(0, 1)                       [T][h]
  W_g     ~ N(0, 1/h')                    [h'][E]   (router, the pages' x·W_g orientation)
  W1, W3  ~ N(0, 1/h')                    [E][d_ff][h']   (gate and up projections, K-major)
  W2      ~ N(0, 1/d_ff)                  [E][h'][d_ff]   (down projection, K-major)
  select bias b ~ U(-0.1, 0.1)            [E]  (fine-grained sigmoid workload only)
  logit bias = Zipf(s=1.2) pmf over E     [E]  (skewed workload only)
bf16 workloads round every tensor above except the two biases to bf16 (round to nearest even)
once; the bits are what both sides consume. The fp32 workload keeps float32.

Determinism: every tensor is cut into fixed-size pieces, and piece j of tensor `tid` (for expert e)
draws from its own numpy PCG64 stream seeded with [seed, tid, e, j]. The result therefore does not
depend on how many threads generate it, and one expert's weights can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

__all__ = [
    "MoEShape", "WORKLOADS", "workload", "scaled", "Generator", "f32_to_bf16_bits",
    "bf16_bits_to_f32",
]

SCORE_SOFTMAX = "softmax"
SCORE_SIGMOID = "sigmoid"


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Shape and routing options of one MoE layer workload.

    T: tokens; h: token width (all heads); E: experts; K: experts per routed unit;
    d_ff: expert hidden width; n_heads: H > 1 splits each token into H sub-tokens of h/H;
    n_groups/topk_groups: group-limited Top-K (1/1 = off); capacity_factor: None = no drop;
    score: "softmax" or "sigmoid"; dtype: "bf16" or "f32"; select_bias: "uniform0.1" or None;
    logit_bias: "zipf1.2" or None; aux_alpha: weight of the auxiliary balance loss.
    """
    name: str
    T: int
    h: int
    E: int
    K: int
    d_ff: int
    score: str = SCORE_SOFTMAX
    dtype: str = "bf16"
    n_heads: int = 1
    n_groups: int = 1
    topk_groups: int = 1
    capacity_factor: Optional[float] = None
    select_bias: Optional[str] = None
    logit_bias: Optional[str] = None
    aux_alpha: float = 0.01

    @property
    def h_unit(self) -> int:
        """Width of one routed unit (h' = h / H)."""
        return self.h // self.n_heads

    @property
    def T_units(self) -> int:
        """Number of routed units (T' = T * H)."""
        return self.T * self.n_heads

    def describe(self) -> str:
        s = (f"{self.name}: T={self.T} h={self.h} E={self.E} K={self.K} d_ff={self.d_ff} "
             f"{self.score} {self.dtype}")
        if self.n_heads > 1:
            s += f" H={self.n_heads} (T'={self.T_units}, h'={self.h_unit})"
        if self.n_groups > 1:
            s += f" groups={self.n_groups} topk_groups={self.topk_groups}"
        s += f" CF={'inf' if self.capacity_factor is None else self.capacity_factor}"
        if self.select_bias:
            s += f" select_bias={self.select_bias}"
        if self.logit_bias:
            s += f" logit_bias={self.logit_bias}"
        return s


# The five workloads the layer is measured and checked on.
WORKLOADS = {
    "tiny_f32": MoEShape("tiny_f32", T=256, h=128, E=8, K=2, d_ff=256, dtype="f32",
                         capacity_factor=1.25),
    "mixtral_bf16": MoEShape("mixtral_bf16", T=4096, h=4096, E=8, K=2, d_ff=14336),
    "finegrained_bf16": MoEShape("finegrained_bf16", T=4096, h=7168, E=256, K=8, d_ff=2048,
                                 score=SCORE_SIGMOID, n_groups=8, topk_groups=4,
                                 select_bias="uniform0.1"),
    "skewed_bf16": MoEShape("skewed_bf16", T=16384, h=2048, E=64, K=2, d_ff=1408,
                            capacity_factor=1.25, logit_bias="zipf1.2"),
    "multihead_bf16": MoEShape("multihead_bf16", T=16384, h=2048, E=64, K=2, d_ff=1024,
                               n_heads=4),
}


def workload(name: str) -> MoEShape:
    return WORKLOADS[name]


def scaled(shape: MoEShape, **overrides) -> MoEShape:
    """A copy of `shape` with some fields replaced (smaller parity cases keep the recipe)."""
    d = dataclasses.asdict(shape)
    d.update(overrides)
    if "name" not in overrides:
        d["name"] = shape.name + "_" + "_".join(f"{k}{v}" for k, v in sorted(overrides.items()))
    return MoEShape(**d)


# ---------------------------------------------------------------------------------------------
# bf16 encoding (input encoding only; round to nearest even, finite inputs)

def f32_to_bf16_bits(a: np.ndarray, out: Optional[np.ndarray] = None) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    if out is None:
        return r.astype(np.uint16)
    out[...] = r
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------------------------
# generator

_TID_X, _TID_WG, _TID_W1, _TID_W3, _TID_W2, _TID_SB = 0, 1, 2, 3, 4, 5
_TID_DY = 6
_PIECE = 1 << 22  # elements per independent stream piece


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


class Generator:
    """Seeded tensors of one workload. Arrays are numpy: uint16 bf16 bits or float32."""

    def __init__(self, shape: MoEShape, seed: int = 0, threads: Optional[int] = None):
        self.shape = shape
        self.seed = seed
        self.threads = threads or _threads()

    # -- core: fill a [rows][cols] matrix from pieces of whole rows -------------------------
    def _fill(self, out: np.ndarray, tid: int, sub: int, std: float, bf16: bool,
              pool: Optional[ThreadPoolExecutor] = None) -> None:
        rows, cols = out.shape
        rpp = max(1, _PIECE // cols)
        pieces = [(j, j * rpp, min(rows, (j + 1) * rpp)) for j in range((rows + rpp - 1) // rpp)]

        def work(p):
            j, r0, r1 = p
            g = np.random.default_rng([self.seed, tid, sub, j])
            v = g.standard_normal((r1 - r0, cols), dtype=np.float32)
            if std != 1.0:
                v *= np.float32(std)
            if bf16:
                f32_to_bf16_bits(v, out=out[r0:r1])
            else:
                out[r0:r1] = v

        if pool is None and len(pieces) > 1 and self.threads > 1:
            with ThreadPoolExecutor(self.threads) as ex:
                list(ex.map(work, pieces))
        elif pool is not None:
            list(pool.map(work, pieces))
        else:
            for p in pieces:
                work(p)

    def _alloc(self, shape) -> np.ndarray:
        return np.empty(shape, dtype=np.uint16 if self.shape.dtype == "bf16" else np.float32)

    @property
    def bf16(self) -> bool:
        return self.shape.dtype == "bf16"

    def x(self, rows: Optional[slice] = None) -> np.ndarray:
        """Input tokens [T][h]. `rows` selects a token range without drawing the rest."""
        s = self.shape
        if rows is None:
            out = self._alloc((s.T, s.h))
            self._fill(out, _TID_X, 0, 1.0, self.bf16)
            return out
        # regenerate only the pieces that cover the requested rows
        rpp = max(1, _PIECE // s.h)
        r0, r1 = rows.start or 0, rows.stop if rows.stop is not None else s.T
        j0, j1 = r0 // rpp, (r1 - 1) // rpp
        out = self._alloc((r1 - r0, s.h))
        for j in range(j0, j1 + 1):
            a, b = j * rpp, min(s.T, (j + 1) * rpp)
            g = np.random.default_rng([self.seed, _TID_X, 0, j])
            v = g.standard_normal((b - a, s.h), dtype=np.float32)
            lo, hi = max(a, r0), min(b, r1)
            piece = v[lo - a:hi - a]
            out[lo - r0:hi - r0] = f32_to_bf16_bits(piece) if self.bf16 else piece
        return out

    def w_router(self) -> np.ndarray:
        """Router weight W_g [h'][E] ~ N(0, 1/h')."""
        s = self.shape
        out = self._alloc((s.h_unit, s.E))
        self._fill(out, _TID_WG, 0, 1.0 / math.sqrt(s.h_unit), self.bf16)
        return out

    def expert(self, e: int):
        """(W1_e [d_ff][h'], W3_e [d_ff][h'], W2_e [h'][d_ff]) for one expert."""
        s = self.shape
        w1 = self._alloc((s.d_ff, s.h_unit))
        w3 = self._alloc((s.d_ff, s.h_unit))
        w2 = self._alloc((s.h_unit, s.d_ff))
        self._fill(w1, _TID_W1, e, 1.0 / math.sqrt(s.h_unit), self.bf16)
        self._fill(w3, _TID_W3, e, 1.0 / math.sqrt(s.h_unit), self.bf16)
        self._fill(w2, _TID_W2, e, 1.0 / math.sqrt(s.d_ff), self.bf16)
        return w1, w3, w2

    def experts(self):
        """All experts stacked: W1, W3 [E][d_ff][h'], W2 [E][h'][d_ff] (threads over pieces)."""
        s = self.shape
        w1 = self._alloc((s.E, s.d_ff, s.h_unit))
        w3 = self._alloc((s.E, s.d_ff, s.h_unit))
        w2 = self._alloc((s.E, s.h_unit, s.d_ff))
        with ThreadPoolExecutor(self.threads) as pool:
            for e in range(s.E):
                self._fill(w1[e], _TID_W1, e, 1.0 / math.sqrt(s.h_unit), self.bf16, pool)
                self._fill(w3[e], _TID_W3, e, 1.0 / math.sqrt(s.h_unit), self.bf16, pool)
                self._fill(w2[e], _TID_W2, e, 1.0 / math.sqrt(s.d_ff), self.bf16, pool)
        return w1, w3, w2

    def select_bias(self) -> Optional[np.ndarray]:
        """Selection-only bias b ~ U(-0.1, 0.1) [E] float32, or None."""
        s = self.shape
        if s.select_bias is None:
            return None
        assert s.select_bias == "uniform0.1", s.select_bias
        g = np.random.default_rng([self.seed, _TID_SB, 0, 0])
        return g.uniform(-0.1, 0.1, size=s.E).astype(np.float32)

    def logit_bias(self) -> Optional[np.ndarray]:
        """Per-expert logit shift [E] float32 (Zipf(s=1.2) pmf, expert 0 hottest), or None."""
        s = self.shape
        if s.logit_bias is None:
            return None
        assert s.logit_bias == "zipf1.2", s.logit_bias
        ranks = np.arange(1, s.E + 1, dtype=np.float64)
        w = ranks ** -1.2
        return (w / w.sum()).astype(np.float32)

    def dy(self) -> np.ndarray:
        """Upstream gradient dL/dy [T][h] ~ N(0, 1), in the layer's dtype (for backward checks)."""
        s = self.shape
        out = self._alloc((s.T, s.h))
        self._fill(out, _TID_DY, 0, 1.0, self.bf16)
        return out

    def logits(self, scale: float = 1.0) -> np.ndarray:
        """Seeded fp32 router logits [T'][E] ~ N(0, scale^2), for routing-stage checks."""
        s = self.shape
        g = np.random.default_rng([self.seed, 100, 0, 0])
        return (g.standard_normal((s.T_units, s.E), dtype=np.float32) * np.float32(scale))

    def token_ids(self, vocab: int = 32000) -> np.ndarray:
        """Seeded token ids [T'] int32, uniform in [0, vocab) (the hash gate's input)."""
        s = self.shape
        g = np.random.default_rng([self.seed, 103, 0, 0])
        return g.integers(0, vocab, size=s.T_units, dtype=np.int64).astype(np.int32)

    def topk_idx(self) -> np.ndarray:
        """Seeded routing decisions [T'][K] int32 (K distinct experts per unit, Zipf-skewed),
        for dispatch-stage checks."""
        s = self.shape
        g = np.random.default_rng([self.seed, 101, 0, 0])
        p = np.arange(1, s.E + 1, dtype=np.float64) ** -1.2
        p /= p.sum()
        out = np.empty((s.T_units, s.K), dtype=np.int32)
        for t in range(s.T_units):
            out[t] = g.choice(s.E, size=s.K, replace=False, p=p)
        return out
