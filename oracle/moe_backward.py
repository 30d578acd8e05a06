"""CPU oracle of the MoE FFN layer's backward pass (the gradient of the forward in moe_oracle).

TEST INFRASTRUCTURE, under the same rules as moe_oracle: only the tests, the smoke check and the
benchmark's CPU-baseline leg use it; the library never calls it and shares no code with it.

The pages train this layer (the speed-ups they quote are training speed-ups, [HAI] §"HAI-LLM 上的
使用"; [Lesson 10] §4 adds L_aux to the training loss) but print no backward formulas. The plain
reading, R14 in the design notes:

  The loss seen by the layer is L = <dy, y> + d_aux · L_aux, with dy the gradient arriving at
  the layer output and d_aux the weight of the aux term. The routing decisions (the Top-K picks,
  the group limit, the per-expert counts f_i and the capacity drops) are piecewise constant in the
  inputs and are held fixed; gradients flow through everything continuous: the gate values
  (softmax over the picked logits, or σ(l_i)/Σ_picked σ(l_j)), the expert FFNs, the routing
  probabilities P_i in L_aux, and the router GEMM. The selection-only bias b has no gradient.

Everything below is that calculus written out in float64, following the forward's steps in
reverse: combine → down projection → SwiGLU → gate/up projections → return to token order,
then gates → logits, L_aux → logits, and the router GEMM. Pins (tests/test_oracle_backward_pins.py):
central finite differences of the forward oracle with the routing held fixed, and the dense
special case E = K = 1 against torch.autograd of a plain SwiGLU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from .moe_oracle import (ExpertProvider, capacity, dispatch, expert_counts, gates, merge_heads,
                         route, router_logits, routing_probs, sigmoid, split_heads)


@dataclass
class Grads:
    dx: np.ndarray            # [T][h]
    dw_g: np.ndarray          # [h'][E]
    dw1: np.ndarray           # [E][d_ff][h']
    dw3: np.ndarray           # [E][d_ff][h']
    dw2: np.ndarray           # [E][h'][d_ff]
    dlogits: np.ndarray       # [T'][E]  dL/dl
    dgate: np.ndarray         # [T'][K]  dL/d gate (0 for dropped picks)
    idx: np.ndarray           # [T'][K]  the routing the gradient was taken at
    slot_of: np.ndarray       # [T'][K]


def gate_backward(l: np.ndarray, idx: np.ndarray, dgate: np.ndarray, score: str) -> np.ndarray:
    """dL/dl [T'][E] through the gate values of the picked experts.  [Lesson 10 §1; R1, R2, R14]

    softmax gates g = softmax(l_picked):       dl_picked = g ⊙ (dg − Σ_k g_k dg_k)
    sigmoid gates g = s/Σ s, s = σ(l_picked):  ds = (dg − Σ_k g_k dg_k)/Σ s,  dl_picked = ds ⊙ s(1−s)
    """
    T, E = l.shape
    g = gates(l, idx, score)
    inner = np.sum(g * dgate, axis=1, keepdims=True)
    if score == "softmax":
        dlp = g * (dgate - inner)
    else:
        s = sigmoid(np.take_along_axis(np.asarray(l, np.float64), idx.astype(np.int64), axis=1))
        dlp = (dgate - inner) / s.sum(axis=1, keepdims=True) * s * (1.0 - s)
    dl = np.zeros((T, E), dtype=np.float64)
    rows = np.repeat(np.arange(T), idx.shape[1])
    np.add.at(dl, (rows, idx.reshape(-1).astype(np.int64)), dlp.reshape(-1))
    return dl


def aux_backward(l: np.ndarray, idx: np.ndarray, E: int, K: int, alpha: float, score: str,
                 d_aux: float) -> np.ndarray:
    """dL/dl [T'][E] of d_aux · α·E·Σ_i f_i·P_i with f held fixed.  [Lesson 10 §4; R7, R14]

    P_i = mean_t p[t,i], so dL/dp[t,i] = d_aux·α·E·f_i/T'. Then through p = softmax(l) (or
    p = s/Σ s with s = σ(l) over all E experts).
    """
    T = l.shape[0]
    f = expert_counts(idx, E) / float(T * K)
    dp = np.broadcast_to(d_aux * alpha * E * f[None, :] / T, (T, E))
    p = routing_probs(l, score)
    inner = np.sum(p * dp, axis=1, keepdims=True)
    if score == "softmax":
        return p * (dp - inner)
    s = sigmoid(l)
    return (dp - inner) / s.sum(axis=1, keepdims=True) * s * (1.0 - s)


def backward(x: np.ndarray, w_g: np.ndarray, experts: ExpertProvider, dy: np.ndarray, d_aux: float = 1.0,
             *, E: int, K: int, d_ff: int, score: str = "softmax", n_heads: int = 1, n_groups: int = 1,
             topk_groups: int = 1, capacity_factor: Optional[float] = None, aux_alpha: float = 0.01,
             logit_bias=None, select_bias=None, idx_override: Optional[np.ndarray] = None) -> Grads:
    """Gradients of L = <dy, y> + d_aux·L_aux with respect to x, W_g, W1, W3, W2.  [R14]

    x, dy: [T][h] float64; w_g: [h'][E]; experts(e) → (w1 [d_ff][h'], w3, w2 [h'][d_ff]).
    idx_override: take the gradient at these picks (as the forward does with it).
    """
    xu = split_heads(np.asarray(x, np.float64), n_heads)
    dyu = split_heads(np.asarray(dy, np.float64), n_heads)
    Tu, hu = xu.shape
    l = router_logits(xu, w_g, logit_bias)
    idx, g, _ = route(l, score, K, select_bias, n_groups, topk_groups)
    if idx_override is not None:
        idx = np.asarray(idx_override, np.int32)
        g = gates(l, idx, score)
    d = dispatch(idx, E, capacity(capacity_factor, K, Tu, E))

    dxu = np.zeros_like(xu)
    dgate = np.zeros((Tu, K), dtype=np.float64)
    dw1 = np.zeros((E, d_ff, hu)); dw3 = np.zeros((E, d_ff, hu)); dw2 = np.zeros((E, hu, d_ff))
    # the pick (t, k) behind each packed row
    pick_t = np.full(Tu * K, -1, dtype=np.int64)
    pick_k = np.full(Tu * K, -1, dtype=np.int64)
    for t in range(Tu):
        for k in range(K):
            r = d.slot_of[t, k]
            if r >= 0:
                pick_t[r], pick_k[r] = t, k
    for e in range(E):
        r0, r1 = int(d.offsets[e]), int(d.offsets[e + 1])
        if r1 == r0:
            continue
        w1, w3, w2 = experts(e)
        tok, kk = pick_t[r0:r1], pick_k[r0:r1]
        X = xu[tok]
        G = X @ w1.T
        U = X @ w3.T
        sig = sigmoid(G)
        S = G * sig                      # silu(G)
        H = S * U
        Yp = H @ w2.T
        # combine: y[t] += g[t,k]·Yp[r]
        dYp = g[tok, kk][:, None] * dyu[tok]
        dgate[tok, kk] = np.sum(dyu[tok] * Yp, axis=1)
        # down projection Yp = H·W2ᵀ
        dw2[e] = dYp.T @ H
        dH = dYp @ w2
        # SwiGLU H = silu(G) ⊙ U, silu'(G) = σ(G)·(1 + G·(1 − σ(G)))
        dG = dH * U * (sig * (1.0 + G * (1.0 - sig)))
        dU = dH * S
        # gate/up projections G = X·W1ᵀ, U = X·W3ᵀ
        dw1[e] = dG.T @ X
        dw3[e] = dU.T @ X
        np.add.at(dxu, tok, dG @ w1 + dU @ w3)
    dl = gate_backward(l, idx, dgate, score) + aux_backward(l, idx, E, K, aux_alpha, score, d_aux)
    # router l = x·W_g (+ logit bias)
    dw_g = xu.T @ dl
    dxu = dxu + dl @ np.asarray(w_g, np.float64).T
    return Grads(merge_heads(dxu, n_heads), dw_g, dw1, dw3, dw2, dl, dgate, idx, d.slot_of)


def backward_entries(x: np.ndarray, w_g: np.ndarray, experts: ExpertProvider, dy: np.ndarray, d_aux: float,
                     idx: np.ndarray, *, E: int, K: int, score: str = "softmax", n_heads: int = 1,
                     capacity_factor: Optional[float] = None, aux_alpha: float = 0.01, logit_bias=None,
                     units=(), dw2_at=(), dw1_at=(), dw3_at=()) -> dict:
    """Selected entries of the same gradients as `backward`, each computed from its definition,
    for layers too large to differentiate whole.  [R14]

    Routing at the picks `idx`. units: unit indices whose dgate [K], dlogits [E] and dx rows [h']
    are returned; dw2_at (e, j, f), dw1_at / dw3_at (e, f, i): weight-gradient entries.
    """
    xu = split_heads(np.asarray(x, np.float64), n_heads)
    dyu = split_heads(np.asarray(dy, np.float64), n_heads)
    Tu, hu = xu.shape
    idx = np.asarray(idx, np.int64)
    l = router_logits(xu, w_g, logit_bias)
    g = gates(l, idx, score)
    d = dispatch(idx, E, capacity(capacity_factor, K, Tu, E))
    dl_aux = aux_backward(l, idx, E, K, aux_alpha, score, d_aux)
    rows_of = {}
    for t in range(Tu):
        for k in range(K):
            if d.slot_of[t, k] >= 0:
                rows_of.setdefault(int(idx[t, k]), []).append((t, k))
    need = set(e for e, _, _ in list(dw2_at) + list(dw1_at) + list(dw3_at))
    for u in units:
        need.update(int(idx[u, k]) for k in range(K) if d.slot_of[u, k] >= 0)
    out = {"dgate": {}, "dlogits": {}, "dx": {}, "dw2": {}, "dw1": {}, "dw3": {}}
    dxp = {}  # (t, k) → dX_packed row
    for e in sorted(need):
        w1, w3, w2 = experts(e)
        picks = rows_of.get(e, [])
        if picks:
            tok = np.array([t for t, _ in picks]); kk = np.array([k for _, k in picks])
            X = xu[tok]
            dY = g[tok, kk][:, None] * dyu[tok]
        for (ee, j, f) in dw2_at:
            if ee == e:
                if not picks:
                    out["dw2"][(e, j, f)] = 0.0
                    continue
                G, U = X @ w1[f], X @ w3[f]
                out["dw2"][(e, j, f)] = float(np.sum(dY[:, j] * (G * sigmoid(G) * U)))
        for key, which in (("dw1", dw1_at), ("dw3", dw3_at)):
            for (ee, f, i) in which:
                if ee != e:
                    continue
                if not picks:
                    out[key][(e, f, i)] = 0.0
                    continue
                G, U = X @ w1[f], X @ w3[f]
                sg = sigmoid(G)
                dH = dY @ w2[:, f]
                dcol = dH * U * sg * (1.0 + G * (1.0 - sg)) if key == "dw1" else dH * G * sg
                out[key][(e, f, i)] = float(np.sum(dcol * X[:, i]))
        for u in units:
            for k in range(K):
                if int(idx[u, k]) != e or d.slot_of[u, k] < 0:
                    continue
                xt = xu[u]
                G, U = w1 @ xt, w3 @ xt
                sg = sigmoid(G)
                S = G * sg
                yk = w2 @ (S * U)
                out["dgate"][(u, k)] = float(np.dot(dyu[u], yk))
                dYr = g[u, k] * dyu[u]
                dH = dYr @ w2
                dG = dH * U * sg * (1.0 + G * (1.0 - sg))
                dU = dH * S
                dxp[(u, k)] = dG @ w1 + dU @ w3
    for u in units:
        dg = np.array([out["dgate"].get((u, k), 0.0) for k in range(K)])
        dl_u = gate_backward(l[u:u + 1], idx[u:u + 1], dg[None, :], score)[0] + dl_aux[u]
        out["dlogits"][u] = dl_u
        dx = dl_u @ np.asarray(w_g, np.float64).T
        for k in range(K):
            if (u, k) in dxp:
                dx = dx + dxp[(u, k)]
        out["dgate"].update({(u, k): float(dg[k]) for k in range(K)})
        out["dx"][u] = dx
    return out
