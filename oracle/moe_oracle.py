"""CPU oracle of the single-GPU MoE FFN layer forward.

TEST INFRASTRUCTURE. Only the tests, the smoke check (`__graft_entry__.smoke`) and the
benchmark's CPU-baseline leg import this module. The library's forward path never calls it and
shares no code with it: this file imports numpy and nothing of the CUDA library.

It is a plain, slow, obviously correct restatement of what the layer computes, in float64, with
no blocking, fusion or reordering beyond the definitions below. Sources, by page title and section:

  [Lesson 10] "第 10 课：专家并行 EP" (Lesson 10: Expert Parallelism):
          §1 (router x·W_g; s(x) = Softmax(TopK(x·W_g, K)) or sigmoid; y = Σ_{i∈TopK} s_i(x)·FFN_i(x)),
          §3 (pack per expert, local grouped GEMM, return to source order, gate-weighted sum;
              communication volume 2·Tokens·K·h·sizeof(dtype)),
          §4 (aux loss L_aux = α·E·Σ f_i·P_i; capacity C = CF·K·T/E, overflow tokens dropped),
          §5 (node-limited routing: a token's K experts lie in at most M node groups),
          worked example (expert→rank placement, per-rank load, imbalance, utilisation).
  [HAI]   "HAI-LLM MoE：一键实现大模型的混合专家并行训练", §"HAI-LLM 上的使用" (alpha=0.01, top_k).
  [CH10]  "Chương 10: Song song MoE", §4 (aux-loss-free balancing by a per-expert bias).
  [MHL]   "Multi-Head LatentMoE 与 Head 并行", §摘要 and 评论 §1 (input split into heads, each
          head routed independently).

Readings where the pages are silent (the same list is kept in the design notes):
  R1 Softmax(TopK(l)) = softmax over the K picked logits; selection ranks logits directly.
  R2 Sigmoid scoring ranks σ(l)+b (b: selection-only bias); gates σ(l_i)/Σ_picked σ(l_j) use the
     unbiased score; keys are formed in float64.
  R3 Group limit: E experts in n_groups contiguous groups; group score = sum of the group's two
     largest keys; keep the topk_groups best groups; Top-K among their experts.
  R4 Ties (keys or group scores) go to the lower index.
  R5 C = ceil(CF·K·T'/E) evaluated in float64 from the given CF; CF None/<=0/inf = no drop.
  R6 Drop order: a unit's K picks are distinct, so within an expert the queue is token order; a
     pick whose rank in its expert's queue is >= C is dropped and contributes 0 (no re-norm).
  R7 f_i = pre-drop count_i/(T'·K); P_i = mean over units of the full softmax over all E logits
     (sigmoid: σ_i/Σ_j σ_j); logit biases are part of the logits.
  R8 Expert FFN = SwiGLU without biases: W2·(silu(W1 x) ⊙ W3 x), silu(z) = z/(1+e^{-z}).
  R9 Multi-head: x[T][H·h'] is read as T·H sub-tokens x[t·H+j] = x[t, j·h':(j+1)·h'], each routed
     and computed alone with one shared router and expert pool; y is read back the same way.
  R10 Routing from given fp32 logits: a logit bias is added in fp32 (the decision precision).
  R16 Hash gate: expert = fmix32(token id) mod E (MurmurHash3's finalizer), gate 1, top-1, no aux
     loss (no routing probabilities); capacity as for any gate.

Parity pins (tests/test_oracle_pins.py): brute-force Top-K and group limit on tiny inputs, a
brute-force O(T^2) capacity rank, closed forms (aux = α under uniform routing, softmax-over-picks
= renormalised full softmax), the dense special cases (E=1,K=1 SwiGLU against torch; K=E dense
mixture), head-split equivalence, permutation equivariance and the pages' worked example.
No function here is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np

# ---------------------------------------------------------------------------------------------
# encoding helpers (input widening only)


def widen(a: np.ndarray, bf16: bool) -> np.ndarray:
    """bf16 bits (uint16) or float32 → float64 (exact)."""
    if bf16:
        return (np.asarray(a, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------------------------
# [Lesson 10 §1] router


def router_logits(x: np.ndarray, w_g: np.ndarray, logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """l = x·W_g (+ per-expert logit bias), float64.  [Lesson 10 §1: x ∈ R^h, affinity x·W_g]

    x: [T'][h'] float64, w_g: [h'][E] float64 → [T'][E].
    """
    l = x @ w_g
    if logit_bias is not None:
        l = l + np.asarray(logit_bias, np.float64)[None, :]
    return l


def logits_with_bias_f32(logits_f32: np.ndarray, logit_bias: Optional[np.ndarray]) -> np.ndarray:
    """R10: fp32 logits plus a fp32 logit bias, added in fp32 (the decision precision)."""
    l = np.asarray(logits_f32, np.float32)
    if logit_bias is not None:
        l = (l + np.asarray(logit_bias, np.float32)[None, :]).astype(np.float32)
    return l


def sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))


def selection_keys(l: np.ndarray, score: str, select_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Keys that Top-K ranks, float64.  [Lesson 10 §1; CH10 §4; R1, R2]

    softmax: TopK acts on x·W_g itself, so the key is the logit.
    sigmoid: key = σ(l) + b, b the selection-only bias (zero if absent).
    """
    l = np.asarray(l, np.float64)
    if score == "softmax":
        return l.copy()
    if score == "sigmoid":
        k = sigmoid(l)
        if select_bias is not None:
            k = k + np.asarray(select_bias, np.float64)[None, :]
        return k
    raise ValueError(score)


# ---------------------------------------------------------------------------------------------
# [Lesson 10 §5] group limit, [Lesson 10 §1] Top-K


def group_limit(keys: np.ndarray, n_groups: int, topk_groups: int) -> np.ndarray:
    """Eligibility mask [T'][E] of the experts in each unit's topk_groups best groups.  [Lesson 10 §5; R3, R4]

    Groups are contiguous blocks of E/n_groups experts. A group's score is the sum of its two
    largest keys (its one key if the group has a single expert).
    """
    T, E = keys.shape
    if n_groups <= 1:
        return np.ones((T, E), dtype=bool)
    gs = E // n_groups
    assert gs * n_groups == E
    g = keys.reshape(T, n_groups, gs)
    top = np.sort(g, axis=2)[:, :, ::-1]
    score = top[:, :, 0] + (top[:, :, 1] if gs > 1 else 0.0)
    # rank groups by (score desc, group index asc): a stable sort of -score keeps index order
    order = np.argsort(-score, axis=1, kind="stable")
    chosen = np.zeros((T, n_groups), dtype=bool)
    np.put_along_axis(chosen, order[:, :topk_groups], True, axis=1)
    return np.repeat(chosen, gs, axis=1)


def topk(keys: np.ndarray, K: int, eligible: Optional[np.ndarray] = None) -> np.ndarray:
    """Indices [T'][K] int32 of the K largest eligible keys, in (key desc, index asc) order.  [Lesson 10 §1; R4]"""
    T, E = keys.shape
    if np.isnan(keys).any():
        raise ValueError("NaN key")
    if eligible is None:
        eligible = np.ones((T, E), dtype=bool)
    idx = np.broadcast_to(np.arange(E), (T, E))
    # np.lexsort: last key is primary → eligible first, then key desc, then index asc
    order = np.lexsort((idx, -keys, ~eligible), axis=1)
    out = order[:, :K].astype(np.int32)
    if not np.take_along_axis(eligible, out, axis=1).all():
        raise ValueError("fewer than K eligible experts")
    return out


def gates(l: np.ndarray, idx: np.ndarray, score: str) -> np.ndarray:
    """Gate weights [T'][K] float64 of the picked experts.  [Lesson 10 §1; R1, R2]

    softmax: Softmax(TopK(l, K)) — softmax over the K picked logits.
    sigmoid: σ(l_i) / Σ_{j picked} σ(l_j), unbiased scores.
    """
    lp = np.take_along_axis(np.asarray(l, np.float64), idx.astype(np.int64), axis=1)
    if score == "softmax":
        z = np.exp(lp - lp.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    s = sigmoid(lp)
    return s / s.sum(axis=1, keepdims=True)


def route(l: np.ndarray, score: str, K: int, select_bias=None, n_groups: int = 1, topk_groups: int = 1):
    """(idx [T'][K] int32, gate [T'][K] float64, keys [T'][E]) from logits.  [Lesson 10 §1, §5]"""
    keys = selection_keys(l, score, select_bias)
    elig = group_limit(keys, n_groups, topk_groups)
    idx = topk(keys, K, elig)
    return idx, gates(l, idx, score), keys


# ---------------------------------------------------------------------------------------------
# [Lesson 10 §4] aux loss and capacity


def expert_counts(idx: np.ndarray, E: int) -> np.ndarray:
    """Pre-drop per-expert counts [E] int64 (how many units picked each expert)."""
    return np.bincount(idx.reshape(-1).astype(np.int64), minlength=E)


def routing_probs(l: np.ndarray, score: str) -> np.ndarray:
    """Per-unit probabilities over all E experts, float64.  [Lesson 10 §4: P_i; R7]"""
    l = np.asarray(l, np.float64)
    if score == "softmax":
        z = np.exp(l - l.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    s = sigmoid(l)
    return s / s.sum(axis=1, keepdims=True)


def aux_loss(l: np.ndarray, idx: np.ndarray, E: int, K: int, alpha: float, score: str) -> float:
    """L_aux = α·E·Σ_i f_i·P_i.  [Lesson 10 §4; HAI alpha=0.01; R7]

    f_i = count_i/(T'·K) from the pre-drop picks; P_i = mean over units of the unit's probability
    of expert i.
    """
    T = l.shape[0]
    f = expert_counts(idx, E) / float(T * K)
    P = routing_probs(l, score).mean(axis=0)
    return float(alpha * E * np.sum(f * P))


def capacity(capacity_factor: Optional[float], K: int, T_units: int, E: int) -> Optional[int]:
    """C = ceil(CF·K·T'/E), or None for no drop.  [Lesson 10 §4; R5]"""
    if capacity_factor is None or not (capacity_factor > 0) or math.isinf(capacity_factor):
        return None
    return int(math.ceil(float(capacity_factor) * K * T_units / E))


# ---------------------------------------------------------------------------------------------
# [Lesson 10 §3 step 1] dispatch: pack units per expert, with the capacity drop of [Lesson 10 §4]


@dataclass
class Dispatch:
    counts: np.ndarray      # [E] pre-drop picks per expert
    kept: np.ndarray        # [E] n_e = min(count, C)
    offsets: np.ndarray     # [E+1] exclusive scan of kept
    slot_of: np.ndarray     # [T'][K] packed row of pick (t,k), -1 if dropped
    row_token: np.ndarray   # [T'·K] source unit of packed row r, -1 past the kept rows


def dispatch(idx: np.ndarray, E: int, C: Optional[int]) -> Dispatch:
    """Per-expert queues in token order; picks past the capacity are dropped.  [Lesson 10 §3, §4; R6]

    A sequential walk: units in order t = 0..T'-1, each unit's picks k = 0..K-1; the pick takes the
    next place in its expert's queue and is kept if that place is < C.
    """
    T, K = idx.shape
    rank = np.zeros((T, K), dtype=np.int64)
    queue = [0] * E
    for t in range(T):
        for k in range(K):
            e = int(idx[t, k])
            rank[t, k] = queue[e]
            queue[e] += 1
    counts = np.array(queue, dtype=np.int64)
    kept = counts if C is None else np.minimum(counts, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    slot_of = np.full((T, K), -1, dtype=np.int64)
    row_token = np.full(T * K, -1, dtype=np.int64)
    for t in range(T):
        for k in range(K):
            e = int(idx[t, k])
            if C is None or rank[t, k] < C:
                r = offsets[e] + rank[t, k]
                slot_of[t, k] = r
                row_token[r] = t
    return Dispatch(counts, kept, offsets, slot_of, row_token)


def comm_volume_bytes(tokens: int, K: int, h: int, sizeof: int) -> int:
    """Bytes moved by dispatch + combine of one layer step: 2·Tokens·K·h·sizeof.  [Lesson 10 §3]"""
    return 2 * tokens * K * h * sizeof


# ---------------------------------------------------------------------------------------------
# [Lesson 10 §3 step 2] expert FFN (SwiGLU, R8)


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def expert_ffn(xe: np.ndarray, w1: np.ndarray, w3: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """FFN_e(x) = W2·(silu(W1·x) ⊙ W3·x) for rows xe [n][h'], float64.  [Lesson 10 §1 FFN_i; R8]

    w1, w3: [d_ff][h']; w2: [h'][d_ff].
    """
    return (silu(xe @ w1.T) * (xe @ w3.T)) @ w2.T


# ---------------------------------------------------------------------------------------------
# [Lesson 10 §3 steps 3-4] combine


def combine(y_packed: np.ndarray, slot_of: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """y[t] = Σ_k gate[t,k]·y_packed[slot_of[t,k]] over kept picks.  [Lesson 10 §1 y = Σ s_i·FFN_i; §3 step 4]"""
    T, K = slot_of.shape
    y = np.zeros((T, y_packed.shape[1]), dtype=np.float64)
    for k in range(K):
        s = slot_of[:, k]
        m = s >= 0
        y[m] += gate[m, k][:, None] * y_packed[s[m]]
    return y


# ---------------------------------------------------------------------------------------------
# [MHL §摘要] head view


def split_heads(x: np.ndarray, n_heads: int) -> np.ndarray:
    """x [T][H·h'] → sub-tokens [T·H][h'], sub-token t·H+j = x[t, j·h':(j+1)·h'].  [MHL; R9]"""
    T, h = x.shape
    return x.reshape(T * n_heads, h // n_heads)


def merge_heads(y: np.ndarray, n_heads: int) -> np.ndarray:
    Tu, hu = y.shape
    return y.reshape(Tu // n_heads, hu * n_heads)


# ---------------------------------------------------------------------------------------------
# the whole layer


@dataclass
class Result:
    logits: np.ndarray
    idx: np.ndarray
    gate: np.ndarray
    keys: np.ndarray
    dispatch: Dispatch
    aux: float
    C: Optional[int]
    y: Optional[np.ndarray]           # [T][h] (all units) or None
    y_units: Optional[dict] = None    # unit → [h'] row, when only a sample was computed


ExpertProvider = Callable[[int], tuple]  # e → (w1 [d_ff][h'], w3, w2 [h'][d_ff]) float64


def forward(x: np.ndarray, w_g: np.ndarray, experts: ExpertProvider, *, E: int, K: int,
            score: str = "softmax", n_heads: int = 1, n_groups: int = 1, topk_groups: int = 1,
            capacity_factor: Optional[float] = None, aux_alpha: float = 0.01,
            logit_bias=None, select_bias=None, sample_units: Optional[np.ndarray] = None,
            idx_override: Optional[np.ndarray] = None) -> Result:
    """The layer: router → scores → (group limit) → Top-K → gates → capacity drop → pack →
    expert SwiGLU → gate-weighted combine back to token order, plus the aux loss.  [Lesson 10 §1, §3, §4, §5; MHL]

    x: [T][h] float64; w_g: [h'][E] float64; experts(e) gives expert e's float64 weights.
    sample_units: compute y only for these units (the routing and the queues still cover all
    units, since capacity is global); y_units then maps unit → output row.
    idx_override: route with these picks instead of the oracle's own (used only after the
    caller has checked that they are a valid Top-K under a stated tie window).
    """
    xu = split_heads(x, n_heads)
    Tu = xu.shape[0]
    l = router_logits(xu, w_g, logit_bias)
    idx, g, keys = route(l, score, K, select_bias, n_groups, topk_groups)
    if idx_override is not None:
        idx = np.asarray(idx_override, np.int32)
        g = gates(l, idx, score)
    C = capacity(capacity_factor, K, Tu, E)
    d = dispatch(idx, E, C)
    aux = aux_loss(l, idx, E, K, aux_alpha, score)

    if sample_units is None:
        yp = np.zeros((Tu * K, xu.shape[1]), dtype=np.float64)
        for e in range(E):
            r0, r1 = int(d.offsets[e]), int(d.offsets[e + 1])
            if r1 > r0:
                w1, w3, w2 = experts(e)
                yp[r0:r1] = expert_ffn(xu[d.row_token[r0:r1]], w1, w3, w2)
        y = merge_heads(combine(yp, d.slot_of, g), n_heads)
        return Result(l, idx, g, keys, d, aux, C, y)

    # sampled: y_u = Σ_k kept gate·FFN_{idx[u,k]}(x_u), grouped by expert to widen each once
    units = np.asarray(sample_units, dtype=np.int64)
    acc = {int(u): np.zeros(xu.shape[1]) for u in units}
    need = {}
    for u in units:
        for k in range(K):
            if d.slot_of[u, k] >= 0:
                need.setdefault(int(idx[u, k]), []).append((int(u), k))
    for e, pairs in sorted(need.items()):
        w1, w3, w2 = experts(e)
        rows = np.stack([xu[u] for u, _ in pairs])
        out = expert_ffn(rows, w1, w3, w2)
        for (u, k), o in zip(pairs, out):
            acc[u] += g[u, k] * o
    return Result(l, idx, g, keys, d, aux, C, None, acc)


# ---------------------------------------------------------------------------------------------
# [HAI §"HAI-LLM 上的使用"] hash gate (HashGate: top_k == 1 only). The page names the gate and its
# top-1 limit and nothing more. Reading R16: a hash gate has no learned router; unit u goes to
# expert fmix32(token_id_u) mod E with gate 1, where fmix32 is MurmurHash3's 32-bit finalizer (a
# published integer mix, Austin Appleby, public domain). No router means no routing
# probabilities, so the aux loss is 0. Capacity and drops are as for any gate.


def fmix32(h: int) -> int:
    """MurmurHash3's finalizer of a 32-bit value: xor-shift 16, multiply by 0x85ebca6b, xor-shift 13,
    multiply by 0xc2b2ae35, xor-shift 16 (all mod 2^32)."""
    h &= 0xFFFFFFFF
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h


def hash_route(token_ids: np.ndarray, E: int):
    """(idx [T'][1] int32, gate [T'][1] float64 of ones) for the hash gate.  [HAI; R16]

    token_ids: [T'] integers; each is taken as its 32-bit two's-complement pattern."""
    ids = np.asarray(token_ids).reshape(-1)
    idx = np.array([fmix32(int(t) & 0xFFFFFFFF) % E for t in ids], dtype=np.int32).reshape(-1, 1)
    return idx, np.ones(idx.shape, dtype=np.float64)


def forward_hashed(x: np.ndarray, token_ids: np.ndarray, experts: ExpertProvider, *, E: int,
                   n_heads: int = 1, capacity_factor: Optional[float] = None) -> Result:
    """The layer with the hash gate: y_u = FFN_{h(u)}(x_u) for a kept unit, 0 for a dropped one;
    aux = 0.  [HAI; Lesson 10 §3, §4; R16]"""
    xu = split_heads(x, n_heads)
    Tu = xu.shape[0]
    idx, g = hash_route(token_ids, E)
    C = capacity(capacity_factor, 1, Tu, E)
    d = dispatch(idx, E, C)
    y = np.zeros_like(xu)
    for e in range(E):
        r0, r1 = int(d.offsets[e]), int(d.offsets[e + 1])
        if r1 > r0:
            units = d.row_token[r0:r1]
            w1, w3, w2 = experts(e)
            y[units] = expert_ffn(xu[units], w1, w3, w2)
    return Result(None, idx, g, None, d, 0.0, C, merge_heads(y, n_heads))


# ---------------------------------------------------------------------------------------------
# [Lesson 10 worked example] load reporting of an expert-parallel placement


def expert_to_rank(num_experts: int, experts_per_rank: int) -> np.ndarray:
    """Owning rank of every expert [E] when each rank holds a contiguous block of experts_per_rank
    experts (expert e lives on rank ⌊e / experts_per_rank⌋).  [Lesson 10 §3, worked example]"""
    return np.arange(num_experts, dtype=np.int64) // int(experts_per_rank)


def load_per_rank(tokens_per_expert, experts_per_rank: int) -> list:
    """Tokens each rank's experts receive: the per-expert loads summed over each rank's block.
    [Lesson 10 worked example]"""
    c = np.asarray(tokens_per_expert, dtype=np.int64)
    owner = expert_to_rank(c.size, experts_per_rank)
    return np.bincount(owner, weights=c, minlength=c.size // int(experts_per_rank)).astype(np.int64).tolist()


def imbalance(loads) -> float:
    """Peak-to-mean ratio of the rank loads.  [Lesson 10 worked example]"""
    a = np.asarray(loads, dtype=np.float64)
    if a.size == 0 or not a.sum() > 0:
        raise ValueError("imbalance needs at least one rank and some load")
    return float(a.max() / a.mean())


def routing_volume(tokens_per_expert) -> int:
    """Token copies one step routes (each (token, pick) is one copy): the sum of the per-expert
    loads, the token count of the dispatch traffic.  [Lesson 10 §3]"""
    return int(np.asarray(tokens_per_expert, dtype=np.int64).sum())


def utilisation(loads) -> float:
    """Σ load / (ranks · max load): useful share of the step when the slowest rank sets it.  [Lesson 10 worked example]"""
    a = np.asarray(loads, dtype=np.float64)
    return float(a.sum() / (a.size * a.max()))
