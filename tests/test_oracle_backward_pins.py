"""Pins of the backward oracle against things other than itself (CPU only).

The backward is the gradient of the forward with the routing held fixed (R14). Two independent
checks fix it:
  * central finite differences of the (separately pinned) forward oracle, with the routing held at
    the unperturbed picks, along random directions in every input and parameter, and for single
    entries; with softmax and sigmoid scoring, group limits, capacity drops and head splitting;
  * the dense special case E = K = 1, where the layer is a plain SwiGLU FFN (gate 1, constant aux)
    and torch.autograd gives the gradients.
Planted mistakes (on the CPU) show the finite-difference pin fails on a wrong Jacobian.
"""
import numpy as np
import pytest
import torch

import oracle.moe_backward as B
import oracle.moe_oracle as O


def make_case(T=12, h=8, E=6, K=2, d_ff=10, n_heads=1, seed=0):
    rng = np.random.default_rng(seed)
    hu = h // n_heads
    return dict(
        x=rng.standard_normal((T, h)),
        w_g=rng.standard_normal((hu, E)) * 0.7,
        w1=rng.standard_normal((E, d_ff, hu)) / np.sqrt(hu),
        w3=rng.standard_normal((E, d_ff, hu)) / np.sqrt(hu),
        w2=rng.standard_normal((E, hu, d_ff)) / np.sqrt(d_ff),
        dy=rng.standard_normal((T, h)),
        logit_bias=rng.standard_normal(E) * 0.3,
        select_bias=rng.standard_normal(E) * 0.05,
    )


def loss(p, kw, idx):
    """L = <dy, y> + d_aux·aux at fixed picks idx (the forward oracle routed with idx_override)."""
    r = O.forward(p["x"], p["w_g"], lambda e: (p["w1"][e], p["w3"][e], p["w2"][e]), idx_override=idx,
                  logit_bias=p["logit_bias"], select_bias=p["select_bias"], **kw)
    return float(np.sum(p["dy"] * r.y)) + kw_d_aux(kw) * r.aux


def kw_d_aux(kw):
    return 0.7  # weight of the aux term in the loss used by the pins


def grads_of(p, kw):
    g = B.backward(p["x"], p["w_g"], lambda e: (p["w1"][e], p["w3"][e], p["w2"][e]), p["dy"], kw_d_aux(kw),
                   d_ff=p["w1"].shape[1], logit_bias=p["logit_bias"], select_bias=p["select_bias"], **kw)
    return g


NAMES = {"x": "dx", "w_g": "dw_g", "w1": "dw1", "w3": "dw3", "w2": "dw2"}

CONFIGS = [
    dict(E=6, K=2, score="softmax"),
    dict(E=6, K=2, score="sigmoid"),
    dict(E=8, K=3, score="sigmoid", n_groups=4, topk_groups=2),
    dict(E=6, K=2, score="softmax", capacity_factor=0.5),       # drops
    dict(E=6, K=1, score="softmax", capacity_factor=1.2),       # Switch-style top-1
    dict(E=6, K=2, score="softmax", n_heads=2),
]


def case_for(cfg, seed=0):
    n_heads = cfg.get("n_heads", 1)
    p = make_case(E=cfg["E"], K=cfg["K"], n_heads=n_heads, seed=seed)
    kw = dict(cfg)
    kw.setdefault("aux_alpha", 0.01 * 5)  # a larger α so the aux gradient is well above FD noise
    return p, kw


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_backward_matches_finite_differences_along_random_directions(cfg):
    p, kw = case_for(cfg)
    g = grads_of(p, kw)
    idx = g.idx
    rng = np.random.default_rng(7)
    eps = 1e-6
    for name, gname in NAMES.items():
        for _ in range(2):
            v = rng.standard_normal(p[name].shape)
            pp = dict(p); pm = dict(p)
            pp[name] = p[name] + eps * v
            pm[name] = p[name] - eps * v
            fd = (loss(pp, kw, idx) - loss(pm, kw, idx)) / (2 * eps)
            an = float(np.sum(getattr(g, gname) * v))
            assert an == pytest.approx(fd, rel=1e-6, abs=1e-8), (name, an, fd)


def test_backward_single_entries_match_finite_differences():
    p, kw = case_for(dict(E=6, K=2, score="sigmoid", capacity_factor=0.7))
    g = grads_of(p, kw)
    eps = 1e-6
    for name, gname, index in [("x", "dx", (3, 5)), ("w_g", "dw_g", (2, 4)), ("w1", "dw1", (1, 7, 2)),
                               ("w3", "dw3", (4, 0, 6)), ("w2", "dw2", (0, 3, 9))]:
        pp = dict(p); pm = dict(p)
        pp[name] = p[name].copy(); pm[name] = p[name].copy()
        pp[name][index] += eps
        pm[name][index] -= eps
        fd = (loss(pp, kw, g.idx) - loss(pm, kw, g.idx)) / (2 * eps)
        assert getattr(g, gname)[index] == pytest.approx(fd, rel=1e-6, abs=1e-9), (name, index)


def test_dlogits_is_the_gradient_wrt_the_logits():
    """dL/dl from the oracle equals finite differences in a per-expert logit offset (the logit bias
    enters l additively, so d/d(bias_e) = Σ_t dL/dl[t,e])."""
    p, kw = case_for(dict(E=6, K=2, score="softmax", capacity_factor=0.8))
    g = grads_of(p, kw)
    eps = 1e-6
    for e in range(6):
        pp = dict(p); pm = dict(p)
        pp["logit_bias"] = p["logit_bias"].copy(); pm["logit_bias"] = p["logit_bias"].copy()
        pp["logit_bias"][e] += eps
        pm["logit_bias"][e] -= eps
        fd = (loss(pp, kw, g.idx) - loss(pm, kw, g.idx)) / (2 * eps)
        assert g.dlogits[:, e].sum() == pytest.approx(fd, rel=1e-6, abs=1e-9)


def test_dropped_picks_have_zero_gate_gradient():
    p, kw = case_for(dict(E=6, K=2, score="softmax", capacity_factor=0.4))
    g = grads_of(p, kw)
    assert (g.slot_of < 0).any()
    assert np.all(g.dgate[g.slot_of < 0] == 0.0)


def test_dense_special_case_matches_torch_autograd():
    """E = K = 1: gate = 1 and L_aux = α are constant, so the layer is y = W2·(silu(W1 x) ⊙ W3 x)
    and dL/dW_g = 0."""
    rng = np.random.default_rng(3)
    T, h, d_ff = 9, 6, 7
    x = rng.standard_normal((T, h)); dy = rng.standard_normal((T, h))
    w1 = rng.standard_normal((1, d_ff, h)); w3 = rng.standard_normal((1, d_ff, h)); w2 = rng.standard_normal((1, h, d_ff))
    w_g = rng.standard_normal((h, 1))
    g = B.backward(x, w_g, lambda e: (w1[e], w3[e], w2[e]), dy, 1.0, E=1, K=1, d_ff=d_ff)
    tx = torch.tensor(x, requires_grad=True)
    t1 = torch.tensor(w1[0], requires_grad=True); t3 = torch.tensor(w3[0], requires_grad=True)
    t2 = torch.tensor(w2[0], requires_grad=True)
    y = (torch.nn.functional.silu(tx @ t1.T) * (tx @ t3.T)) @ t2.T
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(g.dx, tx.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g.dw1[0], t1.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g.dw3[0], t3.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g.dw2[0], t2.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(g.dw_g == 0.0)


# ----------------------------------------------------------------------------- planted mistakes
def fd_check_fails(monkeypatch, target, replacement, cfg):
    monkeypatch.setattr(B, target, replacement)
    p, kw = case_for(cfg)
    g = grads_of(p, kw)
    rng = np.random.default_rng(11)
    v = rng.standard_normal(p["w_g"].shape)
    eps = 1e-6
    pp = dict(p); pm = dict(p)
    pp["w_g"] = p["w_g"] + eps * v
    pm["w_g"] = p["w_g"] - eps * v
    fd = (loss(pp, kw, g.idx) - loss(pm, kw, g.idx)) / (2 * eps)
    return float(np.sum(g.dw_g * v)) != pytest.approx(fd, rel=1e-6, abs=1e-8)


def test_pin_catches_a_softmax_jacobian_without_its_inner_term(monkeypatch):
    def wrong(l, idx, dgate, score):
        g = O.gates(l, idx, score)
        dl = np.zeros(l.shape)
        rows = np.repeat(np.arange(l.shape[0]), idx.shape[1])
        np.add.at(dl, (rows, idx.reshape(-1).astype(np.int64)), (g * dgate).reshape(-1))
        return dl
    assert fd_check_fails(monkeypatch, "gate_backward", wrong, dict(E=6, K=2, score="softmax"))


def test_pin_catches_an_aux_gradient_with_the_wrong_sign(monkeypatch):
    right = B.aux_backward
    assert fd_check_fails(monkeypatch, "aux_backward", lambda *a: -right(*a),
                          dict(E=6, K=2, score="sigmoid", aux_alpha=0.5))


@pytest.mark.parametrize("cfg", CONFIGS[:4], ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_entry_oracle_equals_the_whole_gradient(cfg):
    """backward_entries (used where the layer is too large to differentiate whole) gives the same
    numbers as backward, entry by entry."""
    p, kw = case_for(cfg)
    ex = lambda e: (p["w1"][e], p["w3"][e], p["w2"][e])
    g = grads_of(p, kw)
    keep = {k: v for k, v in kw.items() if k in ("E", "K", "score", "n_heads", "capacity_factor", "aux_alpha")}
    units = [0, 5, 11]
    at2, at1, at3 = [(1, 2, 3), (5, 7, 9)], [(0, 4, 6), (3, 9, 1)], [(2, 0, 7), (4, 8, 2)]
    r = B.backward_entries(p["x"], p["w_g"], ex, p["dy"], kw_d_aux(kw), g.idx, logit_bias=p["logit_bias"],
                           units=units, dw2_at=at2, dw1_at=at1, dw3_at=at3, **keep)
    for u in units:
        np.testing.assert_allclose(r["dlogits"][u], g.dlogits[u], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["dx"][u], O.split_heads(g.dx, kw.get("n_heads", 1))[u], rtol=1e-12, atol=1e-14)
        for k in range(cfg["K"]):
            assert r["dgate"][(u, k)] == pytest.approx(g.dgate[u, k], rel=1e-12, abs=1e-14)
    for key, at, full in (("dw2", at2, g.dw2), ("dw1", at1, g.dw1), ("dw3", at3, g.dw3)):
        for a in at:
            assert r[key][a] == pytest.approx(full[a], rel=1e-12, abs=1e-14)


def fd_fails_on(monkeypatch, target, replacement, cfg, name):
    """True when, with B.<target> replaced, the oracle's gradient in `name` along a random
    direction disagrees with central differences of the (unpatched) forward oracle."""
    monkeypatch.setattr(B, target, replacement)
    p, kw = case_for(cfg)
    g = grads_of(p, kw)
    rng = np.random.default_rng(13)
    v = rng.standard_normal(p[name].shape)
    eps = 1e-6
    pp = dict(p); pm = dict(p)
    pp[name] = p[name] + eps * v
    pm[name] = p[name] - eps * v
    fd = (loss(pp, kw, g.idx) - loss(pm, kw, g.idx)) / (2 * eps)
    return float(np.sum(getattr(g, NAMES[name]) * v)) != pytest.approx(fd, rel=1e-6, abs=1e-8)


def test_pin_catches_a_swiglu_derivative_with_a_flipped_sigmoid(monkeypatch):
    wrong = lambda z: 1.0 / (1.0 + np.exp(z))  # σ(−z) in place of σ(z)
    cfg = dict(E=6, K=2, score="softmax")
    assert fd_fails_on(monkeypatch, "sigmoid", wrong, cfg, "w1")


def test_pin_catches_a_dx_without_the_router_path(monkeypatch):
    # drop dL/dl (gates and aux) entirely: dx loses its W_g term, dW_g becomes zero
    cfg = dict(E=6, K=2, score="sigmoid")
    monkeypatch.setattr(B, "aux_backward", lambda l, *a: np.zeros(l.shape))
    assert fd_fails_on(monkeypatch, "gate_backward", lambda l, *a: np.zeros(l.shape), cfg, "x")


def test_pin_catches_gradients_that_ignore_capacity_drops(monkeypatch):
    cfg = dict(E=6, K=2, score="softmax", capacity_factor=0.5)
    p, kw = case_for(cfg)
    assert (grads_of(p, kw).slot_of < 0).any()  # this case drops picks
    assert fd_fails_on(monkeypatch, "capacity", lambda *a: None, cfg, "w2")
