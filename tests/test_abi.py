"""The C-ABI library loads and exports every symbol include/moe.h declares; host-only calls and
argument validation work without a GPU (CPU only)."""
import ctypes
import os
import re

import pytest
import torch

from mixture_experts_layer_96_b300 import moe as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_symbols():
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_workspace_size", "moe_get_status"):
        assert n in names
    assert set(names) == set(M.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = M.load_library()
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert lib.moe_abi_version() == 2


_KEEP = []


def _addr(nbytes: int = 1 << 20, offset: int = 0) -> int:
    """An address for the host-side rejection tests below, which must fail before the library
    enqueues anything. With a GPU present it is real device memory of nbytes (each test sizes it
    to what the rejected call would touch), so even a check that wrongly let a call through would
    stay inside valid memory; without one no kernel can be launched at all, and a fixed,
    256-byte-aligned number stands in."""
    if torch.cuda.is_available():
        t = torch.zeros(nbytes + 256, dtype=torch.uint8, device="cuda")
        _KEEP.append(t)
        return t.data_ptr() + offset
    return 4096 + offset


def _cfg(**kw):
    base = dict(T=256, h=128, E=8, K=2, d_ff=256, capacity_factor=1.25, dtype="f32")
    base.update(kw)
    T, h, E, K, d_ff = (base.pop(k) for k in ("T", "h", "E", "K", "d_ff"))
    return M.make_config(T, h, E, K, d_ff, **base)


def test_capacity_host():
    assert M.capacity(_cfg()) == 80
    assert M.capacity(_cfg(T=16384, h=2048, E=64, K=2, d_ff=1408, dtype="bf16")) == 640
    assert M.capacity(_cfg(capacity_factor=None)) is None
    assert M.capacity(_cfg(T=4, n_heads=4, h=128, capacity_factor=1.0)) == 4  # T' = 16 units


def test_workspace_size_host():
    n = M.workspace_size(_cfg())
    assert n > 0 and n % 1024 == 0
    big = M.workspace_size(_cfg(T=4096, h=4096, E=8, K=2, d_ff=14336, dtype="bf16", capacity_factor=None))
    # packed x, hidden and packed y for T'K = 8192 rows dominate
    assert big >= 8192 * (4096 + 14336 + 4096) * 2


@pytest.mark.parametrize("bad", [
    dict(E=0), dict(K=3, E=2), dict(K=9, E=16), dict(E=257), dict(h=130, n_heads=4),
    dict(n_groups=3), dict(n_groups=4, topk_groups=5), dict(n_groups=4, topk_groups=1, K=3),
    dict(dtype="bf16", h=100), dict(d_ff=0), dict(T=-1),
])
def test_invalid_configs_rejected_on_host(bad):
    cfg = _cfg(**bad)
    lib = M.load_library()
    assert lib.moe_workspace_size(ctypes.byref(cfg)) == 0
    code = lib.moe_forward(ctypes.byref(cfg), None, None, None, None, None, None)
    assert code in (M.MOE_ERR_INVALID_ARG, M.MOE_ERR_UNSUPPORTED)


def test_missing_workspace_and_pointers_rejected():
    lib = M.load_library()
    cfg = _cfg()
    w = M.MoEWeights()
    x, y, ws = _addr(), _addr(), _addr(M.workspace_size(cfg))
    assert lib.moe_forward(ctypes.byref(cfg), x, ctypes.byref(w), y, None, None, None) == M.MOE_ERR_WORKSPACE
    assert lib.moe_forward(ctypes.byref(cfg), x, ctypes.byref(w), y, None, ws, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, ws, None) \
        == M.MOE_ERR_INVALID_ARG
    assert lib.moe_get_status(None, None) == M.MOE_ERR_WORKSPACE
    assert M.status_string(M.MOE_ERR_TIMEOUT) == "kernel wait timed out"


def test_launch_counter_is_readable_on_host():
    assert isinstance(M.launch_count(), int) and M.launch_count() >= 0


def test_backward_sizes_and_support_on_host():
    lib = M.load_library()
    cfg = _cfg(T=4096, h=4096, E=8, K=2, d_ff=14336, dtype="bf16", capacity_factor=None)
    assert M.saved_gu_size(cfg) == 8192 * 2 * 14336 * 2
    n = lib.moe_backward_workspace_size(ctypes.byref(cfg))
    # dY_packed, dG|dU and dX_packed dominate
    assert n >= 8192 * (4096 + 2 * 14336 + 4096) * 2 and n % 1024 == 0
    for bad in (_cfg(), _cfg(dtype="bf16", h=96, d_ff=128), _cfg(dtype="bf16", h=128, d_ff=96)):
        assert lib.moe_backward_workspace_size(ctypes.byref(bad)) == 0  # fp32, or h' / d_ff not multiples of 64
        g = M.MoEGrads()
        ws = _addr(M.workspace_size(bad))
        assert lib.moe_backward(ctypes.byref(bad), None, None, None, ctypes.c_float(1.0), None, None, ws,
                                ctypes.byref(g), ws, None) == M.MOE_ERR_UNSUPPORTED
        assert lib.moe_forward_train(ctypes.byref(bad), None, None, None, None, None, ws, None) \
            == M.MOE_ERR_UNSUPPORTED


def test_backward_rejects_missing_buffers_on_host():
    lib = M.load_library()
    cfg = _cfg(dtype="bf16")
    w, o, g = M.MoEWeights(), M.MoEOutputs(), M.MoEGrads()
    x, dy, gu = _addr(), _addr(), _addr(M.saved_gu_size(cfg))
    ws = _addr(M.workspace_size(cfg))
    bws = _addr(lib.moe_backward_workspace_size(ctypes.byref(cfg)))
    args = lambda ws, bws: (ctypes.byref(cfg), x, ctypes.byref(w), dy, ctypes.c_float(1.0), ctypes.byref(o), gu,
                            ws, ctypes.byref(g), bws, None)
    assert lib.moe_backward(*args(None, bws)) == M.MOE_ERR_WORKSPACE
    assert lib.moe_backward(*args(ws, bws + 4)) == M.MOE_ERR_WORKSPACE   # misaligned backward scratch
    assert lib.moe_backward(*args(ws, bws)) == M.MOE_ERR_INVALID_ARG     # no weights / saved outputs
    # the training forward needs the saved outputs
    assert lib.moe_forward_train(ctypes.byref(cfg), x, ctypes.byref(w), dy, None, gu, ws, None) \
        == M.MOE_ERR_INVALID_ARG


def _weights(cfg, device="cpu", **over):
    dt, hu, E, F = cfg.torch_dtype, cfg.h_unit, cfg.E, cfg.d_ff
    t = dict(w_router=torch.empty((hu, E), dtype=dt, device=device),
             w_gate=torch.empty((E, F, hu), dtype=dt, device=device),
             w_up=torch.empty((E, F, hu), dtype=dt, device=device),
             w_down=torch.empty((E, hu, F), dtype=dt, device=device))
    t.update(over)
    return M.LayerWeights(**t)


def test_binding_rejects_host_tensors_and_wrong_layouts():
    """The binding hands the library device pointers only: host tensors, wrong shapes and dtypes
    are refused in Python, before any call into the library. (Checks run shape, dtype, device,
    contiguity in that order, so host tensors reach the first two.)"""
    cfg = _cfg(dtype="bf16")
    bf = torch.bfloat16
    E, F, hu = cfg.E, cfg.d_ff, cfg.h_unit
    with pytest.raises(ValueError, match="w_router must be on a CUDA device"):
        _weights(cfg).check(cfg)
    with pytest.raises(ValueError, match="w_down: shape"):      # W2 given as [E][d_ff][h']
        M._req(torch.empty((E, F, hu), dtype=bf), "w_down", (E, hu, F), bf)
    with pytest.raises(ValueError, match="w_gate: dtype"):
        M._req(torch.empty((E, F, hu), dtype=torch.float32), "w_gate", (E, F, hu), bf)
    with pytest.raises(TypeError, match="w_up must be a tensor"):
        M._req("not a tensor", "w_up", (E, F, hu), bf)
    with pytest.raises(ValueError, match="w_router: shape"):    # the router weight is [h'][E]
        _weights(cfg, w_router=torch.empty((E, hu), dtype=bf)).check(cfg)


def test_gradient_buffers_are_fp32_except_dx():
    cfg = _cfg(dtype="bf16")
    g = M.Grads.allocate(cfg, "cpu")
    assert g.dx.dtype == torch.bfloat16 and g.dx.shape == (cfg.T, cfg.h)
    for t in (g.dw_router, g.dw_gate, g.dw_up, g.dw_down, g.dlogits, g.dgate):
        assert t.dtype == torch.float32
    assert g.dw_gate.shape == (cfg.E, cfg.d_ff, cfg.h_unit) and g.dw_down.shape == (cfg.E, cfg.h_unit, cfg.d_ff)
    assert g.dlogits.shape == (cfg.T_units, cfg.E) and g.dgate.shape == (cfg.T_units, cfg.K)
    with pytest.raises(ValueError, match="CUDA device"):
        g.check(cfg)
    assert M.Grads.allocate(cfg, "cpu", extras=False).dlogits is None


def test_expert_gemm_choices_are_validated_on_host():
    """moe_set_expert_gemm takes 1, 0 or -1 for each choice (host only, nothing launched); other
    values are refused and leave the automatic choices in place."""
    from mixture_experts_layer_96_b300 import MoEError, set_expert_gemm
    for bad in [(2, -1, -1), (-1, -2, -1), (-1, -1, 5)]:
        with pytest.raises(MoEError):
            set_expert_gemm(*bad)
    set_expert_gemm(1, 0, 1)
    set_expert_gemm(-1, -1, -1)
