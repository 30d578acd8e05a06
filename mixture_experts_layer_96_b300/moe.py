"""Python binding of the C ABI in include/moe.h (argument marshalling only).

Every compute step runs in the CUDA library `libmoe.so`; this module only checks tensor shapes,
dtypes and devices, passes raw device pointers and the current CUDA stream, and turns status codes
into exceptions. It has no fallback: if the library is missing it raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_STATUS, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_F32, MOE_BF16 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1

EXPORTS = ("moe_workspace_size", "moe_workspace_init", "moe_capacity", "moe_route", "moe_route_logits",
           "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward", "moe_get_status",
           "moe_status_string", "moe_launch_count", "moe_abi_version", "moe_dispatch_noalloc",
           "moe_saved_gu_size", "moe_forward_train", "moe_backward_workspace_size", "moe_backward",
           "moe_forward_profiled", "moe_route_hash", "moe_forward_hash", "moe_dispatch_sharded",
           "moe_set_expert_gemm")


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("capacity_factor", ctypes.c_double), ("h", ctypes.c_int32),
                ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("aux_alpha", ctypes.c_float), ("score", ctypes.c_int32), ("dtype", ctypes.c_int32)]

    @property
    def T_units(self) -> int:
        return self.T * self.n_heads

    @property
    def h_unit(self) -> int:
        return self.h // self.n_heads

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == MOE_BF16 else torch.float32


class MoEWeights(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("logit_bias", ctypes.c_void_p),
                ("select_bias", ctypes.c_void_p), ("w_gate", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


class MoEOutputs(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_gate", ctypes.c_void_p),
                ("logits", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("slot_of", ctypes.c_void_p), ("aux", ctypes.c_void_p)]


class MoEGrads(ctypes.Structure):
    _fields_ = [("dx", ctypes.c_void_p), ("dw_router", ctypes.c_void_p), ("dw_gate", ctypes.c_void_p),
                ("dw_up", ctypes.c_void_p), ("dw_down", ctypes.c_void_p), ("dlogits", ctypes.c_void_p),
                ("dgate", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m mixture_experts_layer_96_b300.build`")
    lib = ctypes.CDLL(path)
    P, S, I32, I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    cfgp = ctypes.POINTER(MoEConfig)
    sig = {
        "moe_workspace_size": (S, [cfgp]),
        "moe_workspace_init": (I32, [cfgp, P, P]),
        "moe_capacity": (I64, [cfgp]),
        "moe_route": (I32, [cfgp, P, P, P, P, P, P, P, P, P, P]),
        "moe_route_logits": (I32, [cfgp, P, P, P, P, P, P, P, P]),
        "moe_dispatch": (I32, [cfgp, P, P, P, P, P, P, P, P, P]),
        "moe_expert_ffn": (I32, [cfgp, P, P, P, P, P, P, P, P]),
        "moe_combine": (I32, [cfgp, P, P, P, P, P, P]),
        "moe_forward": (I32, [cfgp, P, ctypes.POINTER(MoEWeights), P, ctypes.POINTER(MoEOutputs), P, P]),
        "moe_route_hash": (I32, [cfgp, P, P, P, P, P]),
        "moe_dispatch_sharded": (I32, [cfgp, P, P, P, I64, P, P, P, P, P, P, P]),
        "moe_forward_hash": (I32, [cfgp, P, P, ctypes.POINTER(MoEWeights), P, ctypes.POINTER(MoEOutputs), P, P]),
        "moe_forward_profiled": (I32, [cfgp, P, ctypes.POINTER(MoEWeights), P, ctypes.POINTER(MoEOutputs), P,
                                       ctypes.POINTER(ctypes.c_void_p), P]),
        "moe_get_status": (I32, [P, P]),
        "moe_status_string": (ctypes.c_char_p, [I32]),
        "moe_launch_count": (ctypes.c_uint64, []),
        "moe_abi_version": (I32, []),
        "moe_set_expert_gemm": (I32, [I32, I32, I32]),
        "moe_dispatch_noalloc": (I32, [cfgp, P, P, P, P, P, P, P, P]),
        "moe_saved_gu_size": (S, [cfgp]),
        "moe_forward_train": (I32, [cfgp, P, ctypes.POINTER(MoEWeights), P, ctypes.POINTER(MoEOutputs), P, P, P]),
        "moe_backward_workspace_size": (S, [cfgp]),
        "moe_backward": (I32, [cfgp, P, ctypes.POINTER(MoEWeights), P, ctypes.c_float, ctypes.POINTER(MoEOutputs),
                               P, P, ctypes.POINTER(MoEGrads), P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().moe_status_string(code).decode()


def make_config(T: int, h: int, E: int, K: int, d_ff: int, *, n_heads: int = 1, n_groups: int = 1,
                topk_groups: int = 1, capacity_factor: Optional[float] = None, aux_alpha: float = 0.01,
                score: str = "softmax", dtype: str = "bf16") -> MoEConfig:
    cf = 0.0 if capacity_factor is None or math.isinf(capacity_factor) else float(capacity_factor)
    return MoEConfig(T=T, capacity_factor=cf, h=h, E=E, K=K, d_ff=d_ff, n_heads=n_heads, n_groups=n_groups,
                     topk_groups=topk_groups, aux_alpha=aux_alpha,
                     score=MOE_SCORE_SIGMOID if score == "sigmoid" else MOE_SCORE_SOFTMAX,
                     dtype=MOE_BF16 if dtype == "bf16" else MOE_F32)


def workspace_size(cfg: MoEConfig) -> int:
    n = load_library().moe_workspace_size(ctypes.byref(cfg))
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    return n


def capacity(cfg: MoEConfig) -> Optional[int]:
    c = load_library().moe_capacity(ctypes.byref(cfg))
    if c == -2:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_capacity")
    return None if c == -1 else int(c)


def launch_count() -> int:
    return int(load_library().moe_launch_count())


def set_expert_gemm(pair_tiles: int = -1, transposed_tails: int = -1, fold_combine: int = -1) -> None:
    """Force the expert GEMMs' choices process-wide (1 on, 0 off, -1 automatic): CTA-pair 256-row
    tiles, transposed pair-tile tails of up to 224 rows, and the combine folded into the down GEMM
    (automatic: K == 1)."""
    _check(load_library().moe_set_expert_gemm(int(pair_tiles), int(transposed_tails), int(fold_combine)),
           "moe_set_expert_gemm")


# ------------------------------------------------------------------------------------------------
def _stream(stream, device=None) -> int:
    """Raw handle of `stream`, or of the current stream of `device` (the tensors' device)."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device} but the tensors are on {device}")
    return stream.cuda_stream


def _one_device(*tensors) -> torch.device:
    """The CUDA device every given tensor (None entries skipped) lives on; raises if they differ.
    The library takes the current device for its per-device state (SM count, static scratch), so
    every call runs with this device made current."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"tensor on {t.device}: every buffer must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on {dev} and {t.device}: every buffer must be on one device")
    return dev


def _run(tensors, stream, fn, *args) -> int:
    """Call library function `fn(*args, stream)` with the tensors' device made current (every
    tensor on that one device, the stream too) and return its status code."""
    dev = _one_device(*tensors)
    with torch.cuda.device(dev):
        return int(fn(*args, _stream(stream, dev)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoEError(code, where)


def _req(t: torch.Tensor, name: str, shape, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} != {dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class Workspace:
    """Device scratch of one config (a torch uint8 tensor), status header zeroed at creation."""

    def __init__(self, cfg: MoEConfig, device="cuda", stream=None):
        self.cfg = cfg
        self.nbytes = workspace_size(cfg)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        assert self.buf.data_ptr() % 1024 == 0 or self.buf.data_ptr() % 256 == 0
        _check(_run([self.buf], stream, load_library().moe_workspace_init, ctypes.byref(cfg), self.ptr),
               "moe_workspace_init")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self, stream=None) -> int:
        """Wait for the stream; read and clear the device status word."""
        return _run([self.buf], stream, load_library().moe_get_status, self.ptr)

    def check(self, stream=None):
        _check(self.status(stream), "moe_get_status")


def moe_get_status(ws: Workspace, stream=None) -> int:
    return ws.status(stream)


def moe_route(cfg: MoEConfig, x, w_router, logit_bias=None, select_bias=None, *, ws: Workspace,
              topk_idx=None, topk_gate=None, logits_out=None, aux_out=None, want_logits=False,
              want_aux=False, stream=None):
    """Router + scoring + Top-K + gates. Returns (topk_idx, topk_gate, logits or None, aux or None)."""
    lib = load_library()
    dt, dev = cfg.torch_dtype, x.device
    Tu, hu, E, K = cfg.T_units, cfg.h_unit, cfg.E, cfg.K
    _req(x, "x", (cfg.T, cfg.h), dt)
    _req(w_router, "w_router", (hu, E), dt)
    for b, n in ((logit_bias, "logit_bias"), (select_bias, "select_bias")):
        if b is not None:
            _req(b, n, (E,), torch.float32)
    topk_idx = topk_idx if topk_idx is not None else torch.empty((Tu, K), dtype=torch.int32, device=dev)
    topk_gate = topk_gate if topk_gate is not None else torch.empty((Tu, K), dtype=torch.float32, device=dev)
    _req(topk_idx, "topk_idx", (Tu, K), torch.int32)
    _req(topk_gate, "topk_gate", (Tu, K), torch.float32)
    if logits_out is None and want_logits:
        logits_out = torch.empty((Tu, E), dtype=torch.float32, device=dev)
    if aux_out is None and want_aux:
        aux_out = torch.empty((1,), dtype=torch.float32, device=dev)
    _check(_run([x, w_router, logit_bias, select_bias, topk_idx, topk_gate, logits_out, aux_out, ws.buf], stream,
                lib.moe_route, ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(select_bias),
                _ptr(topk_idx), _ptr(topk_gate), _ptr(logits_out), _ptr(aux_out), ws.ptr), "moe_route")
    return topk_idx, topk_gate, logits_out, aux_out


def moe_route_logits(cfg: MoEConfig, logits, logit_bias=None, select_bias=None, *, ws: Workspace,
                     topk_idx=None, topk_gate=None, aux_out=None, want_aux=False, stream=None):
    """Routing from given fp32 logits [T'][E]. Returns (topk_idx, topk_gate, aux or None)."""
    lib = load_library()
    Tu, E, K, dev = cfg.T_units, cfg.E, cfg.K, logits.device
    _req(logits, "logits", (Tu, E), torch.float32)
    for b, n in ((logit_bias, "logit_bias"), (select_bias, "select_bias")):
        if b is not None:
            _req(b, n, (E,), torch.float32)
    topk_idx = topk_idx if topk_idx is not None else torch.empty((Tu, K), dtype=torch.int32, device=dev)
    topk_gate = topk_gate if topk_gate is not None else torch.empty((Tu, K), dtype=torch.float32, device=dev)
    if aux_out is None and want_aux:
        aux_out = torch.empty((1,), dtype=torch.float32, device=dev)
    _req(topk_idx, "topk_idx", (Tu, K), torch.int32)
    _req(topk_gate, "topk_gate", (Tu, K), torch.float32)
    _check(_run([logits, logit_bias, select_bias, topk_idx, topk_gate, aux_out, ws.buf], stream,
                lib.moe_route_logits, ctypes.byref(cfg), _ptr(logits), _ptr(logit_bias), _ptr(select_bias),
                _ptr(topk_idx), _ptr(topk_gate), _ptr(aux_out), ws.ptr), "moe_route_logits")
    return topk_idx, topk_gate, aux_out


def moe_dispatch(cfg: MoEConfig, x, topk_idx, *, ws: Workspace, counts=None, offsets=None, slot_of=None,
                 row_token=None, x_packed=None, stream=None):
    """Capacity drop + pack. Returns (counts, offsets, slot_of, row_token, x_packed)."""
    lib = load_library()
    dt, dev = cfg.torch_dtype, x.device
    Tu, hu, E, K = cfg.T_units, cfg.h_unit, cfg.E, cfg.K
    _req(x, "x", (cfg.T, cfg.h), dt)
    _req(topk_idx, "topk_idx", (Tu, K), torch.int32)
    counts = counts if counts is not None else torch.empty((E,), dtype=torch.int32, device=dev)
    offsets = offsets if offsets is not None else torch.empty((E + 1,), dtype=torch.int32, device=dev)
    slot_of = slot_of if slot_of is not None else torch.empty((Tu, K), dtype=torch.int32, device=dev)
    row_token = row_token if row_token is not None else torch.empty((Tu * K,), dtype=torch.int32, device=dev)
    x_packed = x_packed if x_packed is not None else torch.empty((Tu * K, hu), dtype=dt, device=dev)
    _req(counts, "counts", (E,), torch.int32)
    _req(offsets, "offsets", (E + 1,), torch.int32)
    _req(slot_of, "slot_of", (Tu, K), torch.int32)
    _req(row_token, "row_token", (Tu * K,), torch.int32)
    _req(x_packed, "x_packed", (Tu * K, hu), dt)
    _check(_run([x, topk_idx, counts, offsets, slot_of, row_token, x_packed, ws.buf], stream, lib.moe_dispatch,
                ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(offsets), _ptr(slot_of),
                _ptr(row_token), _ptr(x_packed), ws.ptr), "moe_dispatch")
    return counts, offsets, slot_of, row_token, x_packed


def moe_dispatch_sharded(cfg: MoEConfig, x, topk_idx, queue_base, T_global: int, *, ws: Workspace, counts=None,
                         offsets=None, slot_of=None, row_token=None, x_packed=None, stream=None):
    """Dispatch of one token shard of a batch of T_global tokens: queue_base [E] int32 holds each
    expert's picks on the earlier shards; capacity and drop order are the whole batch's.
    Returns (counts, offsets, slot_of, row_token, x_packed), local to the shard."""
    lib = load_library()
    dt, dev = cfg.torch_dtype, x.device
    Tu, hu, E, K = cfg.T_units, cfg.h_unit, cfg.E, cfg.K
    _req(x, "x", (cfg.T, cfg.h), dt)
    _req(topk_idx, "topk_idx", (Tu, K), torch.int32)
    _req(queue_base, "queue_base", (E,), torch.int32)
    counts = counts if counts is not None else torch.empty((E,), dtype=torch.int32, device=dev)
    offsets = offsets if offsets is not None else torch.empty((E + 1,), dtype=torch.int32, device=dev)
    slot_of = slot_of if slot_of is not None else torch.empty((Tu, K), dtype=torch.int32, device=dev)
    row_token = row_token if row_token is not None else torch.empty((Tu * K,), dtype=torch.int32, device=dev)
    x_packed = x_packed if x_packed is not None else torch.empty((Tu * K, hu), dtype=dt, device=dev)
    _check(_run([x, topk_idx, queue_base, counts, offsets, slot_of, row_token, x_packed, ws.buf], stream,
                lib.moe_dispatch_sharded, ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(queue_base),
                ctypes.c_int64(T_global), _ptr(counts), _ptr(offsets), _ptr(slot_of), _ptr(row_token),
                _ptr(x_packed), ws.ptr), "moe_dispatch_sharded")
    return counts, offsets, slot_of, row_token, x_packed


def moe_expert_ffn(cfg: MoEConfig, x_packed, offsets, w_gate, w_up, w_down, *, ws: Workspace,
                   y_packed=None, stream=None):
    """Per-expert SwiGLU FFN over packed rows. Returns y_packed [T'K][h']."""
    lib = load_library()
    dt, dev = cfg.torch_dtype, x_packed.device
    Tu, hu, E, K, F = cfg.T_units, cfg.h_unit, cfg.E, cfg.K, cfg.d_ff
    _req(x_packed, "x_packed", (Tu * K, hu), dt)
    _req(offsets, "offsets", (E + 1,), torch.int32)
    _req(w_gate, "w_gate", (E, F, hu), dt)
    _req(w_up, "w_up", (E, F, hu), dt)
    _req(w_down, "w_down", (E, hu, F), dt)
    y_packed = y_packed if y_packed is not None else torch.empty((Tu * K, hu), dtype=dt, device=dev)
    _req(y_packed, "y_packed", (Tu * K, hu), dt)
    _check(_run([x_packed, offsets, w_gate, w_up, w_down, y_packed, ws.buf], stream, lib.moe_expert_ffn,
                ctypes.byref(cfg), _ptr(x_packed), _ptr(offsets), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                _ptr(y_packed), ws.ptr), "moe_expert_ffn")
    return y_packed


def moe_combine(cfg: MoEConfig, y_packed, slot_of, topk_gate, *, ws: Workspace, y=None, stream=None):
    """Gate-weighted combine back to unit order. Returns y [T][h]."""
    lib = load_library()
    dt, dev = cfg.torch_dtype, y_packed.device
    Tu, hu, K = cfg.T_units, cfg.h_unit, cfg.K
    _req(y_packed, "y_packed", (Tu * K, hu), dt)
    _req(slot_of, "slot_of", (Tu, K), torch.int32)
    _req(topk_gate, "topk_gate", (Tu, K), torch.float32)
    y = y if y is not None else torch.empty((cfg.T, cfg.h), dtype=dt, device=dev)
    _req(y, "y", (cfg.T, cfg.h), dt)
    _check(_run([y_packed, slot_of, topk_gate, y, ws.buf], stream, lib.moe_combine, ctypes.byref(cfg),
                _ptr(y_packed), _ptr(slot_of), _ptr(topk_gate), _ptr(y), ws.ptr), "moe_combine")
    return y


@dataclass
class LayerWeights:
    """Device tensors of one layer."""
    w_router: torch.Tensor
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    logit_bias: Optional[torch.Tensor] = None
    select_bias: Optional[torch.Tensor] = None

    def check(self, cfg: MoEConfig):
        dt, hu, E, F = cfg.torch_dtype, cfg.h_unit, cfg.E, cfg.d_ff
        _req(self.w_router, "w_router", (hu, E), dt)
        _req(self.w_gate, "w_gate", (E, F, hu), dt)
        _req(self.w_up, "w_up", (E, F, hu), dt)
        _req(self.w_down, "w_down", (E, hu, F), dt)
        for b, n in ((self.logit_bias, "logit_bias"), (self.select_bias, "select_bias")):
            if b is not None:
                _req(b, n, (E,), torch.float32)

    def tensors(self):
        return (self.w_router, self.w_gate, self.w_up, self.w_down, self.logit_bias, self.select_bias)

    def c_struct(self) -> MoEWeights:
        return MoEWeights(_ptr(self.w_router), _ptr(self.logit_bias), _ptr(self.select_bias),
                          _ptr(self.w_gate), _ptr(self.w_up), _ptr(self.w_down))


@dataclass
class ForwardOutputs:
    topk_idx: Optional[torch.Tensor] = None
    topk_gate: Optional[torch.Tensor] = None
    logits: Optional[torch.Tensor] = None
    counts: Optional[torch.Tensor] = None
    offsets: Optional[torch.Tensor] = None
    slot_of: Optional[torch.Tensor] = None
    aux: Optional[torch.Tensor] = None

    @staticmethod
    def allocate(cfg: MoEConfig, device, logits=True) -> "ForwardOutputs":
        Tu, E, K = cfg.T_units, cfg.E, cfg.K
        i32, f32 = torch.int32, torch.float32
        return ForwardOutputs(
            topk_idx=torch.empty((Tu, K), dtype=i32, device=device),
            topk_gate=torch.empty((Tu, K), dtype=f32, device=device),
            logits=torch.empty((Tu, E), dtype=f32, device=device) if logits else None,
            counts=torch.empty((E,), dtype=i32, device=device),
            offsets=torch.empty((E + 1,), dtype=i32, device=device),
            slot_of=torch.empty((Tu, K), dtype=i32, device=device),
            aux=torch.empty((1,), dtype=f32, device=device))

    def tensors(self):
        return (self.topk_idx, self.topk_gate, self.logits, self.counts, self.offsets, self.slot_of, self.aux)

    def c_struct(self) -> MoEOutputs:
        return MoEOutputs(_ptr(self.topk_idx), _ptr(self.topk_gate), _ptr(self.logits), _ptr(self.counts),
                          _ptr(self.offsets), _ptr(self.slot_of), _ptr(self.aux))


def moe_forward(cfg: MoEConfig, x, weights: LayerWeights, *, ws: Workspace, y=None,
                outputs: Optional[ForwardOutputs] = None, stream=None):
    """The whole layer: x [T][h] → y [T][h]. `outputs` receives the optional intermediates."""
    lib = load_library()
    dt = cfg.torch_dtype
    _req(x, "x", (cfg.T, cfg.h), dt)
    weights.check(cfg)
    y = y if y is not None else torch.empty((cfg.T, cfg.h), dtype=dt, device=x.device)
    _req(y, "y", (cfg.T, cfg.h), dt)
    cw = weights.c_struct()
    co = outputs.c_struct() if outputs is not None else None
    _check(_run([x, y, ws.buf, *weights.tensors(), *(outputs.tensors() if outputs is not None else ())], stream,
                lib.moe_forward, ctypes.byref(cfg), _ptr(x), ctypes.byref(cw), _ptr(y),
                ctypes.byref(co) if co is not None else None, ws.ptr), "moe_forward")
    return y


def moe_route_hash(cfg: MoEConfig, token_ids, *, ws: Workspace, topk_idx=None, topk_gate=None, stream=None):
    """Hash gate (top-1): expert fmix32(token id) mod E, gate 1. token_ids [T'] int32.
    Returns (topk_idx [T'][1], topk_gate [T'][1])."""
    lib = load_library()
    Tu, dev = cfg.T_units, token_ids.device
    _req(token_ids, "token_ids", (Tu,), torch.int32)
    topk_idx = topk_idx if topk_idx is not None else torch.empty((Tu, cfg.K), dtype=torch.int32, device=dev)
    topk_gate = topk_gate if topk_gate is not None else torch.empty((Tu, cfg.K), dtype=torch.float32, device=dev)
    _req(topk_idx, "topk_idx", (Tu, cfg.K), torch.int32)
    _req(topk_gate, "topk_gate", (Tu, cfg.K), torch.float32)
    _check(_run([token_ids, topk_idx, topk_gate, ws.buf], stream, lib.moe_route_hash, ctypes.byref(cfg),
                _ptr(token_ids), _ptr(topk_idx), _ptr(topk_gate), ws.ptr), "moe_route_hash")
    return topk_idx, topk_gate


def moe_forward_hash(cfg: MoEConfig, x, token_ids, w_gate, w_up, w_down, *, ws: Workspace, y=None,
                     outputs: Optional[ForwardOutputs] = None, stream=None):
    """The layer with the hash gate: x [T][h], token_ids [T'] int32 → y [T][h]. Returns y."""
    lib = load_library()
    dt, hu, E, F = cfg.torch_dtype, cfg.h_unit, cfg.E, cfg.d_ff
    _req(x, "x", (cfg.T, cfg.h), dt)
    _req(token_ids, "token_ids", (cfg.T_units,), torch.int32)
    _req(w_gate, "w_gate", (E, F, hu), dt)
    _req(w_up, "w_up", (E, F, hu), dt)
    _req(w_down, "w_down", (E, hu, F), dt)
    y = y if y is not None else torch.empty((cfg.T, cfg.h), dtype=dt, device=x.device)
    _req(y, "y", (cfg.T, cfg.h), dt)
    cw = MoEWeights(None, None, None, _ptr(w_gate), _ptr(w_up), _ptr(w_down))
    co = outputs.c_struct() if outputs is not None else None
    _check(_run([x, token_ids, y, w_gate, w_up, w_down, ws.buf, *(outputs.tensors() if outputs is not None else ())],
                stream, lib.moe_forward_hash, ctypes.byref(cfg), _ptr(x), _ptr(token_ids), ctypes.byref(cw), _ptr(y),
                ctypes.byref(co) if co is not None else None, ws.ptr), "moe_forward_hash")
    return y


FORWARD_STAGES = ("route", "scan", "pack", "expert_ffn", "combine")


def moe_forward_profiled(cfg: MoEConfig, x, weights: LayerWeights, events, *, ws: Workspace, y=None,
                         outputs: Optional[ForwardOutputs] = None, stream=None):
    """moe_forward with the 6 given torch.cuda.Event (enable_timing=True) recorded at its stage
    boundaries: event i → i+1 brackets FORWARD_STAGES[i]. Returns y."""
    lib = load_library()
    dt = cfg.torch_dtype
    _req(x, "x", (cfg.T, cfg.h), dt)
    weights.check(cfg)
    if len(events) != 6:
        raise ValueError("moe_forward_profiled takes 6 events")
    y = y if y is not None else torch.empty((cfg.T, cfg.h), dtype=dt, device=x.device)
    _req(y, "y", (cfg.T, cfg.h), dt)
    dev = _one_device(x, y)
    with torch.cuda.device(dev):
        st = torch.cuda.current_stream(dev) if stream is None else stream
        for ev in events:  # torch creates the CUDA event at its first record
            if not ev.cuda_event:
                ev.record(st)
        handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
    cw = weights.c_struct()
    co = outputs.c_struct() if outputs is not None else None
    _check(_run([x, y, ws.buf, *weights.tensors(), *(outputs.tensors() if outputs is not None else ())], stream,
                lib.moe_forward_profiled, ctypes.byref(cfg), _ptr(x), ctypes.byref(cw), _ptr(y),
                ctypes.byref(co) if co is not None else None, ws.ptr, handles), "moe_forward_profiled")
    return y


# ------------------------------------------------------------------------------------------------
# training: forward that keeps G | U, and the backward (bf16 layers, h' and d_ff multiples of 64)

def saved_gu_size(cfg: MoEConfig) -> int:
    return int(load_library().moe_saved_gu_size(ctypes.byref(cfg)))


def moe_forward_train(cfg: MoEConfig, x, weights: LayerWeights, outputs: ForwardOutputs, *, ws: Workspace,
                      gu=None, y=None, stream=None):
    """moe_forward that also saves the SwiGLU inputs G | U [T'K][2·d_ff] (bf16) for moe_backward.
    `outputs` must hold topk_idx, topk_gate, logits and slot_of. Returns (y, gu)."""
    lib = load_library()
    dt = cfg.torch_dtype
    _req(x, "x", (cfg.T, cfg.h), dt)
    weights.check(cfg)
    rows = cfg.T_units * cfg.K
    y = y if y is not None else torch.empty((cfg.T, cfg.h), dtype=dt, device=x.device)
    _req(y, "y", (cfg.T, cfg.h), dt)
    gu = gu if gu is not None else torch.empty((rows, 2 * cfg.d_ff), dtype=dt, device=x.device)
    _req(gu, "gu", (rows, 2 * cfg.d_ff), dt)
    cw, co = weights.c_struct(), outputs.c_struct()
    _check(_run([x, y, gu, ws.buf, *weights.tensors(), *outputs.tensors()], stream, lib.moe_forward_train,
                ctypes.byref(cfg), _ptr(x), ctypes.byref(cw), _ptr(y), ctypes.byref(co), _ptr(gu), ws.ptr),
           "moe_forward_train")
    return y, gu


class BackwardWorkspace:
    """Device scratch of the backward for one config."""

    def __init__(self, cfg: MoEConfig, device="cuda"):
        self.nbytes = int(load_library().moe_backward_workspace_size(ctypes.byref(cfg)))
        if self.nbytes == 0:
            raise MoEError(MOE_ERR_UNSUPPORTED, "moe_backward_workspace_size")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


@dataclass
class Grads:
    dx: torch.Tensor
    dw_router: torch.Tensor
    dw_gate: torch.Tensor
    dw_up: torch.Tensor
    dw_down: torch.Tensor
    dlogits: Optional[torch.Tensor] = None
    dgate: Optional[torch.Tensor] = None

    @staticmethod
    def allocate(cfg: MoEConfig, device, extras=True) -> "Grads":
        f32, hu, E, F = torch.float32, cfg.h_unit, cfg.E, cfg.d_ff
        return Grads(dx=torch.empty((cfg.T, cfg.h), dtype=cfg.torch_dtype, device=device),
                     dw_router=torch.empty((hu, E), dtype=f32, device=device),
                     dw_gate=torch.empty((E, F, hu), dtype=f32, device=device),
                     dw_up=torch.empty((E, F, hu), dtype=f32, device=device),
                     dw_down=torch.empty((E, hu, F), dtype=f32, device=device),
                     dlogits=torch.empty((cfg.T_units, E), dtype=f32, device=device) if extras else None,
                     dgate=torch.empty((cfg.T_units, cfg.K), dtype=f32, device=device) if extras else None)

    def check(self, cfg: MoEConfig):
        f32, hu, E, F = torch.float32, cfg.h_unit, cfg.E, cfg.d_ff
        _req(self.dx, "dx", (cfg.T, cfg.h), cfg.torch_dtype)
        _req(self.dw_router, "dw_router", (hu, E), f32)
        _req(self.dw_gate, "dw_gate", (E, F, hu), f32)
        _req(self.dw_up, "dw_up", (E, F, hu), f32)
        _req(self.dw_down, "dw_down", (E, hu, F), f32)
        if self.dlogits is not None:
            _req(self.dlogits, "dlogits", (cfg.T_units, E), f32)
        if self.dgate is not None:
            _req(self.dgate, "dgate", (cfg.T_units, cfg.K), f32)

    def tensors(self):
        return (self.dx, self.dw_router, self.dw_gate, self.dw_up, self.dw_down, self.dlogits, self.dgate)

    def c_struct(self) -> MoEGrads:
        return MoEGrads(_ptr(self.dx), _ptr(self.dw_router), _ptr(self.dw_gate), _ptr(self.dw_up),
                        _ptr(self.dw_down), _ptr(self.dlogits), _ptr(self.dgate))


def moe_backward(cfg: MoEConfig, x, weights: LayerWeights, dy, outputs: ForwardOutputs, gu, *, ws: Workspace,
                 bws: BackwardWorkspace, d_aux: float = 1.0, grads: Optional[Grads] = None, stream=None) -> Grads:
    """Gradients of <dy, y> + d_aux·L_aux for the moe_forward_train that filled ws, outputs and gu
    (routing held fixed). Returns the Grads (dW fp32, dx in x's dtype)."""
    lib = load_library()
    dt = cfg.torch_dtype
    _req(x, "x", (cfg.T, cfg.h), dt)
    _req(dy, "dy", (cfg.T, cfg.h), dt)
    weights.check(cfg)
    _req(gu, "gu", (cfg.T_units * cfg.K, 2 * cfg.d_ff), dt)
    grads = grads if grads is not None else Grads.allocate(cfg, x.device)
    grads.check(cfg)
    cw, co, cg = weights.c_struct(), outputs.c_struct(), grads.c_struct()
    _check(_run([x, dy, gu, ws.buf, bws.buf, *weights.tensors(), *outputs.tensors(), *grads.tensors()], stream,
                lib.moe_backward, ctypes.byref(cfg), _ptr(x), ctypes.byref(cw), _ptr(dy), ctypes.c_float(d_aux),
                ctypes.byref(co), _ptr(gu), ws.ptr, ctypes.byref(cg), bws.ptr), "moe_backward")
    return grads


NOALLOC_SCRATCH_BYTES = 1 << 20


def moe_dispatch_noalloc(cfg: MoEConfig, x, topk_idx, *, counts=None, offsets=None, slot_of=None,
                         row_token=None, x_packed=None, stream=None):
    """moe_dispatch for callers that cannot allocate device memory: no workspace; the library's
    fixed 1 MiB scratch array is used instead (calls that overlap on the GPU race).
    Returns (counts, offsets, slot_of, row_token, x_packed)."""
    lib = load_library()
    dt, dev = cfg.torch_dtype, x.device
    Tu, hu, E, K = cfg.T_units, cfg.h_unit, cfg.E, cfg.K
    _req(x, "x", (cfg.T, cfg.h), dt)
    _req(topk_idx, "topk_idx", (Tu, K), torch.int32)
    counts = counts if counts is not None else torch.empty((E,), dtype=torch.int32, device=dev)
    offsets = offsets if offsets is not None else torch.empty((E + 1,), dtype=torch.int32, device=dev)
    slot_of = slot_of if slot_of is not None else torch.empty((Tu, K), dtype=torch.int32, device=dev)
    row_token = row_token if row_token is not None else torch.empty((Tu * K,), dtype=torch.int32, device=dev)
    x_packed = x_packed if x_packed is not None else torch.empty((Tu * K, hu), dtype=dt, device=dev)
    _req(counts, "counts", (E,), torch.int32)
    _req(offsets, "offsets", (E + 1,), torch.int32)
    _req(slot_of, "slot_of", (Tu, K), torch.int32)
    _req(row_token, "row_token", (Tu * K,), torch.int32)
    _req(x_packed, "x_packed", (Tu * K, hu), dt)
    code = _run([x, topk_idx, counts, offsets, slot_of, row_token, x_packed], stream, lib.moe_dispatch_noalloc,
                ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(offsets), _ptr(slot_of),
                _ptr(row_token), _ptr(x_packed))
    if code == MOE_ERR_UNSUPPORTED:
        raise MoEError(code, f"moe_dispatch_noalloc: {Tu} units x {E} experts need more than the "
                             f"{NOALLOC_SCRATCH_BYTES} bytes of fixed scratch")
    _check(code, "moe_dispatch_noalloc")
    return counts, offsets, slot_of, row_token, x_packed
