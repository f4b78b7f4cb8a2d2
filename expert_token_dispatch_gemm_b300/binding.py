"""ctypes binding of libmoe.so: argument marshalling only.

Every function here has the name and argument order of the C entry point in
include/moe.h. Tensors are torch CUDA tensors (device memory owned by the caller);
the current torch CUDA stream is passed as the stream. No step of the layer runs in
Python: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT = range(6)
MOE_DTYPE_BF16, MOE_DTYPE_FP32 = 0, 1
MOE_MODE_DISPATCH, MOE_MODE_MASK_SUM = 0, 1
MOE_PRIORITY_TOKEN, MOE_PRIORITY_SLOT = 0, 1
MOE_DEV_TIMEOUT, MOE_DEV_BAD_EXPERT_ID = 1, 2

_DTYPES = {MOE_DTYPE_BF16: torch.bfloat16, MOE_DTYPE_FP32: torch.float32}


class MoeError(RuntimeError):
    def __init__(self, status: int, func: str, message: str):
        self.status = status
        super().__init__(f"{func}: status {status}: {message}")


class MoeConfig(ctypes.Structure):
    """struct moe_config."""
    _fields_ = [("num_tokens", ctypes.c_int64), ("hidden", ctypes.c_int64),
                ("intermediate", ctypes.c_int64), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("ep_size", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("mode", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("group_limit", ctypes.c_int32), ("selection_bias", ctypes.c_void_p),
                ("capacity_priority", ctypes.c_int32), ("training", ctypes.c_int32)]

    @property
    def torch_dtype(self):
        return _DTYPES[self.dtype]


class MoeDiagnostics(ctypes.Structure):
    """struct moe_diagnostics."""
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_idx", "topk_w", "routed_counts", "counts", "expert_offsets", "part_offsets",
        "perm", "slot_pos", "stage_events", "router_logits")]
    _ARRAYS = ("topk_idx", "topk_w", "routed_counts", "counts", "expert_offsets",
               "part_offsets", "perm", "slot_pos", "router_logits")


MOE_NUM_STAGES = 7
STAGE_NAMES = ("route", "scan", "assign", "permute", "gate_up", "down", "combine")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with "
                          "expert_token_dispatch_gemm_b300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P, S, I32, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_float
    cfgp = ctypes.POINTER(MoeConfig)
    sig = {
        "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "moe_last_error": (ctypes.c_char_p, []),
        "moe_workspace_size": (ctypes.c_int, [cfgp, ctypes.POINTER(S)]),
        "moe_packed_gate_up_size": (ctypes.c_int, [cfgp, ctypes.POINTER(S)]),
        "moe_pack_weights": (ctypes.c_int, [cfgp, P, P, P, P]),
        "moe_route": (ctypes.c_int, [cfgp, P, P, P, P, P, P]),
        "moe_update_selection_bias": (ctypes.c_int, [cfgp, P, P, ctypes.c_float, P]),
        "moe_dispatch": (ctypes.c_int, [cfgp, P, P, P, P, P, P, P, P, P, P, S, P]),
        "moe_dispatch_noalloc": (ctypes.c_int, [cfgp, P, P, P, P, P, P, P, P, P, P]),
        "moe_expert_ffn": (ctypes.c_int, [cfgp, P, P, I32, I32, P, P, P, P, P, P, S, P]),
        "moe_combine": (ctypes.c_int, [cfgp, P, P, P, P, P, S, P]),
        "moe_layer_forward": (ctypes.c_int, [cfgp, P, P, P, P, P, P,
                                             ctypes.POINTER(MoeDiagnostics), P, S, P]),
        "moe_read_device_status": (ctypes.c_int, [cfgp, P, S, ctypes.POINTER(I32), I32, P]),
        "moe_balance_stats": (ctypes.c_int, [cfgp, P, P, P, P, P, S, P]),
        "moe_layer_backward": (ctypes.c_int, [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, S, P]),
        "moe_tp_slice": (ctypes.c_int, [ctypes.c_int64, I32, I32, ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64)]),
        "moe_tp_reduce": (ctypes.c_int, [cfgp, I32, P, P, P]),
        "moe_check_wait_timeout": (ctypes.c_int, [cfgp, P, S, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    del F
    return lib


lib = _load()


def config(N, H, I, E, top_k, ep_size, capacity_factor=None, mode="dispatch",
           dtype="bf16", has_bias=False, group_limit=0, selection_bias=None,
           capacity_priority="token", training=False) -> MoeConfig:
    """struct moe_config. selection_bias: None or an fp32 [E] CUDA tensor, which the
    caller keeps alive while the config is in use. capacity_priority: "token" or
    "slot"."""
    if capacity_priority not in ("token", "slot"):
        raise ValueError(f"capacity_priority must be 'token' or 'slot', not {capacity_priority!r}")
    return MoeConfig(int(N), int(H), int(I), int(E), int(top_k), int(ep_size),
                     float(capacity_factor) if capacity_factor else 0.0,
                     MOE_MODE_DISPATCH if mode == "dispatch" else MOE_MODE_MASK_SUM,
                     MOE_DTYPE_BF16 if dtype == "bf16" else MOE_DTYPE_FP32, int(bool(has_bias)),
                     int(group_limit or 0),
                     None if selection_bias is None
                     else _ptr(selection_bias, "selection_bias", torch.float32).value,
                     MOE_PRIORITY_SLOT if capacity_priority == "slot" else MOE_PRIORITY_TOKEN,
                     int(bool(training)))


def _check(status: int, func: str):
    if status != MOE_OK:
        raise MoeError(status, func, lib.moe_last_error().decode())


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def moe_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_packed_gate_up_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.moe_packed_gate_up_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_packed_gate_up_size")
    return n.value


def alloc_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    """Zeroed uint8 device buffer of moe_workspace_size(cfg) bytes (the zero status word
    starts clean)."""
    return torch.zeros(moe_workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_pack_weights(cfg, w_gate, w_up, w_gate_up_packed=None):
    dt = cfg.torch_dtype
    if w_gate_up_packed is None:
        n = moe_packed_gate_up_size(cfg) // w_gate.element_size()
        w_gate_up_packed = torch.empty(n, dtype=dt, device=w_gate.device)
    _check(lib.moe_pack_weights(ctypes.byref(cfg), _ptr(w_gate, "w_gate", dt),
                                _ptr(w_up, "w_up", dt),
                                _ptr(w_gate_up_packed, "w_gate_up_packed", dt), _stream()),
           "moe_pack_weights")
    return w_gate_up_packed


def moe_route(cfg, x, w_router, b_router, topk_idx, topk_w):
    dt = cfg.torch_dtype
    _check(lib.moe_route(ctypes.byref(cfg), _ptr(x, "x", dt), _ptr(w_router, "w_router", dt),
                         _ptr(b_router, "b_router", torch.float32),
                         _ptr(topk_idx, "topk_idx", torch.int32),
                         _ptr(topk_w, "topk_w", torch.float32), _stream()), "moe_route")


def moe_update_selection_bias(cfg, routed_counts, selection_bias, gamma):
    _check(lib.moe_update_selection_bias(ctypes.byref(cfg),
                                         _ptr(routed_counts, "routed_counts", torch.int32),
                                         _ptr(selection_bias, "selection_bias", torch.float32),
                                         ctypes.c_float(gamma), _stream()),
           "moe_update_selection_bias")


def moe_dispatch(cfg, topk_idx, x, routed_counts, counts, expert_offsets, part_offsets, perm,
                 slot_pos, send, workspace):
    dt = cfg.torch_dtype
    i32 = torch.int32
    _check(lib.moe_dispatch(ctypes.byref(cfg), _ptr(topk_idx, "topk_idx", i32), _ptr(x, "x", dt),
                            _ptr(routed_counts, "routed_counts", i32), _ptr(counts, "counts", i32),
                            _ptr(expert_offsets, "expert_offsets", i32),
                            _ptr(part_offsets, "part_offsets", i32), _ptr(perm, "perm", i32),
                            _ptr(slot_pos, "slot_pos", i32), _ptr(send, "send", dt),
                            _ptr(workspace, "workspace"), workspace.numel(), _stream()),
           "moe_dispatch")


def moe_dispatch_noalloc(cfg, topk_idx, x, routed_counts, counts, expert_offsets, part_offsets,
                         perm, slot_pos, send):
    """moe_dispatch for callers that cannot allocate: no workspace argument."""
    dt = cfg.torch_dtype
    i32 = torch.int32
    _check(lib.moe_dispatch_noalloc(
        ctypes.byref(cfg), _ptr(topk_idx, "topk_idx", i32), _ptr(x, "x", dt),
        _ptr(routed_counts, "routed_counts", i32), _ptr(counts, "counts", i32),
        _ptr(expert_offsets, "expert_offsets", i32), _ptr(part_offsets, "part_offsets", i32),
        _ptr(perm, "perm", i32), _ptr(slot_pos, "slot_pos", i32), _ptr(send, "send", dt),
        _stream()), "moe_dispatch_noalloc")


def moe_expert_ffn(cfg, send, expert_offsets, expert_begin, expert_end, w_gate_up_packed,
                   w_down, perm, topk_w, out_slots, workspace):
    dt = cfg.torch_dtype
    i32 = torch.int32
    _check(lib.moe_expert_ffn(ctypes.byref(cfg), _ptr(send, "send", dt),
                              _ptr(expert_offsets, "expert_offsets", i32), int(expert_begin),
                              int(expert_end), _ptr(w_gate_up_packed, "w_gate_up_packed", dt),
                              _ptr(w_down, "w_down", dt), _ptr(perm, "perm", i32),
                              _ptr(topk_w, "topk_w", torch.float32),
                              _ptr(out_slots, "out_slots", dt), _ptr(workspace, "workspace"),
                              workspace.numel(), _stream()), "moe_expert_ffn")


def moe_combine(cfg, out_slots, topk_idx, slot_pos, out, workspace):
    dt = cfg.torch_dtype
    i32 = torch.int32
    _check(lib.moe_combine(ctypes.byref(cfg), _ptr(out_slots, "out_slots", dt),
                           _ptr(topk_idx, "topk_idx", i32), _ptr(slot_pos, "slot_pos", i32),
                           _ptr(out, "out", dt), _ptr(workspace, "workspace"), workspace.numel(),
                           _stream()), "moe_combine")


def moe_layer_forward(cfg, x, w_router, b_router, w_gate_up_packed, w_down, out, workspace,
                      diag: Optional[dict] = None, stage_events=None):
    """diag: optional dict name -> preallocated tensor for any moe_diagnostics field.
    stage_events: optional list of MOE_NUM_STAGES + 1 torch.cuda.Event (already recorded
    once, so that their handles exist) to be recorded at the stage boundaries."""
    dt = cfg.torch_dtype
    dg = None
    keep = None
    if diag or stage_events:
        dg = MoeDiagnostics()
        if stage_events is not None:
            if len(stage_events) != MOE_NUM_STAGES + 1:
                raise ValueError("stage_events needs MOE_NUM_STAGES + 1 events")
            keep = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
            dg.stage_events = ctypes.cast(keep, ctypes.c_void_p).value
        for name in MoeDiagnostics._ARRAYS:
            if diag and diag.get(name) is not None:
                want = torch.float32 if name in ("topk_w", "router_logits") else torch.int32
                setattr(dg, name, _ptr(diag[name], name, want).value)
    _check(lib.moe_layer_forward(ctypes.byref(cfg), _ptr(x, "x", dt),
                                 _ptr(w_router, "w_router", dt),
                                 _ptr(b_router, "b_router", torch.float32),
                                 _ptr(w_gate_up_packed, "w_gate_up_packed", dt),
                                 _ptr(w_down, "w_down", dt), _ptr(out, "out", dt),
                                 ctypes.byref(dg) if dg is not None else None,
                                 _ptr(workspace, "workspace"), workspace.numel(), _stream()),
           "moe_layer_forward")


def moe_read_device_status(cfg, workspace, reset=True) -> int:
    flags = ctypes.c_int32(0)
    st = lib.moe_read_device_status(ctypes.byref(cfg), _ptr(workspace, "workspace"),
                                    workspace.numel(), ctypes.byref(flags), int(bool(reset)),
                                    _stream())
    if st not in (MOE_OK, MOE_ERR_TIMEOUT):
        _check(st, "moe_read_device_status")
    return flags.value


def moe_balance_stats(cfg, router_logits, routed_counts, load_frac, prob_mean, workspace):
    """Per-expert load share and mean router probability (moe.h)."""
    f32 = torch.float32
    _check(lib.moe_balance_stats(ctypes.byref(cfg), _ptr(router_logits, "router_logits", f32),
                                 _ptr(routed_counts, "routed_counts", torch.int32),
                                 _ptr(load_frac, "load_frac", f32),
                                 _ptr(prob_mean, "prob_mean", f32), _ptr(workspace, "workspace"),
                                 workspace.numel(), _stream()), "moe_balance_stats")


def moe_tp_slice(num_tokens, tp_size, tp_rank):
    """Token rows (begin, end) that TP rank tp_rank dispatches."""
    b, e = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.moe_tp_slice(int(num_tokens), int(tp_size), int(tp_rank), ctypes.byref(b),
                            ctypes.byref(e)), "moe_tp_slice")
    return b.value, e.value


def moe_tp_reduce(cfg, tp_size, padded, out):
    """out = sum over TP ranks, in order, of the zero-padded slice outputs padded[s]."""
    dt = cfg.torch_dtype
    _check(lib.moe_tp_reduce(ctypes.byref(cfg), int(tp_size), _ptr(padded, "padded", dt),
                             _ptr(out, "out", dt), _stream()), "moe_tp_reduce")


def moe_layer_backward(cfg, x, w_router, w_gate_up_packed, w_down, dout, dx, dw_router, db_router,
                       dw_gate, dw_up, dw_down, workspace):
    """Gradients of the layer (moe.h); after moe_layer_forward with cfg.training = 1 and
    the same workspace."""
    dt = cfg.torch_dtype
    f32 = torch.float32
    _check(lib.moe_layer_backward(
        ctypes.byref(cfg), _ptr(x, "x", dt), _ptr(w_router, "w_router", dt),
        _ptr(w_gate_up_packed, "w_gate_up_packed", dt), _ptr(w_down, "w_down", dt),
        _ptr(dout, "dout", dt), _ptr(dx, "dx", dt), _ptr(dw_router, "dw_router", f32),
        _ptr(db_router, "db_router", f32), _ptr(dw_gate, "dw_gate", dt), _ptr(dw_up, "dw_up", dt),
        _ptr(dw_down, "dw_down", dt), _ptr(workspace, "workspace"), workspace.numel(), _stream()),
        "moe_layer_backward")


def moe_check_wait_timeout(cfg, workspace):
    """Enqueues the bounded-wait check (moe.h); read the result with
    moe_read_device_status."""
    _check(lib.moe_check_wait_timeout(ctypes.byref(cfg), _ptr(workspace, "workspace"),
                                      workspace.numel(), _stream()), "moe_check_wait_timeout")
