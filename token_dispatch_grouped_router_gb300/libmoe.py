"""ctypes binding of libmoe: the C-ABI entry points under the same names.

Argument marshalling only: each wrapper checks shapes/dtypes of the torch
tensors it is given, passes their device pointers and the current CUDA stream
to the library and raises ``MoEError`` on a non-zero status.  Every step of
the layer runs in the library's CUDA kernels; there is no fallback.  If the
library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t

# (name, restype, argtypes) exactly as declared in include/libmoe.h
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "moe_reset_status": (_I, [_P, _P]),
    "moe_get_status": (_I, [_P, _P, _P]),
    "moe_router_logits": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_router_logits_tc": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_router_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_router_gates": (_I, [_P, _I, _I, _P, _P]),
    "moe_router_topk_bwd": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_router_logits_bwd": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_router_logits_bwd_topk": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                        _Z, _P]),
    "moe_expert_offsets": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_offsets_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_expert_offsets_capacity": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_dispatch_rows_capacity": (_I, [_P, _I, _I, _I, _P, _P, _I, _I, _P, _P]),
    "moe_combine_capacity": (_I, [_P, _I, _I, _P, _P, _I, _I, _I, _P, _P]),
    "moe_combine_bwd_capacity": (_I, [_P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_dispatch_rows": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_combine_bwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_swiglu_fwd": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _Z, _P]),
    "moe_grouped_swiglu_bwd": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_mxfp8_quantize_rows": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_mxfp8_quantize_weights": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_mxfp8_quantize_weights_f32": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_mxfp8_dequantize_rows": (_I, [_P, _P, _I, _I, _P, _P]),
    "moe_dispatch_rows_mxfp8": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_mxfp8_weight_atom_bytes": (_Z, [_I, _I, _I]),
    "moe_mxfp8_dx_weight_atom_bytes": (_Z, [_I, _I, _I]),
    "moe_grouped_swiglu_bwd_dact_mxfp8": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                               _P, _P, _P, _P, _Z, _P]),
    "moe_mxfp8_dx_weight_scale_atoms": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_grouped_swiglu_bwd_dx_mxfp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                             _P, _Z, _P]),
    "moe_mxfp8_weight_scale_atoms": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_grouped_swiglu_fwd_mxfp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _P, _P, _Z, _P]),
    "moe_grouped_swiglu_fwd_up": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_grouped_swiglu_fwd_down": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "moe_grouped_swiglu_bwd_dact": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_grouped_swiglu_bwd_dx": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_grouped_swiglu_bwd_wgrad": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _Z, _P]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, call: str, status: int):
        msg = load().moe_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{call} failed with status {status}: {msg}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (once) and declare every entry point's signature."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"libmoe.so not found at {path}; build it with "
                "`python -m token_dispatch_grouped_router_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ok(name: str, status: int) -> None:
    if status != 0:
        raise MoEError(name, status)


def _want(t: torch.Tensor, dtype: torch.dtype, shape, name: str) -> None:
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


# ------------------------------------------------------------------ misc

def moe_version() -> int:
    return load().moe_version()


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


def moe_workspace_size(T: int, E: int, k: int, d: int, h: int) -> int:
    return int(load().moe_workspace_size(T, E, k, d, h))


def moe_reset_status(ws: torch.Tensor) -> None:
    _ok("moe_reset_status", load().moe_reset_status(_ptr(ws), _stream()))


def moe_get_status(ws: torch.Tensor) -> int:
    out = ctypes.c_int32(0)
    _ok("moe_get_status", load().moe_get_status(_ptr(ws), ctypes.byref(out), _stream()))
    return int(out.value)


# ---------------------------------------------------------------- router

def moe_router_logits(x, W_r, b, logits) -> None:
    T, d = x.shape
    E = W_r.shape[1]
    _want(x, torch.bfloat16, (T, d), "x"); _want(W_r, torch.float32, (d, E), "W_r")
    _want(logits, torch.float32, (T, E), "logits")
    if b is not None:
        _want(b, torch.float32, (E,), "b")
    _ok("moe_router_logits", load().moe_router_logits(
        _ptr(x), _ptr(W_r), _ptr(b), T, d, E, _ptr(logits), _stream()))


def moe_router_logits_tc(x, W_r, b, logits, ws) -> None:
    """moe_router_logits on the tensor cores (W_r split into three bf16 parts
    in the workspace; fp32 accuracy)."""
    T, d = x.shape
    E = W_r.shape[1]
    _want(x, torch.bfloat16, (T, d), "x"); _want(W_r, torch.float32, (d, E), "W_r")
    _want(logits, torch.float32, (T, E), "logits")
    if b is not None:
        _want(b, torch.float32, (E,), "b")
    _ok("moe_router_logits_tc", load().moe_router_logits_tc(
        _ptr(x), _ptr(W_r), _ptr(b), T, d, E, _ptr(logits), _ptr(ws), _wsb(ws), _stream()))


def moe_router_topk(logits, k: int, topk_idx, topk_gate) -> None:
    T, E = logits.shape
    _want(logits, torch.float32, (T, E), "logits")
    _want(topk_idx, torch.int32, (T, k), "topk_idx"); _want(topk_gate, torch.float32, (T, k), "topk_gate")
    _ok("moe_router_topk", load().moe_router_topk(
        _ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_gate), _stream()))


def moe_router_gates(sel_logits, topk_gate) -> None:
    T, k = sel_logits.shape
    _want(sel_logits, torch.float32, (T, k), "sel_logits")
    _want(topk_gate, torch.float32, (T, k), "topk_gate")
    _ok("moe_router_gates", load().moe_router_gates(_ptr(sel_logits), T, k, _ptr(topk_gate), _stream()))


def moe_router_topk_bwd(topk_gate, d_gate, topk_idx, E: int, d_logits) -> None:
    T, k = topk_gate.shape
    _want(d_gate, torch.float32, (T, k), "d_gate"); _want(topk_idx, torch.int32, (T, k), "topk_idx")
    _want(d_logits, torch.float32, (T, E), "d_logits")
    _ok("moe_router_topk_bwd", load().moe_router_topk_bwd(
        _ptr(topk_gate), _ptr(d_gate), _ptr(topk_idx), T, E, k, _ptr(d_logits), _stream()))


def moe_router_logits_bwd(x, W_r, d_logits, dx, dW_r, db, ws) -> None:
    T, d = x.shape
    E = W_r.shape[1]
    _want(d_logits, torch.float32, (T, E), "d_logits"); _want(dx, torch.bfloat16, (T, d), "dx")
    _want(dW_r, torch.float32, (d, E), "dW_r")
    _ok("moe_router_logits_bwd", load().moe_router_logits_bwd(
        _ptr(x), _ptr(W_r), _ptr(d_logits), T, d, E, _ptr(dx), _ptr(dW_r), _ptr(db),
        _ptr(ws), ws.numel() * ws.element_size(), _stream()))


def moe_router_logits_bwd_topk(x, W_r, d_logits, topk_idx, offsets, slot_of_row, dx, dW_r, db,
                               ws) -> None:
    """moe_router_logits_bwd for d_logits that is zero outside the top-k
    selection (as moe_router_topk_bwd writes it), through the route map."""
    T, d = x.shape
    E = W_r.shape[1]
    k = topk_idx.shape[1]
    _want(d_logits, torch.float32, (T, E), "d_logits"); _want(dx, torch.bfloat16, (T, d), "dx")
    _want(dW_r, torch.float32, (d, E), "dW_r"); _want(topk_idx, torch.int32, (T, k), "topk_idx")
    _want(offsets, torch.int32, (E + 1,), "offsets"); _want(slot_of_row, torch.int32, (T * k,), "slot_of_row")
    _ok("moe_router_logits_bwd_topk", load().moe_router_logits_bwd_topk(
        _ptr(x), _ptr(W_r), _ptr(d_logits), _ptr(topk_idx), _ptr(offsets), _ptr(slot_of_row),
        T, d, E, k, _ptr(dx), _ptr(dW_r), _ptr(db), _ptr(ws), _wsb(ws), _stream()))


# ------------------------------------------------------------- route map

def moe_expert_offsets(topk_idx, E: int, counts, offsets, row_of_slot, slot_of_row, ws) -> None:
    T, k = topk_idx.shape
    _want(topk_idx, torch.int32, (T, k), "topk_idx"); _want(counts, torch.int32, (E,), "counts")
    _want(offsets, torch.int32, (E + 1,), "offsets")
    _want(row_of_slot, torch.int32, (T * k,), "row_of_slot")
    _want(slot_of_row, torch.int32, (T * k,), "slot_of_row")
    _ok("moe_expert_offsets", load().moe_expert_offsets(
        _ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(row_of_slot),
        _ptr(slot_of_row), _ptr(ws), ws.numel() * ws.element_size(), _stream()))


def moe_expert_offsets_noalloc(topk_idx, E: int, counts, offsets, row_of_slot, slot_of_row,
                               status=None) -> None:
    """moe_expert_offsets without a workspace (static device scratch inside
    the library; T*k <= 262144; see include/libmoe.h)."""
    T, k = topk_idx.shape
    _want(topk_idx, torch.int32, (T, k), "topk_idx"); _want(counts, torch.int32, (E,), "counts")
    _want(offsets, torch.int32, (E + 1,), "offsets")
    _want(row_of_slot, torch.int32, (T * k,), "row_of_slot")
    _want(slot_of_row, torch.int32, (T * k,), "slot_of_row")
    if status is not None:
        _want(status, torch.int32, (1,), "status")
        if status.device != topk_idx.device:
            raise ValueError(f"status: expected a tensor on {topk_idx.device}, got {status.device}")
    _ok("moe_expert_offsets_noalloc", load().moe_expert_offsets_noalloc(
        _ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(row_of_slot),
        _ptr(slot_of_row), _ptr(status), _stream()))


# ------------------------------------------------ capacity-padded layer

def moe_expert_offsets_capacity(topk_idx, E: int, C: int, counts, offsets, row_of_slot,
                                slot_of_row, ws, routed=None) -> None:
    T, k = topk_idx.shape
    _want(topk_idx, torch.int32, (T, k), "topk_idx"); _want(counts, torch.int32, (E,), "counts")
    _want(offsets, torch.int32, (E + 1,), "offsets")
    _want(row_of_slot, torch.int32, (T * k,), "row_of_slot")
    _want(slot_of_row, torch.int32, (E * C,), "slot_of_row")
    if routed is not None:
        _want(routed, torch.int32, (E,), "routed")
    _ok("moe_expert_offsets_capacity", load().moe_expert_offsets_capacity(
        _ptr(topk_idx), T, k, E, C, _ptr(counts), _ptr(offsets), _ptr(row_of_slot),
        _ptr(slot_of_row), _ptr(routed), _ptr(ws), _wsb(ws), _stream()))


def moe_dispatch_rows_capacity(x, row_of_slot, counts, k: int, C: int, xp) -> None:
    T, d = x.shape
    E = counts.shape[0]
    _want(x, torch.bfloat16, (T, d), "x"); _want(xp, torch.bfloat16, (E * C, d), "xp")
    _want(row_of_slot, torch.int32, (T * k,), "row_of_slot"); _want(counts, torch.int32, (E,), "counts")
    _ok("moe_dispatch_rows_capacity", load().moe_dispatch_rows_capacity(
        _ptr(x), T, d, k, _ptr(row_of_slot), _ptr(counts), E, C, _ptr(xp), _stream()))


def moe_combine_capacity(yp, E: int, C: int, row_of_slot, gate, k: int, out) -> None:
    T, d = out.shape
    _want(yp, torch.bfloat16, (E * C, d), "yp"); _want(out, torch.bfloat16, (T, d), "out")
    _want(row_of_slot, torch.int32, (T * k,), "row_of_slot")
    if gate is not None:
        _want(gate, torch.float32, (T, k), "gate")
    _ok("moe_combine_capacity", load().moe_combine_capacity(
        _ptr(yp), E, C, _ptr(row_of_slot), _ptr(gate), T, k, d, _ptr(out), _stream()))


def moe_combine_bwd_capacity(dout, yp, C: int, row_of_slot, counts, gate, k: int, dyp, dgate) -> None:
    T, d = dout.shape
    E = counts.shape[0]
    _want(yp, torch.bfloat16, (E * C, d), "yp"); _want(dyp, torch.bfloat16, (E * C, d), "dyp")
    _want(row_of_slot, torch.int32, (T * k,), "row_of_slot"); _want(counts, torch.int32, (E,), "counts")
    _want(gate, torch.float32, (T, k), "gate"); _want(dgate, torch.float32, (T, k), "dgate")
    _ok("moe_combine_bwd_capacity", load().moe_combine_bwd_capacity(
        _ptr(dout), _ptr(yp), E, C, _ptr(row_of_slot), _ptr(counts), _ptr(gate), T, k, d,
        _ptr(dyp), _ptr(dgate), _stream()))


# ------------------------------------------------------- dispatch/combine

def moe_dispatch_rows(x, row_of_slot, k: int, xp) -> None:
    T, d = x.shape
    _want(x, torch.bfloat16, (T, d), "x"); _want(xp, torch.bfloat16, (T * k, d), "xp")
    _ok("moe_dispatch_rows", load().moe_dispatch_rows(
        _ptr(x), T, d, k, _ptr(row_of_slot), _ptr(xp), _stream()))


def moe_combine(yp, row_of_slot, gate, k: int, out) -> None:
    T, d = out.shape
    _want(yp, torch.bfloat16, (T * k, d), "yp"); _want(out, torch.bfloat16, (T, d), "out")
    if gate is not None:
        _want(gate, torch.float32, (T, k), "gate")
    _ok("moe_combine", load().moe_combine(
        _ptr(yp), _ptr(row_of_slot), _ptr(gate), T, k, d, _ptr(out), _stream()))


def moe_combine_bwd(dout, yp, row_of_slot, gate, k: int, dyp, dgate) -> None:
    T, d = dout.shape
    _want(yp, torch.bfloat16, (T * k, d), "yp"); _want(dyp, torch.bfloat16, (T * k, d), "dyp")
    _want(gate, torch.float32, (T, k), "gate"); _want(dgate, torch.float32, (T, k), "dgate")
    _ok("moe_combine_bwd", load().moe_combine_bwd(
        _ptr(dout), _ptr(yp), _ptr(row_of_slot), _ptr(gate), T, k, d, _ptr(dyp), _ptr(dgate),
        _stream()))


# ------------------------------------------------------ grouped SwiGLU GEMM

def moe_grouped_swiglu_fwd(xp, offsets, W1, W3, W2, h1, h3, a, yp, ws) -> None:
    R, d = xp.shape
    E, _, h = W1.shape
    _want(W1, torch.bfloat16, (E, d, h), "W1"); _want(W3, torch.bfloat16, (E, d, h), "W3")
    _want(W2, torch.bfloat16, (E, h, d), "W2"); _want(offsets, torch.int32, (E + 1,), "offsets")
    for n, t in (("h1", h1), ("h3", h3), ("a", a)):
        _want(t, torch.bfloat16, (R, h), n)
    _want(yp, torch.bfloat16, (R, d), "yp")
    _ok("moe_grouped_swiglu_fwd", load().moe_grouped_swiglu_fwd(
        _ptr(xp), _ptr(offsets), R, E, d, h, _ptr(W1), _ptr(W3), _ptr(W2), _ptr(h1), _ptr(h3),
        _ptr(a), _ptr(yp), _ptr(ws), ws.numel() * ws.element_size(), _stream()))


def moe_grouped_swiglu_bwd(xp, offsets, W1, W3, W2, h1, h3, a, dyp, dh1, dh3, dxp,
                           dW1, dW3, dW2, ws) -> None:
    R, d = xp.shape
    E, _, h = W1.shape
    for n, t in (("h1", h1), ("h3", h3), ("a", a), ("dh1", dh1), ("dh3", dh3)):
        _want(t, torch.bfloat16, (R, h), n)
    _want(dyp, torch.bfloat16, (R, d), "dyp"); _want(dxp, torch.bfloat16, (R, d), "dxp")
    _want(dW1, torch.bfloat16, (E, d, h), "dW1"); _want(dW3, torch.bfloat16, (E, d, h), "dW3")
    _want(dW2, torch.bfloat16, (E, h, d), "dW2")
    _ok("moe_grouped_swiglu_bwd", load().moe_grouped_swiglu_bwd(
        _ptr(xp), _ptr(offsets), R, E, d, h, _ptr(W1), _ptr(W3), _ptr(W2), _ptr(h1), _ptr(h3),
        _ptr(a), _ptr(dyp), _ptr(dh1), _ptr(dh3), _ptr(dxp), _ptr(dW1), _ptr(dW3), _ptr(dW2),
        _ptr(ws), ws.numel() * ws.element_size(), _stream()))


def _wsb(ws):
    return ws.numel() * ws.element_size()


def moe_grouped_swiglu_fwd_up(xp, offsets, W1, W3, h1, h3, a, ws) -> None:
    R, d = xp.shape
    E, _, h = W1.shape
    for n, t in (("h1", h1), ("h3", h3), ("a", a)):
        _want(t, torch.bfloat16, (R, h), n)
    _want(W3, torch.bfloat16, (E, d, h), "W3")
    _ok("moe_grouped_swiglu_fwd_up", load().moe_grouped_swiglu_fwd_up(
        _ptr(xp), _ptr(offsets), R, E, d, h, _ptr(W1), _ptr(W3), _ptr(h1), _ptr(h3), _ptr(a),
        _ptr(ws), _wsb(ws), _stream()))


def moe_grouped_swiglu_fwd_down(a, offsets, W2, yp, ws) -> None:
    R, h = a.shape
    E, _, d = W2.shape
    _want(W2, torch.bfloat16, (E, h, d), "W2"); _want(yp, torch.bfloat16, (R, d), "yp")
    _ok("moe_grouped_swiglu_fwd_down", load().moe_grouped_swiglu_fwd_down(
        _ptr(a), _ptr(offsets), R, E, d, h, _ptr(W2), _ptr(yp), _ptr(ws), _wsb(ws), _stream()))


def moe_grouped_swiglu_bwd_dact(offsets, W2, h1, h3, dyp, dh1, dh3, ws) -> None:
    R, d = dyp.shape
    E, h, _ = W2.shape
    for n, t in (("h1", h1), ("h3", h3), ("dh1", dh1), ("dh3", dh3)):
        _want(t, torch.bfloat16, (R, h), n)
    _ok("moe_grouped_swiglu_bwd_dact", load().moe_grouped_swiglu_bwd_dact(
        _ptr(offsets), R, E, d, h, _ptr(W2), _ptr(h1), _ptr(h3), _ptr(dyp), _ptr(dh1),
        _ptr(dh3), _ptr(ws), _wsb(ws), _stream()))


def moe_grouped_swiglu_bwd_dx(offsets, W1, W3, dh1, dh3, dxp, ws) -> None:
    R, d = dxp.shape
    E, _, h = W1.shape
    _want(dh1, torch.bfloat16, (R, h), "dh1"); _want(dh3, torch.bfloat16, (R, h), "dh3")
    _want(W3, torch.bfloat16, (E, d, h), "W3")
    _ok("moe_grouped_swiglu_bwd_dx", load().moe_grouped_swiglu_bwd_dx(
        _ptr(offsets), R, E, d, h, _ptr(W1), _ptr(W3), _ptr(dh1), _ptr(dh3), _ptr(dxp),
        _ptr(ws), _wsb(ws), _stream()))


def moe_grouped_swiglu_bwd_wgrad(xp, offsets, a, dyp, dh1, dh3, dW1, dW3, dW2, ws) -> None:
    R, d = xp.shape
    E, _, h = dW1.shape
    for n, t in (("a", a), ("dh1", dh1), ("dh3", dh3)):
        _want(t, torch.bfloat16, (R, h), n)
    _want(dyp, torch.bfloat16, (R, d), "dyp")
    _want(dW1, torch.bfloat16, (E, d, h), "dW1"); _want(dW3, torch.bfloat16, (E, d, h), "dW3")
    _want(dW2, torch.bfloat16, (E, h, d), "dW2")
    _ok("moe_grouped_swiglu_bwd_wgrad", load().moe_grouped_swiglu_bwd_wgrad(
        _ptr(xp), _ptr(offsets), R, E, d, h, _ptr(a), _ptr(dyp), _ptr(dh1), _ptr(dh3),
        _ptr(dW1), _ptr(dW3), _ptr(dW2), _ptr(ws), ws.numel() * ws.element_size(), _stream()))


# ------------------------------------------------------------------ MXFP8

def moe_mxfp8_quantize_rows(src, q, scale) -> None:
    rows, K = src.shape
    _want(src, torch.bfloat16, (rows, K), "src"); _want(q, torch.uint8, (rows, K), "q")
    _want(scale, torch.uint8, (rows, K // 32), "scale")
    _ok("moe_mxfp8_quantize_rows", load().moe_mxfp8_quantize_rows(
        _ptr(src), rows, K, _ptr(q), _ptr(scale), _stream()))


def moe_mxfp8_quantize_weights(W, wq, ws) -> None:
    E, K, N = W.shape
    _want(W, torch.bfloat16, (E, K, N), "W"); _want(wq, torch.uint8, (E, N, K), "wq")
    _want(ws, torch.uint8, (E, N, K // 32), "ws")
    _ok("moe_mxfp8_quantize_weights", load().moe_mxfp8_quantize_weights(
        _ptr(W), E, K, N, _ptr(wq), _ptr(ws), _stream()))


def moe_mxfp8_quantize_weights_f32(W, wq, ws) -> None:
    E, K, N = W.shape
    _want(W, torch.float32, (E, K, N), "W"); _want(wq, torch.uint8, (E, N, K), "wq")
    _want(ws, torch.uint8, (E, N, K // 32), "ws")
    _ok("moe_mxfp8_quantize_weights_f32", load().moe_mxfp8_quantize_weights_f32(
        _ptr(W), E, K, N, _ptr(wq), _ptr(ws), _stream()))


def moe_mxfp8_dequantize_rows(q, scale, out) -> None:
    rows, K = q.shape
    _want(q, torch.uint8, (rows, K), "q"); _want(scale, torch.uint8, (rows, K // 32), "scale")
    _want(out, torch.bfloat16, (rows, K), "out")
    _ok("moe_mxfp8_dequantize_rows", load().moe_mxfp8_dequantize_rows(
        _ptr(q), _ptr(scale), rows, K, _ptr(out), _stream()))


def moe_dispatch_rows_mxfp8(x, row_of_slot, k: int, xq, xs, xp=None) -> None:
    T, d = x.shape
    _want(x, torch.bfloat16, (T, d), "x"); _want(xq, torch.uint8, (T * k, d), "xq")
    _want(xs, torch.uint8, (T * k, d // 32), "xs")
    if xp is not None:
        _want(xp, torch.bfloat16, (T * k, d), "xp")
    _ok("moe_dispatch_rows_mxfp8", load().moe_dispatch_rows_mxfp8(
        _ptr(x), T, d, k, _ptr(row_of_slot), _ptr(xq), _ptr(xs), _ptr(xp), _stream()))


def moe_mxfp8_weight_atom_bytes(E: int, d: int, h: int) -> int:
    return int(load().moe_mxfp8_weight_atom_bytes(E, d, h))


def moe_mxfp8_weight_scale_atoms(w1s, w3s, w2s, atoms) -> None:
    """The row-major weight scales in the atom order of the block-scaled GEMM's
    tiles (see include/libmoe.h)."""
    E, h, kd = w1s.shape
    d = kd * 32
    _want(w1s, torch.uint8, (E, h, d // 32), "w1s"); _want(w3s, torch.uint8, (E, h, d // 32), "w3s")
    _want(w2s, torch.uint8, (E, d, h // 32), "w2s")
    _want(atoms, torch.uint8, (moe_mxfp8_weight_atom_bytes(E, d, h),), "atoms")
    _ok("moe_mxfp8_weight_scale_atoms", load().moe_mxfp8_weight_scale_atoms(
        _ptr(w1s), _ptr(w3s), _ptr(w2s), E, d, h, _ptr(atoms), _stream()))


def moe_grouped_swiglu_fwd_mxfp8(xq, xs, offsets, w1q, w3q, w2q, w_atoms,
                                 h1, h3, a, aq, as_, yp, ws) -> None:
    R, d = xq.shape
    E, h, _ = w1q.shape
    _want(xs, torch.uint8, (R, d // 32), "xs")
    for n, t in (("w1q", w1q), ("w3q", w3q)):
        _want(t, torch.uint8, (E, h, d), n)
    _want(w2q, torch.uint8, (E, d, h), "w2q")
    _want(w_atoms, torch.uint8, (moe_mxfp8_weight_atom_bytes(E, d, h),), "w_atoms")
    for n, t in (("h1", h1), ("h3", h3), ("a", a)):
        if t is not None or n != "a":             # a may be None: quantised a only
            _want(t, torch.bfloat16, (R, h), n)
    _want(aq, torch.uint8, (R, h), "aq"); _want(as_, torch.uint8, (R, h // 32), "as")
    _want(yp, torch.bfloat16, (R, d), "yp")
    _ok("moe_grouped_swiglu_fwd_mxfp8", load().moe_grouped_swiglu_fwd_mxfp8(
        _ptr(xq), _ptr(xs), _ptr(offsets), R, E, d, h, _ptr(w1q), _ptr(w3q), _ptr(w2q),
        _ptr(w_atoms), _ptr(h1), _ptr(h3), _ptr(a), _ptr(aq), _ptr(as_), _ptr(yp),
        _ptr(ws), _wsb(ws), _stream()))


def moe_mxfp8_dx_weight_atom_bytes(E: int, d: int, h: int) -> int:
    return int(load().moe_mxfp8_dx_weight_atom_bytes(E, d, h))


def moe_mxfp8_dx_weight_scale_atoms(w1s_h, w3s_h, atoms) -> None:
    """Scales of W1/W3 quantised along h ([E][d][h/32]) in the atom order of
    the MXFP8 dgrad GEMM."""
    E, d, kh = w1s_h.shape
    h = kh * 32
    _want(w1s_h, torch.uint8, (E, d, h // 32), "w1s_h"); _want(w3s_h, torch.uint8, (E, d, h // 32), "w3s_h")
    _want(atoms, torch.uint8, (moe_mxfp8_dx_weight_atom_bytes(E, d, h),), "atoms")
    _ok("moe_mxfp8_dx_weight_scale_atoms", load().moe_mxfp8_dx_weight_scale_atoms(
        _ptr(w1s_h), _ptr(w3s_h), E, d, h, _ptr(atoms), _stream()))


def moe_grouped_swiglu_bwd_dx_mxfp8(dh1q, dh1s, dh3q, dh3s, offsets, w1q_h, w3q_h, dx_atoms,
                                    dxp, ws) -> None:
    R, h = dh1q.shape
    E, d, _ = w1q_h.shape
    for n, t in (("dh1q", dh1q), ("dh3q", dh3q)):
        _want(t, torch.uint8, (R, h), n)
    for n, t in (("dh1s", dh1s), ("dh3s", dh3s)):
        _want(t, torch.uint8, (R, h // 32), n)
    for n, t in (("w1q_h", w1q_h), ("w3q_h", w3q_h)):
        _want(t, torch.uint8, (E, d, h), n)
    _want(dx_atoms, torch.uint8, (moe_mxfp8_dx_weight_atom_bytes(E, d, h),), "dx_atoms")
    _want(dxp, torch.bfloat16, (R, d), "dxp")
    _ok("moe_grouped_swiglu_bwd_dx_mxfp8", load().moe_grouped_swiglu_bwd_dx_mxfp8(
        _ptr(dh1q), _ptr(dh1s), _ptr(dh3q), _ptr(dh3s), _ptr(offsets), R, E, d, h, _ptr(w1q_h),
        _ptr(w3q_h), _ptr(dx_atoms), _ptr(dxp), _ptr(ws), _wsb(ws), _stream()))


def moe_grouped_swiglu_bwd_dact_mxfp8(offsets, W2, h1, h3, dyp, dh1, dh3, dh1q, dh1s, dh3q, dh3s,
                                      ws) -> None:
    """moe_grouped_swiglu_bwd_dact that also writes dh1 / dh3 quantised along h."""
    R, d = dyp.shape
    E, h, _ = W2.shape
    for n, t in (("h1", h1), ("h3", h3), ("dh1", dh1), ("dh3", dh3)):
        _want(t, torch.bfloat16, (R, h), n)
    for n, t in (("dh1q", dh1q), ("dh3q", dh3q)):
        _want(t, torch.uint8, (R, h), n)
    for n, t in (("dh1s", dh1s), ("dh3s", dh3s)):
        _want(t, torch.uint8, (R, h // 32), n)
    _ok("moe_grouped_swiglu_bwd_dact_mxfp8", load().moe_grouped_swiglu_bwd_dact_mxfp8(
        _ptr(offsets), R, E, d, h, _ptr(W2), _ptr(h1), _ptr(h3), _ptr(dyp), _ptr(dh1), _ptr(dh3),
        _ptr(dh1q), _ptr(dh1s), _ptr(dh3q), _ptr(dh3s), _ptr(ws), _wsb(ws), _stream()))
