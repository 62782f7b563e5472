"""Python binding of the C ABI in include/moe.h (argument marshalling only).

Every function has the name of the C entry point it calls and takes torch
tensors where the C function takes device pointers; the computation happens
in the CUDA library.  A non-zero status raises :class:`MoEError`.  If the
library cannot be built or loaded, the first call raises: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional

import torch

from . import _build
from .workloads import ACT_SWIGLU, GATE_SOFTMAX, MoEInputs

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5

GATE_CODES = {GATE_SOFTMAX: 0, "sigmoid_bias": 1}
ACT_CODES = {"relu": 0, ACT_SWIGLU: 1}
DTYPE_CODES = {"f32": 0, "bf16": 1}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str, cuda_error: int):
        super().__init__(f"{fn}: {message} (status {status}, cuda error {cuda_error})")
        self.status = status
        self.cuda_error = cuda_error


class moe_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "H", "n_routed", "n_shared", "top_k", "inter", "gate", "act", "dtype",
                 "n_groups", "topk_groups")]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("centroids", "logit_offset", "select_bias", "w1", "w3", "w2",
                 "sw1", "sw3", "sw2")]


class moe_route_outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "topk_idx", "topk_w", "expert_offsets")]


class moe_weight_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("d_centroids", "dw1", "dw3", "dw2", "dsw1", "dsw3", "dsw2")]


_P = ctypes.c_void_p
_S = ctypes.POINTER(moe_shape)
_W = ctypes.POINTER(moe_weights)
_SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_cuda_error": (ctypes.c_int, []),
    "moe_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_dispatch_workspace_size": (ctypes.c_size_t, [_S]),
    "moe_expert_ffn_workspace_size": (ctypes.c_size_t, [_S]),
    "moe_layer_workspace_size": (ctypes.c_size_t, [_S]),
    "moe_router_logits_workspace_size": (ctypes.c_size_t, [_S]),
    "moe_router_logits": (ctypes.c_int, [_S, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_route": (ctypes.c_int, [_S, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch": (ctypes.c_int, [_S, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_S, _W, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_S, _P, _P, _P, _P, _P, _P, _P]),
    "moe_layer_forward": (ctypes.c_int, [_S, _W, _P, _P, ctypes.POINTER(moe_route_outputs),
                                         _P, ctypes.c_size_t, _P]),
    "moe_layer_forward_host": (ctypes.c_int, [_S, _W, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_layer_forward_host_stream": (ctypes.c_int, [_S, _W, ctypes.c_int, ctypes.POINTER(_P),
                                                     ctypes.POINTER(_P), _P, _P, _P,
                                                     ctypes.c_size_t, _P]),
    "moe_dispatch_static": (ctypes.c_int, [_S, _P, _P, _P, _P, _P, _P, _P]),
    "moe_update_select_bias": (ctypes.c_int, [_S, _P, _P, ctypes.c_float, _P, _P]),
    "moe_balance_stats_workspace_size": (ctypes.c_size_t, [_S]),
    "moe_layer_backward_workspace_size": (ctypes.c_size_t, [_S]),
    "moe_layer_backward": (ctypes.c_int, [_S, _W, _P, _P, _P, ctypes.POINTER(moe_weight_grads),
                                          _P, ctypes.c_size_t, _P, ctypes.c_size_t, _P]),
    "moe_layer_saved_size": (ctypes.c_size_t, [_S]),
    "moe_check_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, _P]),
    "moe_layer_forward_train": (ctypes.c_int, [_S, _W, _P, _P, _P, ctypes.c_size_t, _P,
                                               ctypes.c_size_t, _P]),
    "moe_balance_stats": (ctypes.c_int, [_S, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_ffn_rows_workspace_size": (ctypes.c_size_t, [_S, ctypes.c_int64]),
    "moe_expert_ffn_rows": (ctypes.c_int, [_S, _W, ctypes.c_int64, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_size_t, _P]),
    "moe_ep_regroup": (ctypes.c_int, [_S, ctypes.c_int32, _P, ctypes.c_int64, _P, _P, _P,
                                      ctypes.c_int32, _P]),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (built first if missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            handle = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def library_path() -> str:
    return _build.LIB


def shape_struct(s) -> moe_shape:
    if isinstance(s, moe_shape):
        return s
    return moe_shape(s.T, s.H, s.n_routed, s.n_shared, s.top_k, s.inter,
                     GATE_CODES[s.gate], ACT_CODES[s.act], DTYPE_CODES[s.dtype],
                     s.n_groups, s.topk_groups)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr() or None


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(fn: str, status: int):
    if status != MOE_OK:
        L = lib()
        raise MoEError(fn, status, L.moe_status_string(status).decode(), L.moe_last_cuda_error())


def weights_struct(inp: MoEInputs) -> moe_weights:
    """C weight struct pointing at the tensors of ``inp`` (keep ``inp`` alive)."""
    return moe_weights(_ptr(inp.centroids), _ptr(inp.logit_offset), _ptr(inp.select_bias),
                       _ptr(inp.w1), _ptr(inp.w3), _ptr(inp.w2),
                       _ptr(inp.sw1) if inp.sw1.numel() else None,
                       _ptr(inp.sw3) if inp.sw3 is not None and inp.sw3.numel() else None,
                       _ptr(inp.sw2) if inp.sw2.numel() else None)


def moe_dispatch_workspace_size(shape) -> int:
    return lib().moe_dispatch_workspace_size(ctypes.byref(shape_struct(shape)))


def moe_expert_ffn_workspace_size(shape) -> int:
    return lib().moe_expert_ffn_workspace_size(ctypes.byref(shape_struct(shape)))


def moe_layer_workspace_size(shape) -> int:
    return lib().moe_layer_workspace_size(ctypes.byref(shape_struct(shape)))


def moe_router_logits_workspace_size(shape) -> int:
    return lib().moe_router_logits_workspace_size(ctypes.byref(shape_struct(shape)))


def moe_balance_stats_workspace_size(shape) -> int:
    return lib().moe_balance_stats_workspace_size(ctypes.byref(shape_struct(shape)))


def moe_device_status(stream=None):
    """(status, raw device error word); synchronises the stream."""
    code = ctypes.c_int32(0)
    st = lib().moe_device_status(_stream(stream), ctypes.byref(code))
    return st, code.value


def moe_router_logits(shape, u, centroids, logit_offset, logits, ws=None, stream=None):
    _check("moe_router_logits", lib().moe_router_logits(
        ctypes.byref(shape_struct(shape)), _ptr(u), _ptr(centroids), _ptr(logit_offset),
        _ptr(logits), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_route(shape, logits, select_bias, topk_idx, topk_w, kth_gap=None, stream=None):
    _check("moe_route", lib().moe_route(
        ctypes.byref(shape_struct(shape)), _ptr(logits), _ptr(select_bias), _ptr(topk_idx),
        _ptr(topk_w), _ptr(kth_gap), _stream(stream)))


def moe_dispatch(shape, topk_idx, u, expert_offsets, row_token, slot_row, u_perm, ws,
                 stream=None):
    _check("moe_dispatch", lib().moe_dispatch(
        ctypes.byref(shape_struct(shape)), _ptr(topk_idx), _ptr(u), _ptr(expert_offsets),
        _ptr(row_token), _ptr(slot_row), _ptr(u_perm), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_dispatch_static(shape, topk_idx, u, expert_offsets, row_token, slot_row, u_perm,
                        stream=None):
    """moe_dispatch for callers that cannot provide device scratch: the library
    uses its own fixed array (see include/moe.h for the size limit)."""
    _check("moe_dispatch_static", lib().moe_dispatch_static(
        ctypes.byref(shape_struct(shape)), _ptr(topk_idx), _ptr(u), _ptr(expert_offsets),
        _ptr(row_token), _ptr(slot_row), _ptr(u_perm), _stream(stream)))


def moe_update_select_bias(shape, expert_offsets, select_bias, gamma: float, loads=None,
                           stream=None):
    """One step of the aux-loss-free bias controller, in place on select_bias."""
    _check("moe_update_select_bias", lib().moe_update_select_bias(
        ctypes.byref(shape_struct(shape)), _ptr(expert_offsets), _ptr(select_bias),
        ctypes.c_float(gamma), _ptr(loads), _stream(stream)))


def moe_balance_stats(shape, logits, expert_offsets, f, p, ws, stream=None):
    """f_i and P_i of the expert-level balance loss into f, p [E] fp32."""
    _check("moe_balance_stats", lib().moe_balance_stats(
        ctypes.byref(shape_struct(shape)), _ptr(logits), _ptr(expert_offsets), _ptr(f), _ptr(p),
        _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_expert_ffn(shape, weights: moe_weights, u, u_perm, expert_offsets, y_perm, y_shared,
                   ws, stream=None):
    _check("moe_expert_ffn", lib().moe_expert_ffn(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), _ptr(u), _ptr(u_perm),
        _ptr(expert_offsets), _ptr(y_perm), _ptr(y_shared), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine(shape, u, y_perm, y_shared, topk_w, slot_row, h, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(shape_struct(shape)), _ptr(u), _ptr(y_perm), _ptr(y_shared),
        _ptr(topk_w), _ptr(slot_row), _ptr(h), _stream(stream)))


def moe_layer_forward(shape, weights: moe_weights, u, h, ws, route_out=None, stream=None):
    """route_out: optional dict with any of logits, topk_idx, topk_w, expert_offsets."""
    ro = None
    if route_out:
        ro = moe_route_outputs(*[_ptr(route_out.get(n)) for n in
                                 ("logits", "topk_idx", "topk_w", "expert_offsets")])
    _check("moe_layer_forward", lib().moe_layer_forward(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), _ptr(u), _ptr(h),
        ctypes.byref(ro) if ro is not None else None, _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_forward_host(shape, weights: moe_weights, u_host, h_host, u_dev, h_dev, ws,
                           stream=None):
    _check("moe_layer_forward_host", lib().moe_layer_forward_host(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), _ptr(u_host), _ptr(h_host),
        _ptr(u_dev), _ptr(h_dev), _ptr(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_forward_host_stream(shape, weights: moe_weights, u_hosts, h_hosts, u_dev, h_dev,
                                  ws, stream=None):
    """The layer on each of the host batches u_hosts[b] -> h_hosts[b] (each
    [T, H], pinned), copies pipelined across batches; u_dev and h_dev hold
    2·T·H elements each."""
    if len(u_hosts) != len(h_hosts):
        raise ValueError("one output buffer per input batch")
    n = len(u_hosts)
    ins = (_P * max(n, 1))(*[_ptr(t) for t in u_hosts])
    outs = (_P * max(n, 1))(*[_ptr(t) for t in h_hosts])
    _check("moe_layer_forward_host_stream", lib().moe_layer_forward_host_stream(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), n, ins, outs, _ptr(u_dev),
        _ptr(h_dev), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_layer_backward_workspace_size(shape) -> int:
    return lib().moe_layer_backward_workspace_size(ctypes.byref(shape_struct(shape)))


def weight_grads(d_centroids, dw1, dw3, dw2, dsw1=None, dsw3=None, dsw2=None) -> moe_weight_grads:
    """The gradient outputs of moe_layer_backward (fp32 tensors, or None)."""
    return moe_weight_grads(*[_ptr(t) for t in (d_centroids, dw1, dw3, dw2, dsw1, dsw3, dsw2)])


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def moe_layer_backward(shape, weights: moe_weights, u, dh, du, grads: moe_weight_grads, ws,
                       saved=None, stream=None):
    """du and the weight gradients of the layer for the upstream gradient dh
    (saved: the buffer of moe_layer_forward_train, or None to recompute)."""
    _check("moe_layer_backward", lib().moe_layer_backward(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), _ptr(u), _ptr(dh), _ptr(du),
        ctypes.byref(grads), _ptr(saved), _nbytes(saved), _ptr(ws), _nbytes(ws),
        _stream(stream)))


def moe_check_bounded_wait(limit_us: int, stream=None):
    """Run the bounded-wait self-test (see include/moe.h); read the result with
    moe_device_status()."""
    _check("moe_check_bounded_wait", lib().moe_check_bounded_wait(limit_us, _stream(stream)))


def moe_layer_saved_size(shape) -> int:
    return lib().moe_layer_saved_size(ctypes.byref(shape_struct(shape)))


def moe_layer_forward_train(shape, weights: moe_weights, u, h, saved, ws, stream=None):
    """moe_layer_forward that also fills `saved` for moe_layer_backward."""
    _check("moe_layer_forward_train", lib().moe_layer_forward_train(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), _ptr(u), _ptr(h), _ptr(saved),
        _nbytes(saved), _ptr(ws), _nbytes(ws), _stream(stream)))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A byte buffer for the ``ws`` argument (at least 256 bytes)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def moe_expert_ffn_rows_workspace_size(shape, max_rows: int) -> int:
    return lib().moe_expert_ffn_rows_workspace_size(ctypes.byref(shape_struct(shape)),
                                                     int(max_rows))


def moe_expert_ffn_rows(shape, weights: moe_weights, n_rows: int, u, x_rows, expert_offsets,
                        y_rows, y_shared, ws, stream=None):
    """Expert FFNs on explicitly given rows (an expert-parallel rank's received
    rows): see include/moe.h."""
    _check("moe_expert_ffn_rows", lib().moe_expert_ffn_rows(
        ctypes.byref(shape_struct(shape)), ctypes.byref(weights), int(n_rows), _ptr(u),
        _ptr(x_rows), _ptr(expert_offsets), _ptr(y_rows), _ptr(y_shared), _ptr(ws), _nbytes(ws),
        _stream(stream)))


def moe_ep_regroup(shape, n_ranks: int, counts, n_rows: int, src, dst, expert_offsets=None,
                   to_expert_major: bool = True, stream=None):
    """Source-major <-> expert-major order of the rows a rank received."""
    _check("moe_ep_regroup", lib().moe_ep_regroup(
        ctypes.byref(shape_struct(shape)), int(n_ranks), _ptr(counts), int(n_rows), _ptr(src),
        _ptr(dst), _ptr(expert_offsets), 1 if to_expert_major else 0, _stream(stream)))
