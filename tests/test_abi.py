"""The C-ABI library loads without a GPU, exports every entry point declared
in include/moe.h, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from fine_grained_shared_gemm_b300 import moe as M
from fine_grained_shared_gemm_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    for n in ("moe_router_logits", "moe_route", "moe_dispatch", "moe_expert_ffn",
              "moe_combine", "moe_layer_forward", "moe_layer_forward_host",
              "moe_layer_workspace_size", "moe_device_status", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = M.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in M._SIGNATURES, f"binding has no signature for {name}"


def test_only_declared_symbols_are_exported():
    out = os.popen(f"nm -D --defined-only {M.library_path()}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    moe_syms = {s for s in exported if s.startswith("moe_")}
    assert moe_syms == set(declared_symbols())


def test_status_strings():
    lib = M.lib()
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(M.MOE_ERR_WORKSPACE).startswith(b"workspace")
    assert lib.moe_status_string(99) == b"unknown status"


def _shape(**kw):
    base = dict(T=100, H=256, n_routed=16, n_shared=1, top_k=4, inter=128,
                gate=0, act=1, dtype=1)
    base.update(kw)
    return M.moe_shape(**base)


def test_workspace_sizes_cover_the_buffers():
    for name in ("tiny_f32", "dsmoe16b_bf16", "v3_prefill_bf16", "decode_bf16", "sweep_m16"):
        s = W.SHAPES[name]
        st = M.shape_struct(s)
        e = 4 if s.dtype == "f32" else 2
        lay = M.lib().moe_layer_workspace_size(ctypes.byref(st))
        # permuted rows in and out plus shared outputs and the intermediate activation
        need = (2 * s.T * s.top_k * s.H + s.n_shared * s.T * s.H
                + s.T * (s.top_k + s.n_shared) * s.inter) * e
        assert lay >= need
        assert M.lib().moe_expert_ffn_workspace_size(ctypes.byref(st)) >= \
            s.T * (s.top_k + s.n_shared) * s.inter * e


@pytest.mark.parametrize("bad,code", [
    (dict(top_k=17), M.MOE_ERR_INVALID_ARG),        # k > E
    (dict(T=-1), M.MOE_ERR_INVALID_ARG),
    (dict(H=0), M.MOE_ERR_INVALID_ARG),
    (dict(gate=7), M.MOE_ERR_INVALID_ARG),
    (dict(dtype=3), M.MOE_ERR_INVALID_ARG),
    (dict(n_routed=1100), M.MOE_ERR_UNSUPPORTED),  # E + Ks > 1024
    (dict(n_routed=64, top_k=33), M.MOE_ERR_UNSUPPORTED),
    (dict(H=200), M.MOE_ERR_UNSUPPORTED),            # bf16 needs H % 128
    (dict(inter=96), M.MOE_ERR_UNSUPPORTED),         # bf16 SwiGLU needs inter % 64
    # group-limited routing
    (dict(n_groups=3, topk_groups=1), M.MOE_ERR_INVALID_ARG),   # 16 % 3 != 0
    (dict(n_groups=4, topk_groups=0), M.MOE_ERR_INVALID_ARG),
    (dict(n_groups=4, topk_groups=5), M.MOE_ERR_INVALID_ARG),
    (dict(n_groups=8, topk_groups=1), M.MOE_ERR_INVALID_ARG),   # 1 group of 2 < top_k 4
    (dict(n_groups=0, topk_groups=2), M.MOE_ERR_INVALID_ARG),
    (dict(n_groups=-1, topk_groups=1), M.MOE_ERR_INVALID_ARG),
    (dict(n_routed=64, n_groups=64, topk_groups=8), M.MOE_ERR_UNSUPPORTED),  # > 32 groups
])
def test_bad_shapes_rejected_on_host(bad, code):
    s = _shape(**bad)
    assert M.lib().moe_layer_workspace_size(ctypes.byref(s)) == 0
    st = M.lib().moe_route(ctypes.byref(s), 256, None, 256, 256, None, None)
    assert st == code


def test_group_limited_shape_accepted():
    s = _shape(n_groups=4, topk_groups=2)
    assert M.lib().moe_layer_workspace_size(ctypes.byref(s)) > 0


def test_null_and_misaligned_pointers_rejected():
    s = _shape()
    L = M.lib()
    assert L.moe_route(ctypes.byref(s), None, None, 256, 256, None, None) == M.MOE_ERR_INVALID_ARG
    assert L.moe_route(ctypes.byref(s), 258, None, 256, 256, None, None) == M.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(s), 256, 256, None, 256, 256, 256, None) == \
        M.MOE_ERR_INVALID_ARG   # n_shared = 1 needs y_shared
    w = M.moe_weights(256, None, None, 256, None, 256, 256, 256, 256)  # SwiGLU without w3
    assert L.moe_expert_ffn(ctypes.byref(s), ctypes.byref(w), 256, 256, 256, 256, 256,
                            256, 1 << 30, None) == M.MOE_ERR_INVALID_ARG


def test_workspace_too_small_rejected():
    s = _shape()
    L = M.lib()
    w = M.moe_weights(256, None, None, 256, 256, 256, 256, 256, 256)
    need = L.moe_layer_workspace_size(ctypes.byref(s))
    assert L.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), 256, 256, None, 256,
                               need - 1, None) == M.MOE_ERR_WORKSPACE
    assert L.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), 256, 256, None, None,
                               need, None) == M.MOE_ERR_WORKSPACE
    need_d = L.moe_dispatch_workspace_size(ctypes.byref(s))
    assert L.moe_dispatch(ctypes.byref(s), 256, 256, 256, 256, 256, 256, 256, need_d - 1,
                          None) == M.MOE_ERR_WORKSPACE


def test_bias_update_rejects_bad_gamma_and_pointers():
    s = _shape()
    L = M.lib()
    f = ctypes.c_float
    for g in (-0.1, float("nan"), float("inf")):
        assert L.moe_update_select_bias(ctypes.byref(s), 256, 256, f(g), None, None) == \
            M.MOE_ERR_INVALID_ARG, g
    assert L.moe_update_select_bias(ctypes.byref(s), None, 256, f(0.1), None, None) == \
        M.MOE_ERR_INVALID_ARG
    assert L.moe_update_select_bias(ctypes.byref(s), 256, 258, f(0.1), None, None) == \
        M.MOE_ERR_INVALID_ARG


def test_balance_stats_rejects_bad_pointers_and_workspace():
    s = _shape()
    L = M.lib()
    need = L.moe_balance_stats_workspace_size(ctypes.byref(s))
    assert need >= s.n_routed * 4 * ((s.T + 255) // 256) and need % 256 == 0
    args = [256, 256, 256, 256, 256, need, None]
    for i in range(4):   # logits, offsets, f, p
        bad = list(args)
        bad[i] = None
        assert L.moe_balance_stats(ctypes.byref(s), *bad) == M.MOE_ERR_INVALID_ARG, i
        bad[i] = 258
        assert L.moe_balance_stats(ctypes.byref(s), *bad) == M.MOE_ERR_INVALID_ARG, i
    assert L.moe_balance_stats(ctypes.byref(s), 256, 256, 256, 256, 256, need - 1, None) == \
        M.MOE_ERR_WORKSPACE
    assert L.moe_balance_stats(ctypes.byref(s), 256, 256, 256, 256, None, need, None) == \
        M.MOE_ERR_WORKSPACE


def test_training_entry_points_reject_bad_arguments():
    s = _shape()
    L = M.lib()
    need = L.moe_layer_saved_size(ctypes.byref(s))
    assert need > 0 and need % 256 == 0
    assert L.moe_layer_saved_size(ctypes.byref(_shape(dtype=0))) == 0   # fp32: not supported
    w = M.moe_weights(256, None, None, 256, 256, 256, 256, 256, 256)
    ws = L.moe_layer_workspace_size(ctypes.byref(s))
    assert L.moe_layer_forward_train(ctypes.byref(s), ctypes.byref(w), 256, 256, None, need,
                                     256, ws, None) == M.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward_train(ctypes.byref(s), ctypes.byref(w), 256, 256, 256, need - 1,
                                     256, ws, None) == M.MOE_ERR_INVALID_ARG
    g = M.moe_weight_grads(256, 256, 256, 256, 256, 256, 256)
    bws = L.moe_layer_backward_workspace_size(ctypes.byref(s))
    assert L.moe_layer_backward(ctypes.byref(s), ctypes.byref(w), 256, 256, 256, ctypes.byref(g),
                                258, need, 256, bws, None) == M.MOE_ERR_INVALID_ARG
    assert L.moe_layer_backward(ctypes.byref(s), ctypes.byref(w), 256, 256, 256, ctypes.byref(g),
                                256, need - 1, 256, bws, None) == M.MOE_ERR_INVALID_ARG
    assert L.moe_layer_backward(ctypes.byref(s), ctypes.byref(w), 256, 256, 256, ctypes.byref(g),
                                None, 0, 256, bws - 1, None) == M.MOE_ERR_WORKSPACE


def test_bounded_wait_self_test_rejects_bad_limits():
    L = M.lib()
    assert L.moe_check_bounded_wait(0, None) == M.MOE_ERR_INVALID_ARG
    assert L.moe_check_bounded_wait(1000001, None) == M.MOE_ERR_INVALID_ARG


def test_host_stream_rejects_bad_arguments_on_host():
    """moe_layer_forward_host_stream checks its batch count, its host pointer
    arrays, the device slots and the workspace before any copy or launch."""
    s = _shape()
    L = M.lib()
    w = M.moe_weights(256, None, None, 256, 256, 256, 256, 256, 256)
    need = L.moe_layer_workspace_size(ctypes.byref(s))
    P = ctypes.c_void_p
    two = (P * 2)(4096, 8192)
    one_null = (P * 2)(4096, None)
    f = L.moe_layer_forward_host_stream
    assert f(ctypes.byref(s), ctypes.byref(w), -1, two, two, 256, 256, 256, need, None) == \
        M.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(s), ctypes.byref(w), 2, None, two, 256, 256, 256, need, None) == \
        M.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(s), ctypes.byref(w), 2, two, one_null, 256, 256, 256, need, None) == \
        M.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(s), ctypes.byref(w), 2, two, two, 258, 256, 256, need, None) == \
        M.MOE_ERR_INVALID_ARG     # device slots must be 16-byte aligned
    assert f(ctypes.byref(s), ctypes.byref(w), 2, two, two, 256, 256, 256, need - 1, None) == \
        M.MOE_ERR_WORKSPACE
    # nothing to do: no copy, no launch
    assert f(ctypes.byref(s), ctypes.byref(w), 0, None, None, None, None, 256, need, None) == \
        M.MOE_OK
