"""Host logic of bench.py (no GPU): the algorithmic work it divides by, the
roof it reports against, its launch counts and the traffic record's guard."""
import numpy as np
import pytest

import bench
from fine_grained_shared_gemm_b300 import workloads as W

PEAKS = {"hbm_gbs": 6490.8, "bf16_tflops": 1755.6}


def _even_offsets(s):
    return np.concatenate([[0], np.cumsum(np.full(s.n_routed, s.T * s.top_k // s.n_routed))])


def test_algorithmic_work_by_hand():
    s = W.MoEShape("hand", T=10, H=128, n_routed=4, n_shared=1, top_k=2, inter=64)
    # FLOPs: 10 tokens x (2 routed + 1 shared) rows x 3 matrices x 2 H I
    assert bench.expert_flops(s) == 10 * 3 * 3 * 2 * 128 * 64
    off = np.array([0, 5, 5, 12, 20])          # expert 1 has no token
    # bytes: 3 touched routed + 1 shared experts' weights, rows in/out, act out/in
    rows = 10 * 3
    want = (4 * 3 * 128 * 64 + rows * 128 * 2 + rows * 64 * 2) * 2
    assert bench.ffn_alg_bytes(s, off) == want


@pytest.mark.parametrize("name,bound", [("dsmoe16b_bf16", "tensor"),
                                        ("v3_prefill_bf16", "hbm"),
                                        ("sweep_m1", "tensor"),
                                        ("decode_bf16", "hbm")])
def test_binding_roof(name, bound):
    s = W.SHAPES[name]
    r = bench.ffn_roofline(s, _even_offsets(s), 1e-3, PEAKS)
    assert r["bound"] == bound
    assert 0 < r["frac"] and r["achieved"] > 0
    if name != "decode_bf16":
        other = r["other_roof"]
        assert other["bound"] != bound
        # the binding roof is the one whose lower bound on the time is larger
        t = {"tensor": bench.expert_flops(s) / (PEAKS["bf16_tflops"] * 1e12),
             "hbm": bench.ffn_alg_bytes(s, _even_offsets(s)) / (PEAKS["hbm_gbs"] * 1e9)}
        assert t[bound] >= t[other["bound"]]


def test_backward_launch_counts():
    s = W.SHAPES["dsmoe16b_bf16"]          # SwiGLU, 2 shared, top-6
    # recompute: logits, route, 4 dispatch, 2 pre-activation GEMMs, then the
    # common 19: gather dh, row gate, 2 plans, dm, 3 derivative launches (2
    # shared + routed), gate, 2 router GEMMs + u transpose, dx, du, 3 operand
    # transposes, 2 weight-gradient GEMMs
    assert bench.backward_launches(s, saved=True) == 19
    assert bench.backward_launches(s) == 19 + 6 + 2
    relu = W.MoEShape("r", T=64, H=128, n_routed=8, n_shared=0, top_k=0, inter=128,
                      act=W.ACT_RELU)
    # no expert rows at all: no gathers, dm, derivative, dx or routed
    # transposes; dispatch is one scan when recomputing
    assert bench.backward_launches(relu, saved=True) == 2 + 4 + 1 + 1 + 2
    assert bench.backward_launches(relu) == 2 + 4 + 1 + 1 + 2 + 3
    assert bench.forward_launches(s) == 10 and bench.forward_launches(relu) == 7


def test_traffic_record_needs_the_current_kernel_source():
    assert bench.recorded_traffic("no_such_workload") is None
    rec = bench.recorded_traffic("dsmoe16b_bf16")
    lines = [l.split() for l in open(bench.os.path.join(bench.ROOT, "profiles",
                                                        "expert_ffn_dram_traffic.txt"))
             if l.startswith("dsmoe16b_bf16")]
    if lines[0][1] == bench.kernel_source_hash():
        assert rec == float(lines[0][2])
    else:
        assert rec is None
