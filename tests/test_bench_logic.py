"""Host logic of bench.py (no GPU): the algorithmic work it divides by, the
roof it reports against, its launch counts and the traffic record's guard."""
import numpy as np
import pytest

import bench
from fine_grained_shared_gemm_b300 import workloads as W

PEAKS = {"hbm_gbs": 6490.8, "bf16_tflops": 1755.6, "bf16_tflops_sustained": 1384.1}


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


@pytest.mark.parametrize("name", ["dsmoe16b_bf16", "v3_prefill_bf16", "sweep_m1"])
def test_prefill_roofline_is_the_tensor_peak(name):
    s = W.SHAPES[name]
    off = _even_offsets(s)
    r = bench.prefill_roofline(s, off, 1e-3, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(bench.expert_flops(s) / 1e-3 / 1e12, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops"], rel=1e-3)
    assert r["frac_of_nominal"] == pytest.approx(r["achieved"] / 2250.0, rel=1e-3)
    other = r["other_roof"]
    assert other["bound"] == "hbm"
    assert other["algorithmic_bytes"] == bench.ffn_alg_bytes(s, off)
    # the V3-shaped layer sits just on the memory side of the ridge
    t_f = bench.expert_flops(s) / (PEAKS["bf16_tflops"] * 1e12)
    t_b = bench.ffn_alg_bytes(s, off) / (PEAKS["hbm_gbs"] * 1e9)
    assert r["ridge"] == ("memory side" if t_b > t_f else "tensor side")
    # the fraction of the power-capped rate sits beside the burst one
    if PEAKS.get("bf16_tflops_sustained"):
        assert r["frac_of_sustained"] == pytest.approx(
            r["achieved"] / PEAKS["bf16_tflops_sustained"], rel=1e-3)
        assert r["frac_of_sustained"] > r["frac"]
    assert bench.sustained_frac(1.3841e12, 1.0, {"bf16_tflops_sustained": 1384.1}) == \
        pytest.approx(1.0, rel=1e-4)
    assert bench.sustained_frac(1e12, 1.0, {}) is None


def test_decode_roofline_counts_bytes_over_the_layer_time():
    s = W.SHAPES["decode_bf16"]
    assert bench.is_decode(s) and not bench.is_decode(W.SHAPES["v3_prefill_bf16"])
    off = np.zeros(s.n_routed + 1, dtype=np.int64)
    off[1:] = np.cumsum(np.r_[np.full(100, 5), np.zeros(s.n_routed - 100, dtype=np.int64)])
    # 100 routed experts with a token + 1 shared, 3 matrices of H x I bf16
    w = 101 * 3 * s.H * s.inter * 2
    assert bench.touched_weight_bytes(s, off) == w
    b = w + s.n_routed * s.H * 2 + 2 * s.T * s.H * 2
    assert bench.decode_alg_bytes(s, off) == b
    r = bench.decode_roofline(s, off, 2e-3, 1.8e-3, PEAKS)
    assert r["bound"] == "hbm" and r["experts_touched"] == 101
    assert r["achieved"] == pytest.approx(b / 2e-3 / 1e9, rel=1e-3)
    assert r["ffn_only"]["achieved"] == pytest.approx(w / 1.8e-3 / 1e9, rel=1e-3)
    assert r["frac_of_nominal"] == pytest.approx(r["achieved"] / 8000.0, rel=1e-3)
    assert "note" not in r
    fast = bench.decode_roofline(s, off, 1e-4, 1e-4, PEAKS)   # above the copy rate
    assert fast["frac"] > 1 and "note" in fast


def test_backward_launch_counts():
    s = W.SHAPES["dsmoe16b_bf16"]          # SwiGLU, 2 shared, top-6
    # recompute: logits, route, 4 dispatch, 2 pre-activation GEMMs, then the
    # common 13: scatter dh rows, row gate, 2 plans, dm with the SwiGLU
    # derivative, gate, 2 router GEMMs, the router gradient's partial sums,
    # dx, du, 2 weight-gradient GEMMs
    assert bench.backward_launches(s, saved=True) == 13
    assert bench.backward_launches(s) == 13 + 6 + 2
    relu = W.MoEShape("r", T=64, H=128, n_routed=8, n_shared=0, top_k=0, inter=128,
                      act=W.ACT_RELU)
    # no expert rows at all: no row scatter, dm, derivative or dx; dispatch
    # is one scan when recomputing
    assert bench.backward_launches(relu, saved=True) == 2 + 4 + 1 + 2
    assert bench.backward_launches(relu) == 2 + 4 + 1 + 2 + 3
    # ReLU with rows: the derivative is its own launch per shared expert and
    # one for the routed rows
    relu_rows = W.MoEShape("rr", T=64, H=128, n_routed=8, n_shared=1, top_k=2, inter=128,
                           act=W.ACT_RELU)
    assert bench.backward_launches(relu_rows, saved=True) == 2 + 2 + 1 + 2 + 4 + 2 + 2
    assert bench.forward_launches(s) == 10 and bench.forward_launches(relu) == 7


def test_router_split_rule():
    # decode: 3 tiles of 128 experts x 64 tokens over 112 k-blocks -> 28
    # ranges of 4 k-blocks, and one more launch (the partial sums)
    dec = W.SHAPES["decode_bf16"]
    assert bench.router_splits(dec) == 28
    assert bench.forward_launches(dec) == 11
    # prefill batches have enough tiles to stay whole
    for name in ("v3_prefill_bf16", "dsmoe16b_bf16"):
        assert bench.router_splits(W.SHAPES[name]) == 1
        assert bench.forward_launches(W.SHAPES[name]) == 10
    # H = 128: one stage of two k-blocks, nothing to cut; fp32 runs unsplit
    tiny = W.MoEShape("t", T=8, H=128, n_routed=8, n_shared=0, top_k=2, inter=64)
    assert bench.router_splits(tiny) == 1
    f32 = W.MoEShape("f", T=8, H=1024, n_routed=8, n_shared=0, top_k=2, inter=64, dtype="f32")
    assert bench.router_splits(f32) == 1
    # the library's own rule: its workspace holds exactly the ranges' partials
    from fine_grained_shared_gemm_b300 import moe as M
    for s in (dec, W.SHAPES["decode_e48_bf16"], W.SHAPES["v3_prefill_bf16"], tiny, f32):
        n = bench.router_splits(s)
        assert M.moe_router_logits_workspace_size(s) == (n * s.T * s.n_routed * 4 if n > 1 else 0)
    # at most 32 ranges of at least one two-k-block stage each
    for H in (256, 384, 1024, 2048, 7168):
        s = W.MoEShape("h", T=16, H=H, n_routed=64, n_shared=0, top_k=2, inter=64)
        n = bench.router_splits(s)
        assert 2 <= n <= min(32, H // 128)


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
