"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each check is written so that a plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, renormalised softmax gates, the
wrong tie rule) fails at least one of them; ``test_planted_mistakes`` plants
such slips in a copy of the oracle and checks that they are caught.
"""
import itertools
import json
import math
import os
import types

import numpy as np
import pytest

import oracle.moe_oracle as O
from fine_grained_shared_gemm_b300 import workloads as W


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _f32(xs):
    return np.array([float(x) for x in xs], dtype=np.float32)


# ---------------------------------------------------------------- checks
# Each check takes the oracle module so that a mutated copy can be run.

def check_combinations(o, golden_dir):
    for c in _load(golden_dir, "combinations.json")["cases"]:
        assert o.routing_combinations(c["n_routed"], c["top_k"]) == c["value"], c


def check_routing_handworked(o, golden_dir):
    for c in _load(golden_dir, "routing_handworked.json")["cases"]:
        z = _f32(c["logits"])[None, :]
        b = None if c["bias"] is None else _f32(c["bias"])
        r = o.route(z, c["gate"], c["top_k"], b)
        assert r["idx"][0].tolist() == c["idx"], c["name"]
        np.testing.assert_allclose(r["weights"][0], c["weights"], atol=2e-6,
                                   err_msg=c["name"])


def check_ffn_handworked(o, golden_dir):
    g = _load(golden_dir, "ffn_handworked.json")
    for c in g["ffn"]:
        w3 = None if c["w3"] is None else np.array(c["w3"], float)
        y = o.expert_ffn(np.array([c["u"]], float), np.array(c["w1"], float),
                         np.array(c["w2"], float), w3, c["act"])
        np.testing.assert_allclose(y[0], c["y"], atol=2e-6, err_msg=c["name"])
    for c in g["layer"]:
        u = np.array([c["u"]], float)
        z = o.router_logits(u, np.array(c["centroids"], float))
        r = o.route(z, c["gate"], c["top_k"])
        mk = lambda d: (np.array(d["w1"], float), None, np.array(d["w2"], float))
        h = o.layer_forward(u, r, lambda e: mk(c["routed"][e]),
                            lambda j: mk(c["shared"][j]), len(c["shared"]),
                            c["act"])
        np.testing.assert_allclose(h[0], c["h"], atol=2e-6, err_msg=c["name"])


def _brute_topk(key_row, k):
    """Exhaustive: the unique k-subset whose every member beats every
    non-member under the order (larger key first, lower index on ties)."""
    E = len(key_row)
    beats = lambda i, j: key_row[i] > key_row[j] or (key_row[i] == key_row[j] and i < j)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all(beats(i, j) for i in S for j in rest):
            found.append(S)
    assert len(found) == 1
    S = list(found[0])
    # order inside the set: by the same total order (insertion sort by beats)
    out = []
    for i in S:
        pos = 0
        while pos < len(out) and beats(out[pos], i):
            pos += 1
        out.insert(pos, i)
    return out


def check_topk_bruteforce(o):
    rng = np.random.default_rng(1)
    for trial in range(150):
        E = int(rng.integers(1, 9))
        k = int(rng.integers(0, E + 1))
        if trial % 2:
            key = rng.integers(-1, 2, size=(3, E)).astype(np.float32)  # many ties
        else:
            key = rng.standard_normal((3, E)).astype(np.float32)
        got = o.topk_by_rank(key, k)
        for t in range(3):
            assert got[t].tolist() == _brute_topk(key[t].tolist(), k), (key[t], k)


def check_softmax_properties(o):
    rng = np.random.default_rng(2)
    z = rng.standard_normal((7, 5)).astype(np.float32) * 3
    s = o.softmax_scores(z)
    np.testing.assert_allclose(s.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    # two experts: closed form 1 / (1 + e^(b - a))
    a, b = 0.75, -1.25
    s2 = o.softmax_scores(np.array([[a, b]], np.float32))
    assert abs(s2[0, 0] - 1.0 / (1.0 + math.exp(b - a))) < 1e-15
    # chosen gates are a subset of a distribution: sum <= 1, strictly < 1 if k < E
    r = o.route(z, O.SOFTMAX, 3)
    assert np.all(r["weights"].sum(axis=1) < 1.0)
    np.testing.assert_allclose(r["weights"], np.take_along_axis(s, r["idx"], 1),
                               rtol=0, atol=0)


def check_softmax_choice_is_score_order(o):
    """The choice taken on the logits equals the top-k of the float64 scores."""
    rng = np.random.default_rng(3)
    z = rng.standard_normal((200, 40)).astype(np.float32)
    r = o.route(z, O.SOFTMAX, 6)
    s = o.softmax_scores(z)
    by_score = np.argsort(-s, axis=1, kind="stable")[:, :6]
    assert np.array_equal(r["idx"], by_score)


def check_sigmoid_properties(o):
    rng = np.random.default_rng(4)
    z = rng.standard_normal((300, 24)).astype(np.float32)
    # Eq. 15: weights sum to one
    b = rng.uniform(-0.1, 0.1, 24).astype(np.float32)
    r = o.route(z, O.SIGMOID_BIAS, 8, b)
    np.testing.assert_allclose(r["weights"].sum(axis=1), 1.0, atol=1e-14)
    # sigmoid closed form at 0 and its symmetry
    s = o.sigmoid_scores(np.array([[0.0, 2.0, -2.0]], np.float32))
    assert s[0, 0] == 0.5 and abs(s[0, 1] + s[0, 2] - 1.0) < 1e-15
    # no bias: choice equals the top-k of the logits (sigmoid is increasing)
    r0 = o.route(z, O.SIGMOID_BIAS, 8, None)
    ok = r0["gap"] > 1e-5
    assert np.array_equal(r0["idx"][ok], np.argsort(-z, 1, kind="stable")[ok, :8])
    # weights depend on the chosen set only, not on the bias values
    sc = o.sigmoid_scores(z)
    g = np.take_along_axis(sc, r["idx"], 1)
    np.testing.assert_allclose(r["weights"], g / g.sum(1, keepdims=True), atol=1e-15)
    # the bias moves the choice: a huge bias on expert 5 makes every token pick it
    bb = np.zeros(24, np.float32)
    bb[5] = 10.0
    rb = o.route(z, O.SIGMOID_BIAS, 8, bb)
    assert np.all(rb["idx"][:, 0] == 5)
    assert np.all(rb["weights"][:, 0] < 0.5)   # its weight still uses the raw score


def check_segmentation_identity(o):
    """One dense FFN of width M split along the intermediate dimension into m
    experts of width M/m, all chosen with weight 1, equals the dense FFN."""
    rng = np.random.default_rng(5)
    H, M, m = 6, 12, 4
    x = rng.standard_normal((5, H))
    for act in (O.RELU, O.SWIGLU):
        w1 = rng.standard_normal((M, H))
        w3 = rng.standard_normal((M, H)) if act == O.SWIGLU else None
        w2 = rng.standard_normal((H, M))
        dense = o.expert_ffn(x, w1, w2, w3, act)
        I = M // m
        parts = sum(o.expert_ffn(x, w1[p * I:(p + 1) * I], w2[:, p * I:(p + 1) * I],
                                 None if w3 is None else w3[p * I:(p + 1) * I], act)
                    for p in range(m))
        np.testing.assert_allclose(parts, dense, rtol=1e-12, atol=1e-12)


def _loop_ffn(u, w1, w2, w3, act):
    """Element loops over the FFN definition: y_h = Σ_j W2[h][j] · φ_j,
    φ_j = act(Σ_d W1[j][d] u_d) (times Σ_d W3[j][d] u_d for SwiGLU)."""
    I, H = len(w1), len(u)
    y = []
    for h in range(len(w2)):
        acc = 0.0
        for j in range(I):
            a = sum(w1[j][d] * u[d] for d in range(H))
            if act == O.RELU:
                phi = a if a > 0 else 0.0
            else:
                c = sum(w3[j][d] * u[d] for d in range(H))
                phi = a / (1.0 + math.exp(-a)) * c
            acc += w2[h][j] * phi
        y.append(acc)
    return y


def check_ffn_bruteforce(o):
    rng = np.random.default_rng(6)
    H, I = 5, 3
    for act in (O.RELU, O.SWIGLU):
        u = rng.standard_normal(H)
        w1, w3, w2 = rng.standard_normal((I, H)), rng.standard_normal((I, H)), rng.standard_normal((H, I))
        got = o.expert_ffn(u[None], w1, w2, w3 if act == O.SWIGLU else None, act)[0]
        want = _loop_ffn(u.tolist(), w1.tolist(), w2.tolist(), w3.tolist(), act)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def _gshard_topk_moe(u, cents, experts, K):
    """Classic top-K MoE (m = 1, no shared experts) written with Python loops:
    logits by dot products, softmax by math.exp, choice by sorting."""
    T, E = len(u), len(cents)
    h = []
    for t in range(T):
        z = [float(np.float32(sum(u[t][d] * cents[i][d] for d in range(len(u[t])))))
             for i in range(E)]
        mx = max(z)
        ex = [math.exp(v - mx) for v in z]
        tot = sum(ex)
        order = sorted(range(E), key=lambda i: (-z[i], i))[:K]
        out = list(u[t])
        for i in order:
            w1, w2 = experts[i]
            y = _loop_ffn(u[t], w1, w2, None, O.RELU)
            out = [a + ex[i] / tot * b for a, b in zip(out, y)]
        h.append(out)
    return h


def check_classic_moe(o):
    rng = np.random.default_rng(7)
    T, H, E, I, K = 6, 4, 5, 3, 2
    u = rng.standard_normal((T, H))
    cents = rng.standard_normal((E, H))
    ex = [(rng.standard_normal((I, H)), rng.standard_normal((H, I))) for _ in range(E)]
    z = o.router_logits(u, cents)
    r = o.route(z, O.SOFTMAX, K)
    h = o.layer_forward(u, r, lambda e: (ex[e][0], None, ex[e][1]),
                        lambda j: None, 0, O.RELU)
    want = _gshard_topk_moe(u.tolist(), cents.tolist(),
                            [(a.tolist(), b.tolist()) for a, b in ex], K)
    np.testing.assert_allclose(h, want, rtol=1e-10, atol=1e-10)


def check_shared_equals_forced_routed(o):
    """A shared expert behaves like a routed expert that every token chooses
    with weight 1: one routed expert under softmax always has s = 1."""
    rng = np.random.default_rng(8)
    T, H, I = 9, 5, 4
    u = rng.standard_normal((T, H))
    w = (rng.standard_normal((I, H)), rng.standard_normal((I, H)), rng.standard_normal((H, I)))
    as_shared = o.layer_forward(u, o.route(np.zeros((T, 1), np.float32), O.SOFTMAX, 0),
                                lambda e: None, lambda j: w, 1, O.SWIGLU)
    z = o.router_logits(u, rng.standard_normal((1, H)))
    as_routed = o.layer_forward(u, o.route(z, O.SOFTMAX, 1), lambda e: w,
                                lambda j: None, 0, O.SWIGLU)
    np.testing.assert_allclose(as_shared, as_routed, rtol=1e-13, atol=1e-13)
    # no shared and no routed work: h = u exactly
    none = o.layer_forward(u, o.route(np.zeros((T, 3), np.float32), O.SOFTMAX, 0),
                           lambda e: None, lambda j: None, 0, O.SWIGLU)
    assert np.array_equal(none, u)


def check_combine_zero_gates(o):
    rng = np.random.default_rng(9)
    u = rng.standard_normal((4, 3))
    y = rng.standard_normal((4, 2, 3))
    assert np.array_equal(o.combine(u, [], y, np.zeros((4, 2))), u)
    # ordering of terms: one shared and one routed slot, weights (0.5)
    ys = rng.standard_normal((4, 3))
    h = o.combine(u, [ys], y, np.array([[0.5, 0.0]] * 4))
    np.testing.assert_allclose(h, u + ys + 0.5 * y[:, 0], rtol=0, atol=1e-15)


def check_dispatch(o):
    rng = np.random.default_rng(10)
    T, E, k = 37, 7, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    d = o.dispatch(idx, E)
    assert d["counts"].sum() == T * k
    assert np.all(np.diff(d["offsets"]) >= 0) and d["offsets"][-1] == T * k
    assert sorted(d["slot_row"].reshape(-1).tolist()) == list(range(T * k))
    # brute force from the definition: expert-major, token order inside
    rows = [(t, s) for e in range(E) for t in range(T) for s in range(k) if idx[t, s] == e]
    assert [t for t, _ in rows] == d["row_token"].tolist()
    for r, (t, s) in enumerate(rows):
        assert d["slot_row"][t, s] == r
    for e in range(E):
        assert d["counts"][e] == sum(1 for t in range(T) if e in idx[t])


def check_bias_update_handworked(o, golden_dir):
    for c in _load(golden_dir, "bias_update_handworked.json")["cases"]:
        got = o.update_select_bias(np.array(c["loads"]), _f32(c["bias"]), c["gamma"],
                                   c["routed_rows"])
        assert got.dtype == np.float32
        assert np.array_equal(got, _f32(c["expected"])), (c, got)


def check_bias_controller_balances(o):
    """[CH7] §7.4: the bias controller exists to even out expert loads.  A
    router whose centroids have very different norms sends most tokens to a
    few experts; repeated steps of route -> loads -> bias update must bring
    the most loaded expert close to the mean and keep the loads summing to
    T·k (the bias never changes how many experts a token gets)."""
    rng = np.random.default_rng(3)
    T, H, E, k = 2048, 32, 16, 2
    u = rng.standard_normal((T, H))
    cents = rng.standard_normal((E, H)) * np.linspace(0.02, 0.4, E)[:, None]
    z = o.router_logits(u, cents)
    bias = np.zeros(E, np.float32)
    imbalance = []
    for _ in range(300):
        r = o.route(z, o.SIGMOID_BIAS, k, bias)
        loads = o.expert_loads(r["idx"], E)
        assert loads.sum() == T * k
        imbalance.append(loads.max() * E / (T * k))
        bias = o.update_select_bias(loads, bias, 0.002, T * k)
    assert imbalance[0] > 1.6, imbalance[0]          # the router starts skewed
    assert max(imbalance[-20:]) < 1.1, imbalance[-20:]


def check_group_routing_handworked(o, golden_dir):
    g = _load(golden_dir, "group_routing_handworked.json")
    keys = _f32(g["keys"])
    bias = (keys - np.float32(0.5)).astype(np.float32)   # sigmoid(0) = 0.5 exactly
    z = np.zeros((1, keys.shape[0]), np.float32)
    for c in g["cases"]:
        r = o.route(z, o.SIGMOID_BIAS, c["top_k"], bias, g["n_groups"], c["topk_groups"])
        assert r["idx"][0].tolist() == c["idx"], (c, r["idx"])
        assert np.allclose(r["weights"], 1.0 / c["top_k"])


def check_group_routing_bruteforce(o):
    """Chosen groups maximise the summed group score over all group subsets,
    chosen experts maximise the summed key over all subsets of their experts
    (random keys, no ties); keeping every group is plain top-k; one expert
    per group with as many groups as k chooses the plain top-k set."""
    rng = np.random.default_rng(7)
    E, G, M, k = 12, 4, 2, 3
    gs = E // G
    for gate in (o.SOFTMAX, o.SIGMOID_BIAS):
        z = rng.standard_normal((40, E)).astype(np.float32)
        bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
        r = o.route(z, gate, k, bias, G, M)
        gkey = (r["scores"].astype(np.float32) if gate == o.SOFTMAX else r["key"]).astype(np.float64)
        for t in range(z.shape[0]):
            gsum = gkey[t].reshape(G, gs).sum(axis=1)
            best_groups = max(itertools.combinations(range(G), M),
                              key=lambda c: sum(gsum[list(c)]))
            pool = [e for gg in best_groups for e in range(gg * gs, gg * gs + gs)]
            best = max(itertools.combinations(pool, k),
                       key=lambda c: sum(float(r["key"][t, e]) for e in c))
            assert sorted(r["idx"][t].tolist()) == sorted(best), (gate, t)
        plain = o.route(z, gate, k, bias)
        assert np.array_equal(o.route(z, gate, k, bias, G, G)["idx"], plain["idx"])
        if gate == o.SIGMOID_BIAS:
            one = o.route(z, gate, k, bias, E, k)
            assert np.array_equal(np.sort(one["idx"], 1), np.sort(plain["idx"], 1))


def _exact(v):
    """'ln3' -> log(3), '4/3' -> 4/3, '0' -> 0 (values of the hand-worked fixtures)."""
    if v.startswith("ln"):
        return math.log(float(v[2:]))
    num, _, den = v.partition("/")
    return float(num) / float(den or 1)


def check_balance_stats_handworked(o, golden_dir):
    for c in _load(golden_dir, "balance_stats_handworked.json")["cases"]:
        z = np.array([[_exact(v) for v in row] for row in c["logits"]], np.float32)
        idx = np.array(c["idx"])
        r = o.route(z, c["gate"], c["top_k"])
        assert np.array_equal(r["idx"], idx), (c, r["idx"])
        f, p = o.balance_stats(z, idx, z.shape[1], c["top_k"], c["gate"])
        assert f.dtype == np.float32
        assert np.array_equal(f, np.array([_exact(v) for v in c["f"]], np.float32)), (c, f)
        assert np.allclose(p, [_exact(v) for v in c["P"]], rtol=0, atol=1e-7), (c, p)


def check_balance_stats_properties(o):
    """Σ f_i = E and Σ P_i = 1 on random routings; an even routing gives
    f_i = 1; f depends on the choice only, P on the logits only; when every
    expert is chosen (k = E) P_i is the token mean of the gate weights the
    router gives expert i (no renormalisation under softmax, normalisation
    over all E under sigmoid)."""
    rng = np.random.default_rng(11)
    T, E, k = 96, 8, 3
    for gate in (o.SOFTMAX, o.SIGMOID_BIAS):
        z = (rng.standard_normal((T, E)) * 2).astype(np.float32)
        r = o.route(z, gate, k)
        f, p = o.balance_stats(z, r["idx"], E, k, gate)
        assert abs(float(f.astype(np.float64).sum()) - E) < 1e-5
        assert abs(p.sum() - 1.0) < 1e-12
        even = np.array([[(t + j) % E for j in range(k)] for t in range(T)])
        f_even, p2 = o.balance_stats(z, even, E, k, gate)
        assert np.array_equal(f_even, np.ones(E, np.float32))
        assert np.array_equal(p2, p)
        f3, _ = o.balance_stats(z[::-1] * 0.5, r["idx"], E, k, gate)
        assert np.array_equal(f3, f)
        full = o.route(z, gate, E)
        w = np.zeros((T, E))
        np.put_along_axis(w, full["idx"], full["weights"], axis=1)
        _, p_full = o.balance_stats(z, full["idx"], E, E, gate)
        assert np.allclose(p_full, w.mean(axis=0), rtol=1e-12, atol=1e-15)


CHECKS = [check_routing_handworked, check_ffn_handworked, check_combinations,
          check_bias_update_handworked, check_group_routing_handworked,
          check_balance_stats_handworked]
PLAIN_CHECKS = [check_topk_bruteforce, check_softmax_properties,
                check_softmax_choice_is_score_order, check_sigmoid_properties,
                check_segmentation_identity, check_ffn_bruteforce,
                check_classic_moe, check_shared_equals_forced_routed,
                check_combine_zero_gates, check_dispatch, check_bias_controller_balances,
                check_group_routing_bruteforce, check_balance_stats_properties]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_golden(check, golden_dir):
    check(O, golden_dir)


@pytest.mark.parametrize("check", PLAIN_CHECKS, ids=lambda c: c.__name__)
def test_property(check):
    check(O)


def test_iso_identities_every_shape():
    """[FG] §2.1: every segmented shape keeps total and active expert
    parameters equal to the base N dense FFNs with K active."""
    seen = 0
    for s in W.SHAPES.values():
        if s.seg is None:
            continue
        N, M, m, K = s.seg
        assert O.segmented_shape(N, M, m, K, s.n_shared) == (s.n_routed, s.inter, s.top_k)
        (p0, p1), (a0, a1) = O.iso_identities(N, M, m, K, s.n_shared, s.H)
        assert p0 == p1 and a0 == a1, s.name
        seen += 1
    assert seen == 11
    # the pages' worked example: 16 experts top-2 -> m = 4 gives 64 experts top-8
    assert O.segmented_shape(16, 4096, 4, 2) == (64, 1024, 8)


def test_layer_flops_iso_across_granularity():
    f = {m: O.layer_flops(16384, 2048, 4096 // m, 2 * m, 0, O.SWIGLU) for m in (1, 2, 4, 8, 16)}
    assert len(set(f.values())) == 1
    assert f[1] == 16384 * 2 * 3 * 2 * 2048 * 4096


# ---------------------------------------------------------------- mutations

def _mutant(**overrides):
    m = types.ModuleType("mutant")
    m.__dict__.update({k: v for k, v in O.__dict__.items() if not k.startswith("__")})
    m.__dict__.update(overrides)
    # functions look up globals in their own module; rebind them to the mutant
    for name, fn in list(m.__dict__.items()):
        if isinstance(fn, types.FunctionType) and name not in overrides:
            m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, name,
                                                  fn.__defaults__, fn.__closure__)
    return m


def _fails(check, o, *args):
    try:
        check(o, *args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_planted_mistakes(golden_dir):
    """Plant plausible slips in a copy of the oracle; some pin must fail."""
    def renormalised_softmax(z, gate, top_k, select_bias=None):
        r = O.route(z, gate, top_k, select_bias)
        r["weights"] = r["weights"] / r["weights"].sum(1, keepdims=True)
        return r

    def ties_to_higher(key, k):
        key = np.asarray(key)
        return key.shape[1] - 1 - O.topk_by_rank(key[:, ::-1], k)

    def no_residual(u, y_shared, y_routed, weights):
        return O.combine(u, y_shared, y_routed, weights) - u

    def w2_rows_permuted(x, w1, w2, w3, act):
        return O.expert_ffn(x, w1, np.asarray(w2)[::-1], w3, act)

    def w1_w3_swapped(x, w1, w2, w3, act):
        return O.expert_ffn(x, w3 if w3 is not None else w1, w2, w1, act)

    def bias_in_weight(z, gate, top_k, select_bias=None):
        r = O.route(z, gate, top_k, select_bias)
        if select_bias is not None:
            g = np.take_along_axis(r["key"].astype(float), r["idx"], 1)
            r["weights"] = g / g.sum(1, keepdims=True)
        return r

    def sigmoid_sign(z):
        return 1.0 / (1.0 + np.exp(np.asarray(z, np.float64)))

    def bias_sign_flipped(loads, select_bias, gamma, routed_rows):
        return O.update_select_bias(loads, select_bias, -gamma, routed_rows)

    def bias_mean_over_tokens(loads, select_bias, gamma, routed_rows):
        # mean taken as T instead of T·k (k = 2 in the controller check)
        return O.update_select_bias(loads, select_bias, gamma, routed_rows // 2)

    def group_by_max(group_key, n_groups, topk_groups):
        gk = np.asarray(group_key, np.float64)
        T, E = gk.shape
        gmax = gk.reshape(T, n_groups, E // n_groups).max(axis=2)
        gidx = O.topk_by_rank(gmax, topk_groups)
        allowed = np.zeros((T, n_groups), dtype=bool)
        np.put_along_axis(allowed, gidx, True, axis=1)
        return np.repeat(allowed, E // n_groups, axis=1), np.full(T, np.inf)

    def f_over_tokens(z, idx, n_routed, top_k, gate):
        f, p = O.balance_stats(z, idx, n_routed, top_k, gate)
        return (f * np.float32(top_k) / np.float32(n_routed)).astype(np.float32), p

    def sigmoid_unnormalised(z, idx, n_routed, top_k, gate):
        f, p = O.balance_stats(z, idx, n_routed, top_k, gate)
        if gate != O.SOFTMAX:
            p = O.sigmoid_scores(z).mean(axis=0)
        return f, p

    cases = [
        (dict(balance_stats=f_over_tokens), check_balance_stats_handworked, (golden_dir,)),
        (dict(balance_stats=f_over_tokens), check_balance_stats_properties, ()),
        (dict(balance_stats=sigmoid_unnormalised), check_balance_stats_handworked, (golden_dir,)),
        (dict(balance_stats=sigmoid_unnormalised), check_balance_stats_properties, ()),
        (dict(group_choice=group_by_max), check_group_routing_handworked, (golden_dir,)),
        (dict(group_choice=group_by_max), check_group_routing_bruteforce, ()),
        (dict(update_select_bias=bias_sign_flipped), check_bias_update_handworked, (golden_dir,)),
        (dict(update_select_bias=bias_sign_flipped), check_bias_controller_balances, ()),
        (dict(update_select_bias=bias_mean_over_tokens), check_bias_controller_balances, ()),
        (dict(route=renormalised_softmax), check_routing_handworked, (golden_dir,)),
        (dict(topk_by_rank=ties_to_higher), check_topk_bruteforce, ()),
        (dict(combine=no_residual), check_ffn_handworked, (golden_dir,)),
        (dict(expert_ffn=w2_rows_permuted), check_ffn_bruteforce, ()),
        (dict(expert_ffn=w1_w3_swapped), check_ffn_handworked, (golden_dir,)),
        (dict(route=bias_in_weight), check_routing_handworked, (golden_dir,)),
        (dict(sigmoid_scores=sigmoid_sign), check_sigmoid_properties, ()),
    ]
    for overrides, check, args in cases:
        assert _fails(check, _mutant(**overrides), *args), (list(overrides), check.__name__)
