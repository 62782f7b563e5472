"""Pins of the oracle's layer backward against the mathematics.

The backward is checked against central finite differences of the forward
(the pinned expert FFN and combine, with the gate weights of the fixed
expert choice), on tiny float64 layers for both gates, both activations,
with and without shared experts; closed forms cover the degenerate cases.
``test_planted_backward_mistakes`` plants slips in copies of the backward
functions and checks that the finite-difference pin catches each.
"""
import math
import types

import numpy as np
import pytest

import oracle.moe_oracle as O

CASES = [(gate, act, ks) for gate in (O.SOFTMAX, O.SIGMOID_BIAS)
         for act in (O.SWIGLU, O.RELU) for ks in (0, 2)]


def _layer(rng, T, H, E, Ks, I, k, gate, act):
    u = rng.standard_normal((T, H))
    cents = rng.standard_normal((E, H)) / math.sqrt(H) * 2
    ws = []
    for _ in range(E + Ks):
        w1 = rng.standard_normal((I, H)) / math.sqrt(H)
        w3 = rng.standard_normal((I, H)) / math.sqrt(H) if act == O.SWIGLU else None
        w2 = rng.standard_normal((H, I)) / math.sqrt(I)
        ws.append([w1, w3, w2])
    z = u @ cents.T
    idx = O.route(z.astype(np.float32), gate, k)["idx"]
    dh = rng.standard_normal((T, H))
    return dict(u=u, cents=cents, ws=ws, idx=idx, dh=dh, E=E, Ks=Ks, k=k, gate=gate, act=act)


def _loss(o, L):
    """Σ dh ⊙ h with the choice held fixed (forward from the pinned pieces)."""
    u, E, Ks = L["u"], L["E"], L["Ks"]
    z = u @ L["cents"].T
    g, _ = o.gate_weights(z, L["idx"], L["gate"])
    T, k = L["idx"].shape
    y_sh = [o.expert_ffn(u, L["ws"][E + j][0], L["ws"][E + j][2], L["ws"][E + j][1], L["act"])
            for j in range(Ks)]
    y_r = np.zeros((T, k, u.shape[1]))
    for t in range(T):
        for s in range(k):
            w1, w3, w2 = L["ws"][L["idx"][t, s]]
            y_r[t, s] = o.expert_ffn(u[t:t + 1], w1, w2, w3, L["act"])[0]
    return float((L["dh"] * o.combine(u, y_sh, y_r, g)).sum())


def _grads(o, L):
    E, Ks = L["E"], L["Ks"]
    z = L["u"] @ L["cents"].T
    return o.layer_backward(L["u"], L["dh"], L["cents"], z, L["idx"], L["gate"],
                            lambda e: (L["ws"][e][0], L["ws"][e][1], L["ws"][e][2]),
                            lambda j: (L["ws"][E + j][0], L["ws"][E + j][1], L["ws"][E + j][2]),
                            E, Ks, L["act"])


def _params(L, G):
    """(getter-setter of a parameter array, its analytic gradient) pairs."""
    E, Ks = L["E"], L["Ks"]
    out = [(("u",), G["du"]), (("cents",), G["d_centroids"])]
    names = {0: "dw1", 1: "dw3", 2: "dw2"}
    for e in range(E + Ks):
        for m in (0, 1, 2):
            if L["ws"][e][m] is None:
                continue
            key = names[m] if e < E else "ds" + names[m][1:]
            grad = G[key][e if e < E else e - E]
            out.append((("ws", e, m), grad))
    return out


def _get(L, path):
    return L[path[0]] if len(path) == 1 else L["ws"][path[1]][path[2]]


def _set(L, path, v):
    if len(path) == 1:
        L[path[0]] = v
    else:
        L["ws"][path[1]][path[2]] = v


def check_finite_differences(o, L, rng, eps=1e-6):
    G = _grads(o, L)
    for path, grad in _params(L, G):
        p0 = _get(L, path)
        v = rng.standard_normal(p0.shape)
        _set(L, path, p0 + eps * v)
        lp = _loss(o, L)
        _set(L, path, p0 - eps * v)
        lm = _loss(o, L)
        _set(L, path, p0)
        fd = (lp - lm) / (2 * eps)
        an = float((np.asarray(grad) * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (path, fd, an)


@pytest.mark.parametrize("gate,act,ks", CASES)
def test_backward_matches_finite_differences(gate, act, ks):
    rng = np.random.default_rng(CASES.index((gate, act, ks)))
    L = _layer(rng, T=5, H=6, E=5, Ks=ks, I=4, k=2, gate=gate, act=act)
    check_finite_differences(O, L, rng)


def test_gate_weights_match_route():
    """gate_weights on fp32 logits equals the pinned router's weights."""
    rng = np.random.default_rng(5)
    z = (rng.standard_normal((50, 9)) * 2).astype(np.float32)
    for gate in (O.SOFTMAX, O.SIGMOID_BIAS):
        r = O.route(z, gate, 3)
        g, s = O.gate_weights(z, r["idx"], gate)
        assert np.array_equal(g, r["weights"])
        assert np.array_equal(s, r["scores"])


def test_backward_closed_forms():
    """k = 0 and no shared experts: du = dh and every other gradient is zero.
    A ReLU expert whose pre-activations are all positive is linear:
    dx = dy W2 W1, dW2 = dyᵀ (x W1ᵀ), dW1 = (dy W2)ᵀ x."""
    rng = np.random.default_rng(9)
    T, H, E, I = 4, 6, 3, 5
    u = rng.standard_normal((T, H))
    dh = rng.standard_normal((T, H))
    cents = rng.standard_normal((E, H))
    w = lambda e: (rng.standard_normal((I, H)), None, rng.standard_normal((H, I)))
    G = O.layer_backward(u, dh, cents, u @ cents.T, np.zeros((T, 0), np.int64), O.SOFTMAX,
                         w, w, E, 0, O.RELU)
    assert np.array_equal(G["du"], dh)
    assert not G["d_centroids"].any() and not G["dw1"].any() and not G["dw2"].any()
    x = np.abs(rng.standard_normal((T, H)))
    w1 = np.abs(rng.standard_normal((I, H)))
    w2 = rng.standard_normal((H, I))
    dy = rng.standard_normal((T, H))
    dx, dw1, dw3, dw2 = O.expert_ffn_backward(x, w1, w2, None, O.RELU, dy)
    assert dw3 is None
    assert np.allclose(dx, dy @ w2 @ w1, rtol=1e-13, atol=1e-12)
    assert np.allclose(dw2, dy.T @ (x @ w1.T), rtol=1e-13, atol=1e-12)
    assert np.allclose(dw1, (dy @ w2).T @ x, rtol=1e-13, atol=1e-12)


def test_gate_backward_invariants():
    """softmax: Σ_j dz_j = 0 (the scores sum to 1); sigmoid: the weights are
    invariant to a common scale of the chosen scores, so Σ_chosen ds_i s_i = 0,
    and unchosen experts get no gradient."""
    rng = np.random.default_rng(13)
    z = rng.standard_normal((20, 7)) * 2
    idx = O.route(z.astype(np.float32), O.SOFTMAX, 3)["idx"]
    dg = rng.standard_normal((20, 3))
    dz = O.gate_backward(z, idx, O.SOFTMAX, dg)
    assert np.abs(dz.sum(axis=1)).max() < 1e-14
    dz = O.gate_backward(z, idx, O.SIGMOID_BIAS, dg)
    s = 1 / (1 + np.exp(-z))
    ds = dz / (s * (1 - s))
    assert np.abs((ds * s).sum(axis=1)).max() < 1e-13
    mask = np.ones_like(dz, dtype=bool)
    np.put_along_axis(mask, idx, False, axis=1)
    assert not dz[mask].any()


def _copy_oracle(**overrides):
    m = types.ModuleType("mutant")
    m.__dict__.update({k: v for k, v in O.__dict__.items() if not k.startswith("__")})
    for name, fn in list(m.__dict__.items()):
        if isinstance(fn, types.FunctionType):
            m.__dict__[name] = types.FunctionType(fn.__code__, m.__dict__, name,
                                                  fn.__defaults__, fn.__closure__)
    m.__dict__.update(overrides)
    return m


def test_planted_backward_mistakes():
    def silu_prime_without_second_term(x, w1, w2, w3, act, dy):
        if act != O.SWIGLU:
            return O.expert_ffn_backward(x, w1, w2, w3, act, dy)
        a, c = x @ w1.T, x @ w3.T
        sg = 1 / (1 + np.exp(-a))
        dm = dy @ w2
        da, dc = dm * c * sg, dm * a * sg
        return da @ w1 + dc @ w3, da.T @ x, dc.T @ x, dy.T @ (a * sg * c)

    def dw2_from_preactivation(x, w1, w2, w3, act, dy):
        dx, dw1, dw3, _ = O.expert_ffn_backward(x, w1, w2, w3, act, dy)
        return dx, dw1, dw3, dy.T @ (x @ w1.T)

    def softmax_without_centering(z, idx, gate, dg):
        if gate != O.SOFTMAX:
            return O.gate_backward(z, idx, gate, dg)
        _, s = O.gate_weights(z, idx, gate)
        ds = np.zeros_like(s)
        np.put_along_axis(ds, idx, dg, axis=1)
        return s * ds

    def sigmoid_without_derivative(z, idx, gate, dg):
        if gate == O.SOFTMAX:
            return O.gate_backward(z, idx, gate, dg)
        g, s = O.gate_weights(z, idx, gate)
        sc = np.take_along_axis(s, idx, axis=1)
        dz = np.zeros_like(s)
        np.put_along_axis(dz, idx, (dg - (dg * g).sum(1, keepdims=True)) / sc.sum(1, keepdims=True),
                          axis=1)
        return dz

    def no_residual(u, dh, *args):
        G = O.layer_backward(u, dh, *args)
        G["du"] = G["du"] - dh
        return G

    cases = [
        (dict(expert_ffn_backward=silu_prime_without_second_term), O.SOFTMAX, O.SWIGLU),
        (dict(expert_ffn_backward=dw2_from_preactivation), O.SOFTMAX, O.RELU),
        (dict(gate_backward=softmax_without_centering), O.SOFTMAX, O.SWIGLU),
        (dict(gate_backward=sigmoid_without_derivative), O.SIGMOID_BIAS, O.RELU),
        (dict(layer_backward=no_residual), O.SIGMOID_BIAS, O.SWIGLU),
    ]
    for overrides, gate, act in cases:
        m = _copy_oracle(**overrides)
        rng = np.random.default_rng(1)
        L = _layer(rng, T=5, H=6, E=5, Ks=1, I=4, k=2, gate=gate, act=act)
        with pytest.raises(AssertionError):
            check_finite_differences(m, L, rng)


def test_expert_subset_matches_full_evaluation():
    """Evaluating only the chosen experts gives the same du and the same
    per-expert gradients as evaluating all of them."""
    rng = np.random.default_rng(21)
    L = _layer(rng, T=6, H=6, E=7, Ks=1, I=4, k=2, gate=O.SIGMOID_BIAS, act=O.SWIGLU)
    full = _grads(O, L)
    used = np.unique(L["idx"])
    z = L["u"] @ L["cents"].T
    E = L["E"]
    sub = O.layer_backward(L["u"], L["dh"], L["cents"], z, L["idx"], L["gate"],
                           lambda e: tuple(L["ws"][e]), lambda j: tuple(L["ws"][E + j]),
                           E, L["Ks"], L["act"], experts=used)
    assert np.array_equal(sub["du"], full["du"])
    for e in used:
        for key in ("dw1", "dw3", "dw2"):
            assert np.array_equal(sub[key][e], full[key][e])
    with pytest.raises(ValueError):
        O.layer_backward(L["u"], L["dh"], L["cents"], z, L["idx"], L["gate"],
                         lambda e: tuple(L["ws"][e]), lambda j: tuple(L["ws"][E + j]),
                         E, L["Ks"], L["act"], experts=used[1:])


def test_backward_hand_derived_single_token():
    """One token u = (1, 2), centroids e0 = (1, 0), e1 = (0, 1): z = (1, 2),
    softmax s = (1, e) / (1 + e), top-1 picks expert 1 with g = s1.  Expert 1
    is ReLU with W1 = [1 1], W2 = [1 2]ᵀ: a = 3, y = (3, 6).  For dh = (1, 1):
    dg = <dh, y> = 9; dz_1 = s1 (dg − dg s1) = 9 s1 s0, dz_0 = −9 s1 s0;
    J = W2 W1 (a > 0), Jᵀ dh = (3, 3); du = dh + g Jᵀ dh + (dz_0, dz_1);
    dm = W2ᵀ (g dh) = 3 g, dW1 = 3 g (1, 2), dW2 = (3 g, 3 g)ᵀ;
    d e_i = dz_i (1, 2).  Expert 0 was not chosen: zero gradients."""
    e = math.e
    s1 = e / (1 + e)
    s0 = 1 - s1
    g = s1
    u = np.array([[1.0, 2.0]])
    dh = np.array([[1.0, 1.0]])
    cents = np.array([[1.0, 0.0], [0.0, 1.0]])
    W = {0: (np.array([[0.5, -0.5]]), None, np.array([[1.0], [1.0]])),
         1: (np.array([[1.0, 1.0]]), None, np.array([[1.0], [2.0]]))}
    z = u @ cents.T
    idx = O.route(z.astype(np.float32), O.SOFTMAX, 1)["idx"]
    assert idx.tolist() == [[1]]
    G = O.layer_backward(u, dh, cents, z, idx, O.SOFTMAX, lambda k: W[k], lambda j: None,
                         2, 0, O.RELU)
    dz0, dz1 = -9 * s1 * s0, 9 * s1 * s0
    assert np.allclose(G["dg"], [[9.0]], rtol=1e-14)
    assert np.allclose(G["dz"], [[dz0, dz1]], rtol=1e-12)
    assert np.allclose(G["du"], [[1 + 3 * g + dz0, 1 + 3 * g + dz1]], rtol=1e-12)
    assert np.allclose(G["dw1"][1], [[3 * g, 6 * g]], rtol=1e-12)
    assert np.allclose(G["dw2"][1], [[3 * g], [3 * g]], rtol=1e-12)
    assert not G["dw1"][0].any() and not G["dw2"][0].any()
    assert np.allclose(G["d_centroids"], [[dz0, 2 * dz0], [dz1, 2 * dz1]], rtol=1e-12)


def test_backward_hand_derived_sigmoid_two_chosen():
    """Sigmoid gate, both of two experts chosen, z = (0, 0): s = (1/2, 1/2),
    g = s / Σ s = (1/2, 1/2).  Linear ReLU experts (positive pre-activation)
    give y_0 = (1, 0), y_1 = (0, 3) for u = (1, 0), so for dh = (2, 1):
    dg = (2, 3); ds_j = (dg_j − Σ_i dg_i g_i) / S = (−1/2, 1/2);
    dz_j = ds_j s_j (1 − s_j) = (−1/8, 1/8)."""
    u = np.array([[1.0, 0.0]])
    dh = np.array([[2.0, 1.0]])
    cents = np.zeros((2, 2))                       # z = 0 for both experts
    W = {0: (np.array([[1.0, 0.0]]), None, np.array([[1.0], [0.0]])),
         1: (np.array([[1.0, 0.0]]), None, np.array([[0.0], [3.0]]))}
    z = u @ cents.T
    idx = np.array([[0, 1]])
    G = O.layer_backward(u, dh, cents, z, idx, O.SIGMOID_BIAS, lambda k: W[k], lambda j: None,
                         2, 0, O.RELU)
    assert np.allclose(G["dg"], [[2.0, 3.0]], rtol=1e-14)
    assert np.allclose(G["dz"], [[-0.125, 0.125]], rtol=1e-14)
    # du = dh + Σ_s g_s J_sᵀ dh + centroidsᵀ dz; J_0ᵀ dh = (2, 0), J_1ᵀ dh = (3, 0)
    assert np.allclose(G["du"], [[2.0 + 0.5 * 2 + 0.5 * 3, 1.0]], rtol=1e-14)
