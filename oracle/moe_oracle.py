"""CPU oracle for the DeepSeekMoE layer forward and its backward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

Plain NumPy in float64, written straight from the equations on the source
pages, with no blocking, fusion or reordering beyond what the equations state.
Page titles cited below:

  [FG]  "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE" (llm-infra-atlas): §2.1
        segmentation and its Eq. 6–8 (softmax gating, top-mK, no
        renormalisation); §2.2 the combination counts; §3.1 shared-expert
        isolation Eq. 9–11 (h = Σ shared + Σ g·routed + u) and the DeepSeek-V3
        form Eq. 12–15 (sigmoid scores, weights normalised over the selected).
  [CH7] "MoE 的分水岭——DeepSeek 配方与 2026 年的主流形态" (ibossgateway,
        ch. 7): §7.4, the per-expert bias b_i is added to the scores for the
        choice only, the weights use the raw scores; §7.2 the counts C(8,2)
        and "64 choose 8".
  [PS]  "19-deepseek-moe" (ai.tomabc.com paper story): the expert FFN written
        as ReLU(x W_i) then a projection (we drop the biases), and the
        three-term forward (shared, routed, residual).

Readings where the pages are silent or disagree (each also listed in the
design notes):
  * Softmax is applied over the routed experts' logits and the selected
    scores are NOT renormalised (FG Eq. 6–8); the [PS] wording that masks the
    non-selected logits to -inf before the softmax is not followed.
  * Softmax is strictly increasing in the logit with a common denominator, so
    the top mK of the exact scores are the top mK of the logits: the choice
    is taken on the fp32 logits themselves (exact), ties to the lower index.
  * The V3 choice key is s_i + b_i taken in fp32, as the kernel takes it:
    fp32(fp32(sigmoid(z_i)) + b_i), with sigmoid evaluated in float64 and
    rounded once.  Gate weights use float64 scores.
  * No FFN biases; SwiGLU is (SiLU(x W1ᵀ) ⊙ x W3ᵀ) W2ᵀ; SiLU(a) = a/(1+e^-a).
  * An optional per-expert logit offset o_i is added to the logit before
    scoring (it changes choice and weight alike, unlike b_i).
  * Dispatch order: permuted rows sorted by expert, then token (each token
    picks an expert at most once, so slot order never decides).

Weight layout (nn.Linear convention, contracted dimension last):
  centroids [E, H]; w1, w3 [I, H] per expert; w2 [H, I] per expert.
"""
from __future__ import annotations

from math import comb
from typing import Callable, Optional, Sequence

import numpy as np

SOFTMAX = "softmax"
SIGMOID_BIAS = "sigmoid_bias"
RELU = "relu"
SWIGLU = "swiglu"


# --------------------------------------------------------------------------
# Shapes from the segmentation rule ([FG] §2.1, §3.1)
# --------------------------------------------------------------------------

def segmented_shape(N: int, M: int, m: int, K: int, Ks: int = 0):
    """Fine-grained segmentation plus shared isolation, as in [FG] §2.1/§3.1.

    N base experts of width M, K active, split m ways: mN experts of width
    M/m with mK active; Ks of the mN are made shared (always on), so the
    router chooses mK - Ks among the remaining mN - Ks.
    Returns (n_routed, inter, top_k).
    """
    if M % m:
        raise ValueError("M must divide by m")
    return m * N - Ks, M // m, m * K - Ks


def iso_identities(N, M, m, K, Ks, H):
    """[FG] §2.1: parameters mN·H·(M/m) = N·H·M and active mK·H·(M/m) = K·H·M.

    Counts shared experts inside mN and mK (FG Eq. 9–11 numbers them as part
    of the mN pool).  Returns ((lhs, rhs) params, (lhs, rhs) active).
    """
    n_routed, inter, top_k = segmented_shape(N, M, m, K, Ks)
    params = ((n_routed + Ks) * H * inter, N * H * M)
    active = ((top_k + Ks) * H * inter, K * H * M)
    return params, active


def routing_combinations(n_routed: int, top_k: int) -> int:
    """Number of distinct expert sets a token can pick ([FG] §2.2)."""
    return comb(n_routed, top_k)


# --------------------------------------------------------------------------
# Router ([FG] Eq. 6–8, Eq. 12–15; [CH7] §7.4)
# --------------------------------------------------------------------------

def router_logits(u: np.ndarray, centroids: np.ndarray,
                  logit_offset: Optional[np.ndarray] = None) -> np.ndarray:
    """z_{t,i} = u_tᵀ e_i (+ o_i), accumulated in float64, rounded to fp32."""
    z = np.asarray(u, np.float64) @ np.asarray(centroids, np.float64).T
    if logit_offset is not None:
        z = z + np.asarray(logit_offset, np.float64)[None, :]
    return z.astype(np.float32)


def softmax_scores(z: np.ndarray) -> np.ndarray:
    """s_{i,t} = softmax_i(z_{t,i}) over the routed experts, float64."""
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def sigmoid_scores(z: np.ndarray) -> np.ndarray:
    """s_{i,t} = 1 / (1 + exp(-z_{t,i})), float64 ([FG] Eq. 12)."""
    z = np.asarray(z, np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def topk_by_rank(key: np.ndarray, k: int) -> np.ndarray:
    """Top-k by the counting definition, ties to the lower index.

    Expert i's rank is #{j : key_j > key_i} + #{j < i : key_j == key_i};
    i is chosen iff rank < k, and the output lists the chosen experts by
    rank (descending key, lower index first on ties).  Returns int64 [T, k].
    """
    key = np.asarray(key)
    T, E = key.shape
    out = np.empty((T, k), dtype=np.int64)
    lower = np.tril(np.ones((E, E), dtype=bool), -1)  # lower[i, j] = j < i
    step = max(1, (1 << 22) // max(1, E * E))
    for t0 in range(0, T, step):
        kc = key[t0:t0 + step]
        ki = kc[:, :, None]   # [c, i, 1]
        kj = kc[:, None, :]   # [c, 1, j]
        rank = (kj > ki).sum(axis=2) + ((kj == ki) & lower[None]).sum(axis=2)
        for c in range(kc.shape[0]):
            chosen = np.nonzero(rank[c] < k)[0]
            out[t0 + c, rank[c, chosen]] = chosen
    return out


def selection_key(z: np.ndarray, gate: str,
                  select_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """The quantity the top-k is taken on (see the module readings)."""
    if gate == SOFTMAX:
        return np.asarray(z, np.float32)
    if gate == SIGMOID_BIAS:
        s32 = sigmoid_scores(z).astype(np.float32)
        b = (np.zeros(z.shape[1], np.float32) if select_bias is None
             else np.asarray(select_bias, np.float32))
        return s32 + b[None, :]          # fp32 + fp32 -> fp32, one rounding
    raise ValueError(gate)


def group_choice(group_key: np.ndarray, n_groups: int, topk_groups: int):
    """Node/group-limited routing, first stage ([FG] §4): the E routed experts
    form n_groups groups of E / n_groups consecutive experts; a group's score
    is the sum of its experts' scores (float64); the topk_groups best groups
    are kept, ties to the lower group index.  Returns (allowed [T,E] bool,
    gap [T]: the topk_groups-th minus the next group score, +inf if all kept).
    """
    group_key = np.asarray(group_key, np.float64)
    T, E = group_key.shape
    gs = E // n_groups
    gsum = group_key.reshape(T, n_groups, gs).sum(axis=2)
    gidx = topk_by_rank(gsum, min(topk_groups + 1, n_groups))
    allowed = np.zeros((T, n_groups), dtype=bool)
    np.put_along_axis(allowed, gidx[:, :topk_groups], True, axis=1)
    gap = np.full(T, np.inf)
    if topk_groups < n_groups:
        rows = np.arange(T)
        gap = gsum[rows, gidx[:, topk_groups - 1]] - gsum[rows, gidx[:, topk_groups]]
    return np.repeat(allowed, gs, axis=1), gap


def route(z: np.ndarray, gate: str, top_k: int,
          select_bias: Optional[np.ndarray] = None, n_groups: int = 0,
          topk_groups: int = 0):
    """Scores, choice and gate weights for every token.

    Returns dict(idx [T,k] int64, weights [T,k] float64, scores [T,E] float64,
    key [T,E], gap [T] float64, group_gap [T]).  gap is the k-th minus the
    (k+1)-th largest score (softmax) or key (sigmoid + bias) among the experts
    the token may choose; +inf when there is no (k+1)-th.  With n_groups > 0
    the choice is group-limited ([FG] §4): groups are scored by the sum of the
    scores the choice is made on — the softmax scores rounded to fp32, or the
    fp32 keys s + b —
    and only experts of the topk_groups best groups may be chosen; group_gap
    is the margin of the last kept group (+inf without groups).
    """
    z = np.asarray(z, np.float32)
    T, E = z.shape
    scores = softmax_scores(z) if gate == SOFTMAX else sigmoid_scores(z)
    key = selection_key(z, gate, select_bias)
    group_gap = np.full(T, np.inf)
    choice_key = key
    if n_groups > 0:
        # the group decision is taken in the kernel's precision: fp32 scores
        # (softmax) or the fp32 keys, summed in float64
        gkey = scores.astype(np.float32) if gate == SOFTMAX else key
        allowed, group_gap = group_choice(gkey, n_groups, topk_groups)
        choice_key = np.where(allowed, key, np.float32(-np.inf))
    idx = topk_by_rank(choice_key, min(top_k + 1, E))
    gap = np.full(T, np.inf)
    if 0 < top_k < E:
        rows = np.arange(T)
        gap_src = scores if gate == SOFTMAX else key.astype(np.float64)
        nxt = idx[:, top_k]
        has_next = np.isfinite(choice_key[rows, nxt])
        gap = np.where(has_next, gap_src[rows, idx[:, top_k - 1]] - gap_src[rows, nxt], np.inf)
    idx = idx[:, :top_k]
    g = np.take_along_axis(scores, idx, axis=1)
    if gate == SIGMOID_BIAS and top_k > 0:
        g = g / g.sum(axis=1, keepdims=True)     # [FG] Eq. 15, raw scores only
    return dict(idx=idx, weights=g, scores=scores, key=key, gap=gap, group_gap=group_gap)


# --------------------------------------------------------------------------
# Dispatch (grouping rows by expert; no token is dropped)
# --------------------------------------------------------------------------

def dispatch(idx: np.ndarray, n_routed: int):
    """Per-expert counts, offsets and the stable token permutation.

    Rows of the permuted buffer are sorted by expert, then by token; row r
    holds token row_token[r]; slot_row[t, s] is the row of (token t, slot s).
    """
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=n_routed).astype(np.int64)
    offsets = np.zeros(n_routed + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")       # (expert, token, slot)
    row_token = order // max(k, 1)
    slot_row = np.empty(T * k, np.int64)
    slot_row[order] = np.arange(T * k)
    return dict(counts=counts, offsets=offsets, row_token=row_token,
                slot_row=slot_row.reshape(T, k))


# --------------------------------------------------------------------------
# Load balancing without an auxiliary loss ([CH7] §7.4)
# --------------------------------------------------------------------------

def expert_loads(idx: np.ndarray, n_routed: int) -> np.ndarray:
    """Tokens routed to each expert in one step (every (token, slot) counts once)."""
    return np.bincount(np.asarray(idx, np.int64).reshape(-1), minlength=n_routed)


def update_select_bias(loads: np.ndarray, select_bias: np.ndarray, gamma: float,
                       routed_rows: int) -> np.ndarray:
    """One step of the per-expert bias controller of [CH7] §7.4.

    After a step each expert's load is compared with the mean load
    routed_rows / E (routed_rows = T·k): an overloaded expert's bias is lowered
    by the step gamma, an underloaded expert's bias is raised by gamma, an
    expert exactly at the mean keeps its bias.  The pages give no value for
    gamma (FG §5 calls it a step coupled to the score scale): it is a
    parameter.  Returned in float32, the type the router adds it in.
    """
    loads = np.asarray(loads, np.int64)
    E = loads.shape[0]
    over = loads * E > routed_rows           # load_i > mean, compared exactly
    under = loads * E < routed_rows
    b = np.asarray(select_bias, np.float64).copy()
    b[over] -= float(np.float32(gamma))
    b[under] += float(np.float32(gamma))
    return b.astype(np.float32)


def balance_stats(z: np.ndarray, idx: np.ndarray, n_routed: int, top_k: int,
                  gate: str):
    """Per-expert statistics of the expert-level balance loss ([PS], load
    balance section): f_i, the actual routing distribution, and P_i, the
    gate's mean probability for expert i; the loss is proportional to
    Σ_i f_i P_i.  The page's formula did not survive extraction; the reading:

      f_i = E · #{(t, s) : idx[t, s] = i} / (k · T)   (the count runs over all
            E routed experts, so a perfectly even routing gives f_i = 1);
      P_i = (1/T) Σ_t p_{i,t}, p_t the token's gate distribution over the E
            routed experts: the softmax scores, or for the sigmoid gate the
            scores divided by their sum over all E (so Σ_i P_i = 1 for both).

    z are the fp32 logits (logit offset included).  f is returned in float32
    (one rounding of the exact ratio), P in float64.  k = 0 gives f = 0.
    """
    z = np.asarray(z, np.float64)
    T = z.shape[0]
    E = n_routed
    loads = expert_loads(idx, E) if T and top_k else np.zeros(E, np.int64)
    if T == 0 or top_k == 0:
        f = np.zeros(E, np.float32)
    else:
        f = ((E * loads).astype(np.float64) / float(top_k * T)).astype(np.float32)
    if T == 0:
        return f, np.zeros(E, np.float64)
    if gate == SOFTMAX:
        p = softmax_scores(z)
    else:
        s = sigmoid_scores(z)
        p = s / s.sum(axis=1, keepdims=True)
    return f, p.sum(axis=0) / T


# --------------------------------------------------------------------------
# Expert FFN and combine ([PS]; [FG] Eq. 9–11)
# --------------------------------------------------------------------------

def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def expert_ffn(x: np.ndarray, w1: np.ndarray, w2: np.ndarray,
               w3: Optional[np.ndarray], act: str) -> np.ndarray:
    """One expert on the rows of x, float64.

    relu:   y = ReLU(x W1ᵀ) W2ᵀ
    swiglu: y = (SiLU(x W1ᵀ) ⊙ (x W3ᵀ)) W2ᵀ
    """
    x = np.asarray(x, np.float64)
    a = x @ np.asarray(w1, np.float64).T
    if act == RELU:
        hmid = np.maximum(a, 0.0)
    elif act == SWIGLU:
        hmid = silu(a) * (x @ np.asarray(w3, np.float64).T)
    else:
        raise ValueError(act)
    return hmid @ np.asarray(w2, np.float64).T


def combine(u: np.ndarray, y_shared: Sequence[np.ndarray],
            y_routed: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """h_t = Σ_j y^shared_{j,t} + Σ_s g_{t,s} y_{t,s} + u_t  ([FG] Eq. 9–11).

    y_routed is [T, k, H] (the output of the expert chosen in each slot),
    weights [T, k].
    """
    h = np.asarray(u, np.float64).copy()
    for ys in y_shared:
        h += ys
    if y_routed.shape[1]:
        h += (np.asarray(weights, np.float64)[:, :, None] * y_routed).sum(axis=1)
    return h


ExpertFn = Callable[[int], tuple]   # e -> (w1, w3 or None, w2) as float64 arrays


def layer_forward(u: np.ndarray, route_out: dict, routed: ExpertFn,
                  shared: ExpertFn, n_shared: int, act: str,
                  rows: Optional[np.ndarray] = None) -> np.ndarray:
    """h for the tokens ``rows`` (all tokens if None), float64.

    ``route_out`` is the result of :func:`route` for all tokens; ``routed``
    and ``shared`` return an expert's weights on demand, so that large layers
    can be evaluated one expert at a time.
    """
    u = np.asarray(u, np.float64)
    rows = np.arange(u.shape[0]) if rows is None else np.asarray(rows)
    x = u[rows]
    idx = route_out["idx"][rows]
    g = route_out["weights"][rows]
    n, k = idx.shape
    y_sh = []
    for j in range(n_shared):
        w1, w3, w2 = shared(j)
        y_sh.append(expert_ffn(x, w1, w2, w3, act))
    y_r = np.zeros((n, k, u.shape[1]))
    for e in np.unique(idx):
        tt, ss = np.nonzero(idx == e)
        w1, w3, w2 = routed(int(e))
        y_r[tt, ss] = expert_ffn(x[tt], w1, w2, w3, act)
    return combine(x, y_sh, y_r, g)


# --------------------------------------------------------------------------
# Backward of the layer (training side of [FG] Eq. 9–15 and [PS])
# --------------------------------------------------------------------------
# The choice of experts is piecewise constant in the logits, so gradients
# flow through the gate weights, the expert FFNs and the residual, with the
# chosen set held fixed; the selection bias (choice only) gets none.

def gate_weights(z: np.ndarray, idx: np.ndarray, gate: str):
    """Gate weights of the chosen experts as a function of float64 logits.

    softmax: g = s_i for the chosen i, s = softmax over the E routed logits
    ([FG] Eq. 6–8, no renormalisation); sigmoid: g = s_i / Σ_chosen s_j,
    s = sigmoid(z) ([FG] Eq. 12–15).  Returns (g [T,k], s [T,E]).
    """
    z = np.asarray(z, np.float64)
    s = softmax_scores(z) if gate == SOFTMAX else sigmoid_scores(z)
    idx = np.asarray(idx, np.int64)
    g = np.take_along_axis(s, idx, axis=1)
    if gate == SIGMOID_BIAS and idx.shape[1] > 0:
        g = g / g.sum(axis=1, keepdims=True)
    return g, s


def gate_backward(z: np.ndarray, idx: np.ndarray, gate: str, dg: np.ndarray) -> np.ndarray:
    """dL/dz [T,E] from dL/dg [T,k] for the fixed choice idx.

    softmax: ∂s_i/∂z_j = s_i (δ_ij − s_j), so dz_j = s_j (dg_j [j chosen]
    − Σ_chosen dg_i s_i).  sigmoid: ∂g_i/∂s_j = (δ_ij − g_i) / S for chosen
    j (S = Σ_chosen s), ds/dz = s (1 − s), unchosen experts get 0.
    """
    g, s = gate_weights(z, idx, gate)
    idx = np.asarray(idx, np.int64)
    dg = np.asarray(dg, np.float64)
    T, E = s.shape
    dz = np.zeros((T, E))
    if idx.shape[1] == 0:
        return dz
    if gate == SOFTMAX:
        ds = np.zeros((T, E))
        np.put_along_axis(ds, idx, dg, axis=1)
        dz = s * (ds - (ds * s).sum(axis=1, keepdims=True))
    else:
        sc = np.take_along_axis(s, idx, axis=1)
        S = sc.sum(axis=1, keepdims=True)
        ds_sel = (dg - (dg * g).sum(axis=1, keepdims=True)) / S
        np.put_along_axis(dz, idx, ds_sel * sc * (1.0 - sc), axis=1)
    return dz


def expert_ffn_backward(x: np.ndarray, w1: np.ndarray, w2: np.ndarray,
                        w3: Optional[np.ndarray], act: str, dy: np.ndarray):
    """Gradients of y = expert_ffn(x) for the upstream dL/dy, float64.

    With a = x W1ᵀ, c = x W3ᵀ and m = ReLU(a) or SiLU(a) ⊙ c (y = m W2ᵀ):
    dm = dy W2; relu: da = dm ⊙ [a > 0]; swiglu: da = dm ⊙ c ⊙ SiLU'(a),
    dc = dm ⊙ SiLU(a), SiLU'(a) = σ(a) (1 + a (1 − σ(a))).
    Returns (dx, dw1, dw3 or None, dw2) with dw1 = daᵀ x, dw3 = dcᵀ x,
    dw2 = dyᵀ m, dx = da W1 + dc W3.
    """
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    w1 = np.asarray(w1, np.float64)
    w2 = np.asarray(w2, np.float64)
    a = x @ w1.T
    dm = dy @ w2
    if act == RELU:
        m = np.maximum(a, 0.0)
        da = dm * (a > 0)
        return da @ w1, da.T @ x, None, dy.T @ m
    if act != SWIGLU:
        raise ValueError(act)
    w3 = np.asarray(w3, np.float64)
    c = x @ w3.T
    sg = 1.0 / (1.0 + np.exp(-a))
    m = a * sg * c
    da = dm * c * sg * (1.0 + a * (1.0 - sg))
    dc = dm * a * sg
    return da @ w1 + dc @ w3, da.T @ x, dc.T @ x, dy.T @ m


def layer_backward(u: np.ndarray, dh: np.ndarray, centroids: np.ndarray,
                   z: np.ndarray, idx: np.ndarray, gate: str, routed: ExpertFn,
                   shared: ExpertFn, n_routed: int, n_shared: int, act: str,
                   experts: Optional[Sequence[int]] = None):
    """Gradients of L = Σ dh ⊙ h (h from :func:`layer_forward` with the gate
    weights of :func:`gate_weights`) for the fixed choice idx, float64.

    h_t = u_t + Σ_j FFN_j^sh(u_t) + Σ_s g_{t,s} FFN_{idx[t,s]}(u_t) and
    z_t = centroids u_t (+ offset), so
      du_t = dh_t + Σ_j J_j^T dh_t + Σ_s g_{t,s} J_{idx[t,s]}^T dh_t + Σ_i dz_{t,i} e_i,
      dg_{t,s} = <dh_t, FFN_{idx[t,s]}(u_t)>,  d e_i = Σ_t dz_{t,i} u_t.
    Returns dict(du, d_centroids, dg, dz, dw1, dw3, dw2 [E, ...] and the
    shared dsw1, dsw3, dsw2 [Ks, ...]); experts nobody chose get zeros;
    dw3 / dsw3 are None for ReLU.  ``experts`` (for large layers) evaluates
    only those routed experts — every expert a given token chose must be
    among them — and returns dw1 / dw3 / dw2 as dicts expert -> array.
    """
    u = np.asarray(u, np.float64)
    dh = np.asarray(dh, np.float64)
    idx = np.asarray(idx, np.int64)
    T, H = u.shape
    k = idx.shape[1]
    g, _ = gate_weights(z, idx, gate)
    du = dh.copy()
    out = dict(dsw1=[], dsw3=[], dsw2=[])
    for j in range(n_shared):
        w1, w3, w2 = shared(j)
        dx, dw1, dw3, dw2 = expert_ffn_backward(u, w1, w2, w3, act, dh)
        du += dx
        out["dsw1"].append(dw1)
        out["dsw3"].append(dw3)
        out["dsw2"].append(dw2)
    dg = np.zeros((T, k))
    if experts is not None:
        missing = set(np.unique(idx).tolist()) - set(int(e) for e in experts)
        if missing:
            raise ValueError(f"chosen experts not evaluated: {sorted(missing)[:5]}")
    loop = range(n_routed) if experts is None else [int(e) for e in experts]
    dw1s, dw3s, dw2s = {}, {}, {}
    for e in loop:
        w1, w3, w2 = routed(e)
        tt, ss = np.nonzero(idx == e)
        x = u[tt]
        dg[tt, ss] = (dh[tt] * expert_ffn(x, w1, w2, w3, act)).sum(axis=1)
        dy = g[tt, ss][:, None] * dh[tt]
        dx, dw1s[e], dw3s[e], dw2s[e] = expert_ffn_backward(x, w1, w2, w3, act, dy)
        du[tt] += dx            # a token picks an expert at most once
    dz = gate_backward(z, idx, gate, dg)
    cents = np.asarray(centroids, np.float64)
    du += dz @ cents
    if experts is None:
        stack = lambda d: np.stack([d[e] for e in range(n_routed)])
        out.update(dw1=stack(dw1s), dw2=stack(dw2s),
                   dw3=None if act == RELU else stack(dw3s))
    else:
        out.update(dw1=dw1s, dw2=dw2s, dw3=None if act == RELU else dw3s)
    out.update(du=du, d_centroids=dz.T @ u, dg=dg, dz=dz)
    for key in ("dsw1", "dsw2", "dsw3"):
        vals = out[key]
        out[key] = None if (not vals or vals[0] is None) else np.stack(vals)
    return out


def layer_flops(T: int, H: int, inter: int, top_k: int, n_shared: int,
                act: str) -> int:
    """Algorithmic expert-FFN FLOPs: every routed row and shared row computed."""
    mats = 3 if act == SWIGLU else 2
    return T * (top_k + n_shared) * mats * 2 * H * inter
