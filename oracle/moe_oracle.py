"""Plain CPU oracle for the forward pass of a Mixture-of-Experts SwiGLU FFN layer.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the benchmark's CPU
baseline leg may import or run this module.  It shares no code with the CUDA path and
never imports it.  It is written for clarity, not speed: fp64 arithmetic on the exact
bf16/fp32 input values, one definition per step, in the order the pages give.

What the layer computes (source pages, by title and section):
  * "MoE compute and communication", section 二.2 (MoE 层的结构): router s = f(W_r x) with
    W_r in R^{E x d}, f = softmax or sigmoid; top-k; gate weights g_i = s_i / sum_{TopK} s_j;
    y = sum_{i in TopK} g_i FFN_i(x) + sum_shared FFN_shared(x).
  * same page, section 七.3 (aux-loss-free): selection uses s_i + b_i, weights use s_i.
  * "Mixture of Experts: router, token dispatch, grouped GEMM", section "Router 的选择过程":
    top-k on the raw logits, then softmax over the k selected logits.
  * "DeepSeek-V4 MoE", eq. dsv4-moe-softplus: affinity sqrt(Softplus(x)) = sqrt(ln(1+e^x)).
  * "DeepSeek-V4 MoE", section "V3 的节点路由约束" and "MoE compute and communication",
    section 五.3: group-limited routing -- each group is scored by the sum of its top
    K_r/M affinities, the top M groups are kept, then top-k experts inside them.
  * "DeepSeek-V4 MoE sources analysis" (SGLang walk), section 二 (HashTopK): expert ids come
    from tid2eid[token_id]; the experts still compute on the hidden state.
  * SwiGLU expert W2(SiLU(W1 x) * W3 x) with gate/up fused as w13 -- same SGLang page,
    section 四; "MoE compute and communication", section 二.1.
  * Dispatch: expert-major rows, permuted_token_ids / tokens_per_expert -- "Mixture of
    Experts: router, token dispatch, grouped GEMM", section "Token Dispatch".
  * Combine: y[token] += weight * expert_output[position] -- same page, "Token Combine".
  * Selection-bias update (aux-loss-free balancing): after a step, an overloaded expert's bias
    drops by gamma and an underloaded one's rises by gamma (gamma = 0.001) -- "MoE compute and
    communication", section 七.3; "DeepSeek-V4 MoE", section "负载均衡为什么要 Auxiliary-Loss-Free".

Readings where the pages are silent (each is listed with its reason in the design notes):
  * Selection keys and group scores are compared in fp64 (like every other step here), ties
    go to the lower expert (group) id, and the k ids are returned in descending key order.
  * The expert FFN is the plain definition, with no rounding of the activation h between the
    two projections (the layer definition on "MoE compute and communication", sec. 二.1/二.2,
    has none; the FP8 re-quantisation in the "DeepSeek-V4 MoE" stage table belongs to that
    system's FP8 kernels).  cast_h=True evaluates the variant that rounds h to bf16.
  * Gate weights come from the unbiased scores; for softmax_topk they are the softmax of the
    selected logits; the renormalising denominator is clamped to >= 1e-30.
  * Group membership is contiguous: group g holds experts [g*E/G, (g+1)*E/G).
  * Shared experts are added with weight 1 after the routed sum.
  * Bias update: "overloaded" / "underloaded" are relative to the mean load T*k/E (compared
    exactly in integers); an expert exactly at the mean keeps its bias; the bias is fp32 and
    the update is one fp32 addition (the kernel's precision).
"""
from __future__ import annotations

import numpy as np

SCORES = ("softmax_topk", "softmax", "sigmoid", "sqrt_softplus")
DENOM_MIN = 1e-30


# ----------------------------------------------------------------------------- scoring

def router_logits(x, w_r):
    """l[t, e] = sum_i x[t, i] * W_r[e, i], fp64.  W_r is [E, d] (MoEGate weight
    [n_routed_experts, hidden_size]); page 4's x W_g is the same map with W_g = W_r^T."""
    return np.asarray(x, np.float64) @ np.asarray(w_r, np.float64).T


def sigmoid(l):
    """1 / (1 + e^-l)  (DeepSeek-V3 affinity)."""
    l = np.asarray(l, np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-l))


def softplus(l):
    """ln(1 + e^l), evaluated as max(l, 0) + ln(1 + e^-|l|) so that it neither overflows
    nor loses the small-argument tail."""
    l = np.asarray(l, np.float64)
    return np.maximum(l, 0.0) + np.log1p(np.exp(-np.abs(l)))


def sqrt_softplus(l):
    """sqrt(Softplus(l))  (DeepSeek-V4 affinity, eq. dsv4-moe-softplus)."""
    return np.sqrt(softplus(l))


def softmax(l, axis=-1):
    """e^l / sum e^l over `axis`, max-subtracted."""
    l = np.asarray(l, np.float64)
    m = l.max(axis=axis, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=axis, keepdims=True)


def affinity(logits, score):
    """Unbiased per-expert score s[t, e] for each scoring mode (None for softmax_topk,
    whose selection is on raw logits)."""
    if score == "softmax_topk":
        return None
    if score == "softmax":
        return softmax(logits, axis=1)
    if score == "sigmoid":
        return sigmoid(logits)
    if score == "sqrt_softplus":
        return sqrt_softplus(logits)
    raise ValueError(f"unknown score mode {score!r}")


# ----------------------------------------------------------------------------- selection

def _topk_desc(keys, k):
    """Indices of the k largest keys per row, descending; equal keys -> lower index first (a
    stable sort of the negated keys)."""
    order = np.argsort(-keys, axis=1, kind="stable")
    return order[:, :k]


def selection_keys(logits, score, bias=None):
    """Key q[t, e] that top-k ranks: the raw logit for softmax_topk, else the unbiased score
    plus the selection bias (0 when None).  "MoE compute and communication", section 七.3:
    the bias shifts the choice only."""
    logits = np.asarray(logits, np.float64)
    s = affinity(logits, score)
    base = logits if s is None else s
    return base + (0.0 if bias is None else np.asarray(bias, np.float64)[None, :])


def group_scores(keys, n_groups, group_topk):
    """Score of each contiguous group of E / n_groups experts: the sum of its group_topk
    largest keys, added largest first ("DeepSeek-V4 MoE", section "V3 的节点路由约束")."""
    keys = np.asarray(keys, np.float64)
    T, E = keys.shape
    top = -np.sort(-keys.reshape(T, n_groups, E // n_groups), axis=2)[:, :, :group_topk]
    acc = top[..., 0].copy()
    for j in range(1, group_topk):
        acc = acc + top[..., j]
    return acc


def gate_weights(logits, ids, score):
    """Gate weights of the selected experts ids [T, k]: the softmax of the k selected logits
    (softmax_topk), else the unbiased scores of the selected experts renormalised to sum 1
    (denominator clamped to DENOM_MIN).  For "softmax" the score is the softmax over all E, so
    this is its renormalisation over the k."""
    logits = np.asarray(logits, np.float64)
    ids = np.asarray(ids, np.int64)
    rows = np.arange(logits.shape[0])[:, None]
    s = affinity(logits, score)
    if s is None:
        return softmax(logits[rows, ids], axis=1)
    sel = s[rows, ids]
    return sel / np.maximum(sel.sum(axis=1, keepdims=True), DENOM_MIN)


def route(logits, k, score, bias=None, n_groups=0, topk_groups=0, group_topk=0,
          token_ids=None, tid2eid=None, return_order_margin=False):
    """Top-k routing.  Returns (topk_ids [T,k] int32, topk_w [T,k] fp64, margin [T] fp64)
    and, with return_order_margin, also order_margin [T] fp64.

    margin[t] is the gap between the k-th and (k+1)-th selection key (and, when groups are
    used, between the last kept and the first dropped group score), the smallest one that
    decides WHICH experts are selected; order_margin[t] is the smallest gap between two
    consecutive selected keys, which decides the ORDER they are listed in.  Both are +inf
    when nothing is decided by a comparison (hash routing, E=k, k=1).
    """
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    order_margin = np.full(T, np.inf)
    margin = np.full(T, np.inf)
    if tid2eid is not None:
        # HashTopK: ids looked up by token id, in table order; no comparison decides them.
        ids = np.asarray(tid2eid)[np.asarray(token_ids, np.int64)].astype(np.int32)
    else:
        key = selection_keys(logits, score, bias)
        if n_groups:
            gsize = E // n_groups
            gscore = group_scores(key, n_groups, group_topk)                # [T, G]
            gorder = np.argsort(-gscore, axis=1, kind="stable")
            keep = gorder[:, :topk_groups]
            if topk_groups < n_groups:
                gs_sorted = np.take_along_axis(gscore, gorder, axis=1)
                margin = np.minimum(margin, gs_sorted[:, topk_groups - 1] - gs_sorted[:, topk_groups])
            group_mask = np.zeros((T, n_groups), bool)
            np.put_along_axis(group_mask, keep, True, axis=1)
            expert_mask = np.repeat(group_mask, gsize, axis=1)
            key = np.where(expert_mask, key, -np.inf)
        ids = _topk_desc(key, k).astype(np.int32)
        sel_keys = np.take_along_axis(key, ids.astype(np.int64), axis=1)
        if k > 1:
            order_margin = np.min(sel_keys[:, :-1] - sel_keys[:, 1:], axis=1)
        if k < E:
            ks = -np.sort(-key, axis=1)
            kth, nxt = ks[:, k - 1], ks[:, k]
            gap = np.where(np.isfinite(nxt), kth - nxt, np.inf)
            margin = np.minimum(margin, gap)
    w = gate_weights(logits, ids, score)
    if return_order_margin:
        return ids, w, margin, order_margin
    return ids, w, margin


# ----------------------------------------------------------------------------- dispatch

def permute(topk_ids, E):
    """Token dispatch: token-major assignments -> expert-major rows.

    Assignment i = t*k + j (token t, slot j).  Rows are ordered by expert, and inside an
    expert by i ascending (a stable sort by expert id).  Returns
      counts [E]      tokens_per_expert
      offsets [E+1]   exclusive prefix sum of counts
      perm_tok [N]    token of each row (permuted_token_ids)
      inv [N]         row of each assignment i
    """
    ids = np.asarray(topk_ids, np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")
    perm_tok = (order // k).astype(np.int32)
    inv = np.empty(T * k, np.int32)
    inv[order] = np.arange(T * k, dtype=np.int32)
    return counts, offsets, perm_tok, inv


# ----------------------------------------------------------------------------- experts

def round_to_bf16(v):
    """Round fp64 values to the nearest bf16 value (8 significant bits), ties to even.
    Normal range only (|v| >= 2^-126); zeros and non-finite values pass through."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def silu(g):
    """SiLU(g) = g * sigmoid(g) = g / (1 + e^-g)."""
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_expert(xr, w13, w2, cast_h=False):
    """FFN(x) = W2 (SiLU(W1 x) * (W3 x)) for the rows of xr [m, d].

    w13 is [2f, d]: rows 0..f-1 are W1 (gate), rows f..2f-1 are W3 (up); w2 is [d, f]."""
    xr = np.asarray(xr, np.float64)
    w13 = np.asarray(w13, np.float64)
    w2 = np.asarray(w2, np.float64)
    f = w13.shape[0] // 2
    g = xr @ w13[:f].T
    u = xr @ w13[f:].T
    h = silu(g) * u
    if cast_h:
        h = round_to_bf16(h)
    return h @ w2.T


def forward(x, topk_ids, topk_w, expert_weights, shared_weights=None, tokens=None, cast_h=False):
    """Layer output y[t] = sum_j topk_w[t,j] * FFN_{topk_ids[t,j]}(x[t]) + FFN_shared(x[t]).

    expert_weights(e) -> (w13_e [2f, d], w2_e [d, f]); shared_weights: (w13_sh, w2_sh) or
    None.  Only the rows in `tokens` (default: all) are computed; returns [len(tokens), d].
    Experts are visited one at a time (the page's loop reference layer), each on the
    tokens that chose it; the weighted sum then runs over slots j in order."""
    x = np.asarray(x, np.float64)
    ids = np.asarray(topk_ids, np.int64)
    wts = np.asarray(topk_w, np.float64)
    tokens = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, np.int64)
    ids_s, w_s, x_s = ids[tokens], wts[tokens], x[tokens]
    n, k = ids_s.shape
    d = x.shape[1]
    o = np.zeros((n, k, d), np.float64)
    for e in np.unique(ids_s):
        rows, slots = np.nonzero(ids_s == e)
        w13_e, w2_e = expert_weights(int(e))
        o[rows, slots] = swiglu_expert(x_s[rows], w13_e, w2_e, cast_h)
    y = np.zeros((n, d), np.float64)
    for j in range(k):
        y += w_s[:, j:j + 1] * o[:, j]
    if shared_weights is not None:
        y += swiglu_expert(x_s, shared_weights[0], shared_weights[1], cast_h)
    return y


# ----------------------------------------------------------------------------- balancing

def bias_update(counts, bias, total_assignments, gamma=0.001):
    """Aux-loss-free bias step: b_e - gamma if expert e received more than the mean load,
    b_e + gamma if fewer, unchanged at the mean.  counts [E] int, bias [E] fp32; returns the
    new fp32 bias (one fp32 addition per expert)."""
    counts = np.asarray(counts, np.int64)
    E = counts.shape[0]
    b = np.asarray(bias, np.float32)
    excess = counts * E - int(total_assignments)          # sign of count - T*k/E, exactly
    step = np.where(excess > 0, -gamma, np.where(excess < 0, gamma, 0.0)).astype(np.float32)
    return (b + step).astype(np.float32)
