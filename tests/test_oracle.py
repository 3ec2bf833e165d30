"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a worked example the
pages print (tests/golden/*.json, each citing its page and section), a closed form, a
library routine, an invariant, or brute force on tiny inputs.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# ----------------------------------------------------------------------------- router

def test_router_worked_example_softmax_after_topk():
    g = golden("router_worked_example.json")
    logits = np.array([g["scores"]])
    ids, w, margin = oracle.route(logits, g["k"], "softmax_topk")
    assert ids[0].tolist() == g["expected_ids"]
    np.testing.assert_allclose(w[0], g["printed_weights"], atol=g["printed_precision"])
    # closed form: a 2-way softmax is the logistic function of the logit difference
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-(2.1 - 1.2))), rel=1e-14)
    assert w[0, 0] == pytest.approx(0.7109495, abs=1e-7)
    assert margin[0] == pytest.approx(1.2 - 0.8, abs=1e-6)


def test_router_worked_example_softmax_before_topk_is_identical():
    """Softmax over all E, top-k, renormalise == top-k, softmax over the selected k."""
    g = golden("router_worked_example.json")
    ids, w, _ = oracle.route(np.array([g["scores"]]), g["k"], "softmax")
    assert ids[0].tolist() == g["expected_ids"]
    assert w[0, 0] == pytest.approx(0.7109495, abs=1e-7)
    rng = np.random.default_rng(0)
    logits = rng.normal(size=(200, 16)) * 2
    ia, wa, _ = oracle.route(logits, 4, "softmax_topk")
    ib, wb, _ = oracle.route(logits, 4, "softmax")
    assert (ia == ib).all()
    np.testing.assert_allclose(wa, wb, rtol=1e-12)


def test_router_logits_brute_force_loop():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(3, 5))
    w_r = rng.normal(size=(4, 5))
    l = oracle.router_logits(x, w_r)
    for t in range(3):
        for e in range(4):
            assert l[t, e] == pytest.approx(sum(x[t, i] * w_r[e, i] for i in range(5)), rel=1e-13)


def test_score_functions_against_library():
    l = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(oracle.sigmoid(l), scipy.special.expit(l), rtol=1e-14)
    np.testing.assert_allclose(oracle.softplus(l), np.logaddexp(0.0, l), rtol=1e-14)
    m = np.random.default_rng(2).normal(size=(7, 11)) * 5
    np.testing.assert_allclose(oracle.softmax(m, axis=1), scipy.special.softmax(m, axis=1), rtol=1e-13)


def test_sqrt_softplus_closed_forms():
    """'DeepSeek-V4 MoE', eq. dsv4-moe-softplus and the range/derivative notes after it."""
    assert oracle.sqrt_softplus(0.0) == pytest.approx(math.sqrt(math.log(2.0)), rel=1e-15)
    assert oracle.sqrt_softplus(0.0) == pytest.approx(0.8325546, abs=1e-7)
    grid = np.linspace(-40, 40, 8001)
    s = oracle.sqrt_softplus(grid)
    assert (s >= 0).all() and (np.diff(s) > 0).all()          # range [0, inf), monotone
    for big in (50.0, 200.0, 1e4):                              # grows like sqrt(x)
        assert oracle.sqrt_softplus(big) == pytest.approx(math.sqrt(big), rel=1e-12)
    # derivative sigmoid(x) / (2 sqrt(softplus(x))), by central differences
    xs = np.linspace(-8, 8, 33)
    h = 1e-5
    fd = (oracle.sqrt_softplus(xs + h) - oracle.sqrt_softplus(xs - h)) / (2 * h)
    np.testing.assert_allclose(fd, scipy.special.expit(xs) / (2 * oracle.sqrt_softplus(xs)), rtol=1e-7)


@pytest.mark.parametrize("score", oracle.SCORES)
def test_gate_weights_sum_to_one(score):
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(300, 32)) * 1.5
    bias = rng.normal(size=32) * 0.01
    _, w, _ = oracle.route(logits, 6, score, bias=bias)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert (w >= 0).all()


def test_bias_selects_but_does_not_weight():
    """'MoE compute and communication', section 七.3: TopK(s + b) chooses, g = s/sum(s)."""
    logits = np.array([[2.0, 1.0, 0.0, -1.0]])
    bias = np.array([-1.0, 0.0, 0.0, 0.0])
    ids, w, _ = oracle.route(logits, 2, "sigmoid", bias=bias)
    assert ids[0].tolist() == [1, 2]
    s1, s2 = 1 / (1 + math.exp(-1.0)), 0.5
    np.testing.assert_allclose(w[0], [s1 / (s1 + s2), s2 / (s1 + s2)], rtol=1e-14)
    ids0, _, _ = oracle.route(logits, 2, "sigmoid")
    assert ids0[0].tolist() == [0, 1]


def test_order_margin_is_the_smallest_gap_between_selected_keys():
    g = golden("router_worked_example.json")
    _, _, margin, om = oracle.route(np.array([g["scores"]]), 2, "softmax_topk", return_order_margin=True)
    assert om[0] == pytest.approx(2.1 - 1.2, abs=1e-6) and margin[0] == pytest.approx(0.4, abs=1e-6)
    ids, _, margin, om = oracle.route(np.array([[3.0, 2.0, 2.0005, 0.0]]), 3, "softmax_topk",
                                      return_order_margin=True)
    assert ids[0].tolist() == [0, 2, 1]
    assert om[0] == pytest.approx(0.0005, abs=1e-6) and margin[0] == pytest.approx(2.0, abs=1e-6)
    _, _, _, om = oracle.route(np.array([[1.0, 0.0]]), 1, "softmax_topk", return_order_margin=True)
    assert np.isinf(om[0])


def test_topk_ties_go_to_lower_id_and_order_is_descending():
    ids, _, margin = oracle.route(np.array([[1.0, 2.0, 2.0, 0.0, 2.0]]), 2, "softmax_topk")
    assert ids[0].tolist() == [1, 2] and margin[0] == 0.0
    ids, _, _ = oracle.route(np.array([[0.5, 3.0, -1.0, 1.0]]), 3, "softmax_topk")
    assert ids[0].tolist() == [1, 3, 0]


# ----------------------------------------------------------------------------- groups

def test_group_limited_single_group_equals_plain_topk():
    rng = np.random.default_rng(4)
    logits = rng.normal(size=(100, 64))
    bias = rng.normal(size=64) * 0.01
    a, wa, _ = oracle.route(logits, 8, "sigmoid", bias=bias)
    for G in (1, 8):  # keep all groups -> no restriction
        b, wb, _ = oracle.route(logits, 8, "sigmoid", bias=bias, n_groups=G, topk_groups=G, group_topk=2)
        assert (a == b).all()
        np.testing.assert_allclose(wa, wb, rtol=0)


def test_group_score_is_sum_of_top2_not_max():
    # group 0: one strong expert; group 1: two good experts.  Sum of top-2 prefers group 1.
    logits = np.array([[4.0, -4.0, 1.5, 1.4]])
    ids, _, _ = oracle.route(logits, 2, "sigmoid", n_groups=2, topk_groups=1, group_topk=2)
    assert ids[0].tolist() == [2, 3]


def test_group_limited_brute_force_tiny():
    """Against exhaustive search: the kept groups are the M-subset with the largest total
    group score, and the chosen experts are the k-subset of their experts with the largest
    total key (both unique on continuous random data)."""
    rng = np.random.default_rng(5)
    E, G, M, k, gt = 12, 4, 2, 3, 2
    gsz = E // G
    for trial in range(200):
        logits = rng.normal(size=(1, E))
        bias = rng.normal(size=E) * 0.3
        ids, _, _ = oracle.route(logits, k, "sigmoid", bias=bias, n_groups=G, topk_groups=M, group_topk=gt)
        key = scipy.special.expit(logits[0]) + bias
        gscore = [sum(sorted(key[g * gsz:(g + 1) * gsz])[-gt:]) for g in range(G)]
        best_groups = max(itertools.combinations(range(G), M), key=lambda S: sum(gscore[g] for g in S))
        cand = [e for g in best_groups for e in range(g * gsz, (g + 1) * gsz)]
        best = max(itertools.combinations(cand, k), key=lambda S: sum(key[e] for e in S))
        assert set(ids[0].tolist()) == set(best)
        assert list(ids[0]) == sorted(ids[0], key=lambda e: -key[e])


def test_group_limited_invariants_v3_shape():
    rng = np.random.default_rng(6)
    T, E, G, M, k = 64, 256, 8, 4, 8
    logits = rng.normal(size=(T, E)) * 1.3
    bias = rng.normal(size=E) * 0.01
    ids, w, margin = oracle.route(logits, k, "sigmoid", bias=bias, n_groups=G, topk_groups=M, group_topk=2)
    key = oracle.sigmoid(logits) + bias
    for t in range(T):
        groups = set(int(e) // (E // G) for e in ids[t])
        assert len(groups) <= M                         # spans at most M groups
        assert len(set(ids[t].tolist())) == k
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)
    assert (margin >= 0).all()


# ----------------------------------------------------------------------------- hash

def test_hash_routing_uses_table_order_and_unbiased_scores():
    rng = np.random.default_rng(7)
    V, E, k, T = 50, 16, 3, 20
    tid2eid = np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int32)
    token_ids = rng.integers(0, V, size=T)
    logits = rng.normal(size=(T, E))
    ids, w, margin = oracle.route(logits, k, "sqrt_softplus", bias=rng.normal(size=E),
                                  token_ids=token_ids, tid2eid=tid2eid)
    for t in range(T):
        assert ids[t].tolist() == tid2eid[token_ids[t]].tolist()
        s = [math.sqrt(math.log1p(math.exp(logits[t, e]))) for e in ids[t]]
        np.testing.assert_allclose(w[t], np.array(s) / sum(s), rtol=1e-13)
    assert np.isinf(margin).all()


# ----------------------------------------------------------------------------- dispatch

def test_dispatch_worked_example():
    g = golden("dispatch_worked_example.json")
    ids = np.array(g["topk_ids"])
    counts, offsets, perm_tok, inv = oracle.permute(ids, g["E"])
    assert perm_tok.tolist() == g["expected_permuted_token_ids"]
    assert counts.tolist() == g["expected_tokens_per_expert"]
    assert offsets.tolist() == [0, 3, 5, 8]
    wts = np.array(g["topk_w"])
    k = ids.shape[1]
    pos = [None] * len(inv)
    for i, r in enumerate(inv):
        pos[r] = [int(i // k), float(wts[i // k, i % k])]
    assert pos == g["expected_combine_positions"]


def test_ep_routing_example_counts_and_dispatch_matrix():
    g = golden("ep_routing_example.json")
    ids = np.array(g["topk_ids"])
    counts, _, perm_tok, inv = oracle.permute(ids, g["E"])
    assert counts.tolist() == g["expected_tokens_per_expert"]
    R = g["ranks"]
    mat = np.zeros((R, R), int)
    for t in range(ids.shape[0]):
        for e in ids[t]:
            mat[t // 2, e // 2] += 1
    assert mat.tolist() == g["expected_dispatch_matrix"]
    assert mat.sum(0).tolist() == g["expected_received"]


def test_two_token_example_round_trip():
    g = golden("two_token_example.json")
    ids = np.array(g["topk_ids"])
    counts, offsets, perm_tok, inv = oracle.permute(ids, g["E"])
    assert counts.tolist() == g["expected_tokens_per_expert"]
    for e, names in g["expected_rows_per_expert"].items():
        e = int(e)
        rows = perm_tok[offsets[e]:offsets[e + 1]]
        assert [g["tokens"][t] for t in rows] == names
    # inverse permutation then permutation is the identity on assignments
    k = ids.shape[1]
    for i in range(ids.size):
        assert perm_tok[inv[i]] == i // k


def test_permute_brute_force_and_invariants():
    rng = np.random.default_rng(8)
    for (T, E, k) in [(1, 1, 1), (7, 5, 2), (33, 8, 3), (300, 64, 6)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        counts, offsets, perm_tok, inv = oracle.permute(ids, E)
        flat = ids.reshape(-1)
        rows = [i for e in range(E) for i in range(T * k) if flat[i] == e]   # brute force
        assert perm_tok.tolist() == [i // k for i in rows]
        assert sorted(inv.tolist()) == list(range(T * k))
        assert counts.sum() == T * k and offsets[-1] == T * k
        for i in range(T * k):
            r = inv[i]
            assert offsets[flat[i]] <= r < offsets[flat[i] + 1]


# ----------------------------------------------------------------------------- experts

def test_round_to_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(9)
    v = np.concatenate([rng.normal(size=20000), rng.normal(size=2000) * 1e-20, rng.normal(size=2000) * 1e20])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_to_bf16(v32.astype(np.float64)), ref)
    # halfway cases round to even
    assert oracle.round_to_bf16(1.0 + 2.0 ** -8) == 1.0
    assert oracle.round_to_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert oracle.round_to_bf16(0.0) == 0.0


def _torch_swiglu(x, w13, w2):
    """Textbook SwiGLU with torch fp64 ops: W_down(SiLU(W_gate x) * W_up x)."""
    f = w13.shape[0] // 2
    x, w13, w2 = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, w13, w2))
    return (torch.nn.functional.silu(x @ w13[:f].T) * (x @ w13[f:].T) @ w2.T).numpy()


def test_single_expert_equals_dense_swiglu():
    rng = np.random.default_rng(10)
    T, d, f = 9, 16, 12
    x = rng.normal(size=(T, d))
    w13 = rng.normal(size=(1, 2 * f, d)) / 4
    w2 = rng.normal(size=(1, d, f)) / 4
    ids = np.zeros((T, 1), np.int32)
    wts = np.ones((T, 1))
    y = oracle.forward(x, ids, wts, lambda e: (w13[e], w2[e]), cast_h=False)
    np.testing.assert_allclose(y, _torch_swiglu(x, w13[0], w2[0]), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("cast_h", [False, True])
def test_identical_experts_make_routing_irrelevant(cast_h):
    rng = np.random.default_rng(11)
    T, d, f, E, k = 10, 16, 8, 6, 3
    x = rng.normal(size=(T, d))
    w13 = rng.normal(size=(2 * f, d)) / 4
    w2 = rng.normal(size=(d, f)) / 4
    w13s, w2s = rng.normal(size=(2 * f, d)) / 4, rng.normal(size=(d, f)) / 4
    logits = rng.normal(size=(T, E))
    ids, wts, _ = oracle.route(logits, k, "sqrt_softplus")
    y = oracle.forward(x, ids, wts, lambda e: (w13, w2), (w13s, w2s), cast_h=cast_h)
    ref = oracle.swiglu_expert(x, w13, w2, cast_h) + oracle.swiglu_expert(x, w13s, w2s, cast_h)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_layer_equals_dense_all_experts_masked():
    """Brute force: run every expert on every token and mask by the gate weights
    (no dispatch, no permute)."""
    rng = np.random.default_rng(12)
    T, d, f, E, k = 8, 32, 16, 6, 2
    x = rng.normal(size=(T, d))
    w_r = rng.normal(size=(E, d)) / 5
    w13 = rng.normal(size=(E, 2 * f, d)) / 5
    w2 = rng.normal(size=(E, d, f)) / 5
    w13s, w2s = rng.normal(size=(2 * f, d)) / 5, rng.normal(size=(d, f)) / 5
    bias = rng.normal(size=E) * 0.05
    ids, wts, _ = oracle.route(oracle.router_logits(x, w_r), k, "sqrt_softplus", bias=bias)
    gate = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            gate[t, ids[t, j]] += wts[t, j]
    dense = sum(gate[:, e:e + 1] * _torch_swiglu(x, w13[e], w2[e]) for e in range(E))
    dense = dense + _torch_swiglu(x, w13s, w2s)
    y = oracle.forward(x, ids, wts, lambda e: (w13[e], w2[e]), (w13s, w2s), cast_h=False)
    np.testing.assert_allclose(y, dense, rtol=1e-11, atol=1e-12)
    sub = oracle.forward(x, ids, wts, lambda e: (w13[e], w2[e]), (w13s, w2s), tokens=[5, 2], cast_h=False)
    np.testing.assert_allclose(sub, dense[[5, 2]], rtol=1e-11, atol=1e-12)


def test_cast_h_is_bf16_of_the_activation():
    rng = np.random.default_rng(13)
    d, f = 8, 4
    x = rng.normal(size=(3, d))
    w13 = rng.normal(size=(2 * f, d))
    w2 = np.eye(d)[:, :f] if d >= f else None
    h = oracle.silu(x @ w13[:f].T) * (x @ w13[f:].T)
    out = oracle.swiglu_expert(x, w13, w2, cast_h=True)   # w2 picks h out unchanged
    np.testing.assert_array_equal(out[:, :f], oracle.round_to_bf16(h))
    assert not np.array_equal(out[:, :f], h)


# ----------------------------------------------------------------------------- cost model

def test_cost_model_matches_printed_tables():
    from routed_expert_swiglu_gb300 import cost
    g = golden("cost_model.json")
    for row in g["ffn_params"]:
        assert cost.expert_params(row["d"], row["d_ff"]) / 1e6 == pytest.approx(row["params_M"], abs=0.05)
        if "flops_per_token_M" in row:
            assert cost.ffn_flops_per_token(row["d"], row["d_ff"]) / 1e6 == pytest.approx(
                row["flops_per_token_M"], abs=0.6)
    for name, tab in g["expected_active_experts"].items():
        for B, v in zip(tab["B"], tab["value"]):
            assert cost.expected_active_experts(tab["E"], tab["k"], B) == pytest.approx(v, abs=g["printed_precision"])


# ----------------------------------------------------------------------------- balancing

def test_bias_update_direction_and_step():
    """'MoE compute and communication' 七.3: overloaded b - gamma, underloaded b + gamma, 0.001."""
    counts = np.array([5, 1, 2, 0])            # T*k = 8 over E = 4: mean load 2
    bias = np.array([0.5, -0.25, 0.125, 0.0], np.float32)
    new = oracle.bias_update(counts, bias, total_assignments=8)
    assert new.dtype == np.float32
    assert new[0] == np.float32(0.5) - np.float32(0.001)     # overloaded
    assert new[1] == np.float32(-0.25) + np.float32(0.001)   # underloaded
    assert new[2] == np.float32(0.125)                       # exactly at the mean
    assert new[3] == np.float32(0.001)


def test_bias_update_moves_selection_towards_balance():
    """Repeated steps on a skewed router reduce the load spread (the loop the pages describe)."""
    rng = np.random.default_rng(21)
    T, E, k = 512, 16, 2
    logits = rng.normal(size=(T, E)) + np.linspace(1.0, -1.0, E)   # hot low-id experts
    bias = np.zeros(E, np.float32)
    spread0 = None
    for step in range(300):
        ids, _, _ = oracle.route(logits, k, "sigmoid", bias=bias)
        counts = np.bincount(ids.reshape(-1), minlength=E)
        if spread0 is None:
            spread0 = counts.max() - counts.min()
        bias = oracle.bias_update(counts, bias, T * k, gamma=0.01)
    assert counts.max() - counts.min() < spread0 / 2


# ----------------------------------------------------------------------------- selection helpers

def test_gate_weights_of_given_ids_on_the_worked_example():
    """Router page, "Router 的选择过程": experts {3, 0} of the printed scores get 0.7109 / 0.2891
    whichever order they are listed in, and in softmax-over-all mode the same after renormalising."""
    g = golden("router_worked_example.json")
    logits = np.array([g["scores"]])
    p3 = 1.0 / (1.0 + math.exp(-(2.1 - 1.2)))
    for mode in ("softmax_topk", "softmax"):
        w = oracle.gate_weights(logits, np.array([[3, 0]]), mode)
        np.testing.assert_allclose(w[0], g["printed_weights"], atol=g["printed_precision"])
        np.testing.assert_allclose(w[0], [p3, 1.0 - p3], rtol=1e-13)
        w_rev = oracle.gate_weights(logits, np.array([[0, 3]]), mode)
        np.testing.assert_allclose(w_rev[0], [1.0 - p3, p3], rtol=1e-13)


def test_group_scores_brute_force():
    """Sum of the group_topk largest keys of each contiguous group, against a loop over groups."""
    rng = np.random.default_rng(11)
    keys = rng.normal(size=(5, 24))
    for G, gt in ((4, 2), (3, 3), (8, 1)):
        got = oracle.group_scores(keys, G, gt)
        gsz = 24 // G
        for t in range(5):
            for g in range(G):
                assert got[t, g] == pytest.approx(sum(sorted(keys[t, g * gsz:(g + 1) * gsz])[-gt:]), abs=1e-12)


def test_selection_keys_add_the_bias_to_the_unbiased_score():
    rng = np.random.default_rng(12)
    logits, bias = rng.normal(size=(3, 6)), rng.normal(size=6)
    np.testing.assert_array_equal(oracle.selection_keys(logits, "softmax_topk"), logits)
    np.testing.assert_allclose(oracle.selection_keys(logits, "sigmoid", bias),
                               scipy.special.expit(logits) + bias, rtol=1e-15)


def test_a_single_bf16_activation_misses_the_output_tolerance():
    """Why the down projection carries h as a (hi, lo) pair of bf16 values: on a V4-Flash-shaped
    layer (d=4096, d_ff=2048, one shared expert), rounding h once to bf16 between the two
    projections ("MoE compute and communication", sec. 二.1: FFN = W2(SiLU(W1 x) * W3 x), no such
    rounding) moves outputs near zero far beyond max|err| / (|y| + 1e-2) <= 2e-2, while the exact
    h with only the bf16 rounding of y meets it."""
    import dataclasses
    from routed_expert_swiglu_gb300 import inputs, workloads as W
    w = dataclasses.replace(W.V4FLASH_T8192, T=64, E=8, name="v4flash_E8_T64")
    inp = inputs.make_layer_inputs(w, seed=0, device="cpu")
    f64 = lambda t: t.double().numpy()  # noqa: E731
    x = f64(inp.x)
    ids, wts, _ = oracle.route(oracle.router_logits(x, f64(inp.w_r)), w.k, w.score, bias=f64(inp.bias))
    fetch = lambda e: (f64(inp.w13[e]), f64(inp.w2[e]))  # noqa: E731
    sh = (f64(inp.w13_sh), f64(inp.w2_sh))
    ref = oracle.forward(x, ids, wts, fetch, sh)
    elem = lambda y: (np.abs(y - ref) / (np.abs(ref) + 1e-2)).max()  # noqa: E731
    assert elem(oracle.round_to_bf16(oracle.forward(x, ids, wts, fetch, sh, cast_h=True))) > 0.1
    assert elem(oracle.round_to_bf16(ref)) < 5e-3


def test_bf16_expert_outputs_miss_the_output_tolerance():
    """Why the down projection writes its weighted expert outputs O in fp32: on the same
    V4-Flash-shaped layer, rounding each weighted expert output to bf16 before the slot sum (the
    pages' combine, "Mixture of Experts: router, token dispatch, grouped GEMM", Token Combine, sums
    them unrounded) moves outputs where the slots cancel far beyond the 2e-2 bound, while fp32 O
    (exact here) with only the bf16 rounding of y meets it."""
    import dataclasses
    from oracle import moe_oracle as M
    from routed_expert_swiglu_gb300 import inputs, workloads as W
    w = dataclasses.replace(W.V4FLASH_T8192, T=64, E=8, name="v4flash_E8_T64")
    inp = inputs.make_layer_inputs(w, seed=0, device="cpu")
    f64 = lambda t: t.double().numpy()  # noqa: E731
    x = f64(inp.x)
    ids, wts, _ = oracle.route(oracle.router_logits(x, f64(inp.w_r)), w.k, w.score, bias=f64(inp.bias))
    fetch = lambda e: (f64(inp.w13[e]), f64(inp.w2[e]))  # noqa: E731
    sh = (f64(inp.w13_sh), f64(inp.w2_sh))
    ref = oracle.forward(x, ids, wts, fetch, sh)
    y = oracle.round_to_bf16(M.swiglu_expert(x, sh[0], sh[1], False))
    for j in range(w.k):
        for e in np.unique(ids[:, j]):
            r = np.nonzero(ids[:, j] == e)[0]
            y[r] += oracle.round_to_bf16(M.swiglu_expert(x[r], *fetch(int(e)), False) * wts[r, j:j + 1])
    elem = lambda v: (np.abs(v - ref) / (np.abs(ref) + 1e-2)).max()  # noqa: E731
    assert elem(oracle.round_to_bf16(y)) > 0.1
    assert elem(oracle.round_to_bf16(ref)) < 5e-3
