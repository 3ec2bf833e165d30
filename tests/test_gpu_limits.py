"""Library limits and degenerate layers on the GPU, through the C ABI, against the oracle:
the largest expert count, top-k and group count the library accepts; hidden and intermediate
sizes that are not multiples of 128 (partial weight slabs in both projections); the first
batch size that takes the prefill kernels; a one-expert (dense SwiGLU) layer; a layer in which
every token takes every expert; and exact routing ties, whose outcome the tie rule fixes."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from routed_expert_swiglu_gb300 import binding, inputs, workloads as W

from parity_util import (ExpertFetcher, check_output, check_routing, oracle_output, oracle_route,
                         oracle_routing, to64)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_swiglu_gb300 import build
    build.build()
    binding.load()


# E = 512 experts (the library's maximum), k = 8 (maximum), 32 groups of 16 (maximum group
# count), group score from the 4 largest keys, 8 groups kept; sigmoid affinity with bias.
LIMITS = W.Workload("limits_T300", T=300, d=256, d_ff=128, E=512, k=8, n_shared=1, score=W.SCORE_SIGMOID,
                    use_bias=True, n_groups=32, topk_groups=8, group_topk=4)
# d = 320 and d_ff = 192: the last 128-row weight slab of both projections is partial.
RAGGED = W.Workload("ragged_T517", T=517, d=320, d_ff=192, E=24, k=3, n_shared=1, score=W.SCORE_SOFTMAX)
# One expert, top-1: the layer is a dense SwiGLU FFN with gate weight exactly 1.
DENSE = W.Workload("dense_T200", T=200, d=256, d_ff=256, E=1, k=1, n_shared=0, score=W.SCORE_SOFTMAX_TOPK)
# Every token takes every expert.
ALL = W.Workload("all_T130", T=130, d=256, d_ff=128, E=8, k=8, n_shared=1, score=W.SCORE_SQRT_SOFTPLUS)

CASES = [LIMITS, LIMITS.with_T(50), RAGGED, RAGGED.with_T(65), RAGGED.with_T(37), DENSE, DENSE.with_T(64), ALL,
         ALL.with_T(64)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_layer_at_the_limits(w):
    inp = inputs.make_layer_inputs(w, seed=7, device=DEV)
    layer = binding.MoELayer(w, inp)
    y = layer.forward(inp.x, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    gw = v["topk_w"].cpu().numpy()
    ref_w, moved = check_routing(w, gids, gw, oracle_routing(w, inp))
    if w.E == w.k:
        # every expert selected: the set is forced whatever the keys
        assert moved == 0
    if w.E == 1:
        assert (gids == 0).all() and (gw == 1.0).all()
    assert moved <= 0.2 * w.T
    e, n = check_output(y.double().cpu().numpy(), oracle_output(inp, gids, ref_w), label=w.name)
    print(f"{w.name}: max elementwise {e:.2e}, normwise {n:.2e}")
    layer.close()


TIE_CASES = [
    W.Workload("tie_softmax_topk_T70", T=70, d=128, d_ff=64, E=8, k=2, n_shared=0, score=W.SCORE_SOFTMAX_TOPK),
    W.Workload("tie_softmax_T70", T=70, d=128, d_ff=64, E=16, k=4, n_shared=0, score=W.SCORE_SOFTMAX),
    W.Workload("tie_sigmoid_groups_T300", T=300, d=256, d_ff=128, E=64, k=6, n_shared=1, score=W.SCORE_SIGMOID,
               n_groups=8, topk_groups=2, group_topk=2),
    W.Workload("tie_sqrt_softplus_T40", T=40, d=256, d_ff=128, E=384, k=6, n_shared=1,
               score=W.SCORE_SQRT_SOFTPLUS),
]


@pytest.mark.parametrize("w", TIE_CASES, ids=lambda w: w.name)
def test_exact_ties_follow_the_tie_rule(w):
    """Zero router weights make every key equal.  Equal keys go to the lower expert id (and
    equal groups to the lower group id), so every token must select experts 0..k-1 in that
    order with weight 1/k, on the oracle and on the GPU alike."""
    inp = inputs.make_layer_inputs(w, seed=8, device=DEV)
    inp.w_r.zero_()
    layer = binding.MoELayer(w, inp)
    ids, wts = layer.route(inp.x)
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    expect = np.tile(np.arange(w.k, dtype=np.int32), (w.T, 1))
    _, rids, rw, _ = oracle_route(w, inp)
    assert (rids == expect).all()
    np.testing.assert_allclose(rw, 1.0 / w.k, rtol=0, atol=1e-12)
    assert (ids.cpu().numpy() == expect).all()
    np.testing.assert_allclose(wts.cpu().numpy(), 1.0 / w.k, rtol=0, atol=1e-6)
    layer.close()


def test_large_batch():
    """131072 tokens through the toy layer (262144 assignments: 256 dispatch chunks, the
    token-major row copy, thousands of row tiles): dispatch invariants on the whole batch, the
    output against the oracle on a sample of tokens."""
    w = dataclasses.replace(W.TOY, T=131072, name="toy_T131072")
    inp = inputs.make_layer_inputs(w, seed=9, device=DEV)
    layer = binding.MoELayer(w, inp)
    y = layer.forward(inp.x, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    ids = v["topk_ids"].cpu().numpy()
    counts = v["counts"].cpu().numpy()
    offsets = v["offsets"].cpu().numpy()
    perm = v["perm_tok"].cpu().numpy()
    inv = v["inv"].cpu().numpy()
    assert (counts == np.bincount(ids.ravel(), minlength=w.E)).all()
    assert offsets[0] == 0 and (np.diff(offsets) == counts).all() and offsets[-1] == w.T * w.k
    assert (perm[inv] == np.arange(w.T * w.k) // w.k).all()                # inverse map
    assert (np.sort(inv) == np.arange(w.T * w.k)).all()                    # every row used once
    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(w.T, 512, replace=False))
    ref_w, _ = check_routing(w, ids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    check_output(y.double().cpu().numpy()[tok], oracle_output(inp, ids, ref_w, tokens=tok), label=w.name)
    layer.close()
