"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

Routing is compared with the oracle on every token (margin rule, see parity_util); the
layer output on a seeded sample of tokens the oracle evaluates one by one; the dispatch
permutation through properties that hold at any size (it is compared bit for bit with the
oracle on generated ids in test_gpu_parity)."""
import gc

import numpy as np
import pytest
import torch

import oracle
from routed_expert_swiglu_gb300 import binding, inputs, workloads as W

from parity_util import ExpertFetcher, check_output, check_routing, oracle_route, to64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda:0"
SAMPLE = 24

FULL = [W.MIXTRAL_T2048, W.V3_T4096, W.V4FLASH_T64_ZIPF, W.V4FLASH_T8192, W.V4FLASH_T8192_ZIPF,
        W.V4PRO_HASH_T16384, W.V4PRO_LEARNED_T16384]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_swiglu_gb300 import build
    build.build()
    binding.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def check_permutation(w, ids, counts, offsets, perm, inv):
    """Dispatch invariants on the GPU's own routing: counts = histogram of ids, offsets their
    exclusive scan, every assignment in exactly one row of its expert, rows of an expert in
    ascending assignment order, permuted token ids = token of each row."""
    T, k, E = w.T, w.k, w.E
    flat = ids.reshape(-1).astype(np.int64)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(inv), np.arange(T * k))
    assert np.array_equal(perm[inv], np.arange(T * k) // k)
    rows_expert = np.repeat(np.arange(E), counts)
    assert np.array_equal(rows_expert[inv], flat)
    order = np.empty(T * k, np.int64)
    order[inv] = np.arange(T * k)
    for e in np.nonzero(counts)[0][:64]:
        seg = order[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size_layer(w):
    inp = inputs.make_layer_inputs(w, seed=0, device=DEV)
    layer = binding.MoELayer(w, inp)
    y = layer.forward(inp.x, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    check_permutation(w, gids, v["counts"].cpu().numpy(), v["offsets"].cpu().numpy(),
                      v["perm_tok"].cpu().numpy(), v["inv"].cpu().numpy())
    _, rids, rw, margin, omargin = oracle_route(w, inp, with_order=True)
    same = check_routing(w, gids, v["topk_w"].cpu().numpy(), rids, rw, margin, omargin)
    rng = np.random.default_rng(1234)
    cand = np.nonzero(same)[0]
    tok = np.sort(rng.choice(cand, size=min(SAMPLE, cand.size), replace=False))
    fetch = ExpertFetcher(inp)
    x_s = to64(inp.x[torch.from_numpy(tok).to(DEV)])
    ref = oracle.forward(x_s, rids[tok], rw[tok], fetch, fetch.shared())
    e, n = check_output(y[torch.from_numpy(tok).to(DEV)].double().cpu().numpy(), ref, label=w.name)
    print(f"{w.name}: {int((~same).sum())} near-tie tokens routed differently; sample of {tok.size}: "
          f"max elementwise {e:.2e}, normwise {n:.2e}")
    layer.close()
    del layer, inp, y, v
    gc.collect()
    torch.cuda.empty_cache()


def test_full_size_permute_bit_exact():
    """moe_permute at the largest batch (V4-Pro: 16384 tokens x top-6 over 384 experts)."""
    w = W.V4PRO_LEARNED_T16384
    ids = inputs.random_topk_ids(w.T, w.E, w.k, seed=7, device=DEV, skew=1.0)
    small = inputs.make_layer_inputs(W.TOY, device=DEV)
    import dataclasses
    layer = binding.MoELayer(dataclasses.replace(w, d=128, d_ff=128), small, max_tokens=w.T)
    counts, offsets, perm, inv = layer.permute(ids)
    rc, ro, rp, ri = oracle.permute(ids.cpu().numpy(), w.E)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp) and np.array_equal(inv.cpu().numpy(), ri)
    layer.close()
