"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on seeded inputs."""
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
    torch.set_num_threads(max(1, (torch.get_num_threads())))


def small(w, T, **kw):
    return dataclasses.replace(w, T=T, name=f"{w.name.rsplit('_T', 1)[0]}_T{T}", **kw)


ROUTE_CASES = [
    W.TOY,
    small(W.TOY, 333),
    W.MIXTRAL_T16,
    small(W.V3_T4096, 300),
    small(W.V3_T4096, 300, zipf_s=0.0),
    small(W.V3_T4096, 48, E=64),  # the fused small-batch router: 28 K slices, groups, sigmoid, bias
    W.V4FLASH_T64,
    small(W.V4FLASH_T8192, 1000),
    small(W.V4FLASH_T8192_ZIPF, 500),
    small(W.V4PRO_HASH_T16384, 200),
    small(W.V4PRO_LEARNED_T16384, 200),
]


@pytest.mark.parametrize("w", ROUTE_CASES, ids=lambda w: w.name)
def test_router_logits_and_routing(w):
    inp = inputs.make_layer_inputs(w, seed=0, device=DEV)
    layer = binding.MoELayer(w, inp)
    ids, wts, logits = layer.route(inp.x, inp.token_ids, with_logits=True)
    assert layer.check_status() == 0
    R = oracle_routing(w, inp)
    # fp32 accumulation of d bf16 products: error bounded by a few ulps of sum |x_i w_i|
    bound = np.abs(to64(inp.x)) @ np.abs(to64(inp.w_r)).T
    err = np.abs(logits.double().cpu().numpy() - R.logits)
    assert (err <= 1e-5 * bound + 1e-6).all(), f"logit error {(err / (bound + 1e-6)).max():.3e} of sum|xw|"
    _, moved = check_routing(w, ids.cpu().numpy(), wts.cpu().numpy(), R)
    print(f"{w.name}: {moved} tokens inside the margin routed differently; "
          f"{int((R.margin <= 1e-3).sum())} tokens within margin")
    layer.close()


PERMUTE_CASES = [(1, 1, 1, 0.0), (5, 8, 2, 0.0), (64, 8, 2, 0.0), (1000, 256, 6, 0.0), (777, 256, 8, 3.0),
                 (4099, 384, 6, 0.0), (2048, 8, 2, 0.0), (300, 256, 6, 50.0),
                 # one chunk of assignments (the single-block path) at its limit with the most experts,
                 # and just past it
                 (128, 512, 8, 3.0), (171, 64, 6, 0.0)]


@pytest.mark.parametrize("T,E,k,skew", PERMUTE_CASES)
def test_permute_bit_exact(T, E, k, skew):
    w = dataclasses.replace(W.V4FLASH_T64, T=T, E=E, k=k, d=128, d_ff=128)
    ids = inputs.random_topk_ids(T, E, k, seed=T + E, device=DEV, skew=skew)
    inp = inputs.make_layer_inputs(dataclasses.replace(w, T=1), device=DEV)
    layer = binding.MoELayer(w, inp, max_tokens=T)
    counts, offsets, perm, inv = layer.permute(ids)
    assert layer.check_status() == 0
    rc, ro, rp, ri = oracle.permute(ids.cpu().numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)
    layer.close()


def test_permute_worked_example():
    """Router page, section 'Token Dispatch': 4 tokens, 3 experts, top-2."""
    w = dataclasses.replace(W.TOY, T=4, E=3, k=2)
    ids = torch.tensor([[0, 2], [1, 2], [0, 1], [0, 2]], dtype=torch.int32, device=DEV)
    inp = inputs.make_layer_inputs(dataclasses.replace(w, T=1), device=DEV)
    layer = binding.MoELayer(w, inp, max_tokens=4)
    counts, offsets, perm, inv = layer.permute(ids)
    assert perm.cpu().tolist() == [0, 2, 3, 1, 2, 0, 1, 3]
    assert counts.cpu().tolist() == [3, 2, 3]
    layer.close()


FORWARD_CASES = [
    W.TOY,
    small(W.TOY, 333),
    small(W.TOY, 1),
    W.MIXTRAL_T16,
    W.V4FLASH_T64,
    small(W.V4FLASH_T8192, 300),
    small(W.V3_T4096, 200),
    small(W.V4PRO_HASH_T16384, 48),
    # more than 48 routed rows per expert on average: the CTA-pair kernels at the layers' own
    # dims, with partly filled and ragged token tiles (the cases above stream the weights)
    dataclasses.replace(W.V4FLASH_T8192, T=300, E=16, name="v4flash_E16_T300"),
    dataclasses.replace(W.V3_T4096, T=300, E=24, name="v3_E24_T300"),
]


@pytest.mark.parametrize("w", FORWARD_CASES, ids=lambda w: w.name)
def test_forward_routed_vs_oracle(w):
    """Dispatch + grouped GEMMs + combine with routing fixed by the oracle."""
    inp = inputs.make_layer_inputs(w, seed=1, device=DEV)
    _, rids, rw, _ = oracle_route(w, inp)
    layer = binding.MoELayer(w, inp)
    ids_d = torch.from_numpy(rids).to(DEV)
    w_d = torch.from_numpy(rw.astype(np.float32)).to(DEV)
    y = layer.forward_routed(inp.x, ids_d, w_d)
    assert layer.check_status() == 0
    fetch = ExpertFetcher(inp)
    ref = oracle.forward(to64(inp.x), rids, rw.astype(np.float32).astype(np.float64), fetch, fetch.shared())
    e, n = check_output(y.double().cpu().numpy(), ref, label=w.name)
    print(f"{w.name}: max elementwise {e:.2e}, normwise {n:.2e}")
    layer.close()


@pytest.mark.parametrize("w", [W.TOY, W.V4FLASH_T64, small(W.V4FLASH_T8192, 300)], ids=lambda w: w.name)
def test_forward_vs_oracle(w):
    inp = inputs.make_layer_inputs(w, seed=2, device=DEV)
    layer = binding.MoELayer(w, inp)
    y = layer.forward(inp.x, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    check_output(y.double().cpu().numpy(), oracle_output(inp, gids, ref_w), label=w.name)
    layer.close()


def test_forward_deterministic():
    w = small(W.V4FLASH_T8192, 300)
    inp = inputs.make_layer_inputs(w, seed=3, device=DEV)
    layer = binding.MoELayer(w, inp)
    y1 = layer.forward(inp.x).clone()
    y2 = layer.forward(inp.x).clone()
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    layer.close()
