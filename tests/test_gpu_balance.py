"""GPU: the aux-loss-free selection-bias step (moe_update_bias) against the oracle, and the
closed balancing loop on a Zipf-skewed router."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from routed_expert_swiglu_gb300 import binding, inputs, workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_swiglu_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("T,skew", [(8192, 0.0), (777, 3.0), (1, 0.0)])
def test_bias_update_bit_exact(T, skew):
    w = dataclasses.replace(W.V4FLASH_T64, T=T, d=128, d_ff=128)
    inp = inputs.make_layer_inputs(dataclasses.replace(w, T=1), seed=2, device=DEV)
    layer = binding.MoELayer(w, inp, max_tokens=T)
    ids = inputs.random_topk_ids(T, w.E, w.k, seed=T, device=DEV, skew=skew)
    counts = torch.bincount(ids.reshape(-1).long(), minlength=w.E).to(torch.int32)
    bias = (torch.randn(w.E, device=DEV) * 0.01).float()
    ref = oracle.bias_update(counts.cpu().numpy(), bias.cpu().numpy(), T * w.k, gamma=0.001)
    binding.moe_update_bias(layer.plan, T, counts, bias, 0.001)
    torch.cuda.synchronize()
    assert np.array_equal(bias.cpu().numpy().view(np.int32), ref.view(np.int32))
    layer.close()


def test_balancing_loop_reduces_load_spread():
    """forward -> counts -> bias step, repeated: the hottest expert's load falls."""
    w = dataclasses.replace(W.V4FLASH_T8192_ZIPF, T=2048, d=512, d_ff=128, name="zipf_small")
    inp = inputs.make_layer_inputs(w, seed=4, device=DEV)
    layer = binding.MoELayer(w, inp)
    first = None
    for _ in range(40):
        layer.forward(inp.x)
        counts = layer.views(w.T)["counts"].clone()
        if first is None:
            first = counts.cpu().numpy()
        binding.moe_update_bias(layer.plan, w.T, counts, inp.bias, 0.02)
    last = counts.cpu().numpy()
    assert last.max() < first.max()
    assert np.std(last) < np.std(first)
    layer.close()
