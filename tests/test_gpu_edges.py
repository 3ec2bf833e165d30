"""Edge cases and error behaviour through the C ABI on the GPU."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from routed_expert_swiglu_gb300 import binding, inputs, workloads as W

from parity_util import ExpertFetcher, check_output, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_swiglu_gb300 import build
    build.build()
    binding.load()


def test_zero_tokens_is_a_no_op():
    w = W.TOY
    inp = inputs.make_layer_inputs(w, device=DEV)
    layer = binding.MoELayer(w, inp)
    out = torch.full((1, w.d), 7.0, dtype=torch.bfloat16, device=DEV)
    binding.moe_forward(layer.plan, 0, inp.x, None, inp.w_r, None, inp.w13, inp.w2, None, None, out, layer.ws)
    torch.cuda.synchronize()
    assert (out.float() == 7.0).all()
    layer.close()


@pytest.mark.parametrize("T", [1000, 40])
def test_all_tokens_on_the_same_experts(T):
    """Maximum skew: every token picks experts 0..5 -> groups of T rows (several row tiles,
    ragged last tile), every other expert empty."""
    w = dataclasses.replace(W.V4FLASH_T64, T=T, E=16, name=f"skew_T{T}")
    inp = inputs.make_layer_inputs(w, seed=5, device=DEV)
    ids = torch.tensor([[0, 1, 2, 3, 4, 5]], dtype=torch.int32, device=DEV).repeat(T, 1)
    wts = torch.rand((T, w.k), device=DEV)
    wts = wts / wts.sum(1, keepdim=True)
    layer = binding.MoELayer(w, inp)
    y = layer.forward_routed(inp.x, ids, wts)
    assert layer.check_status() == 0
    fetch = ExpertFetcher(inp)
    ref = oracle.forward(to64(inp.x), ids.cpu().numpy(), wts.double().cpu().numpy(), fetch, fetch.shared())
    check_output(y.double().cpu().numpy(), ref, label=f"skew T={T}")
    layer.close()


def test_bad_topk_ids_are_clamped_and_reported():
    E, k, T = 8, 2, 100
    w = dataclasses.replace(W.TOY, T=T)
    inp = inputs.make_layer_inputs(w, device=DEV)
    layer = binding.MoELayer(w, inp)
    ids = inputs.random_topk_ids(T, E, k, seed=3, device=DEV)
    ids[5, 0] = -3
    ids[17, 1] = E + 4
    counts, offsets, perm, inv = layer.permute(ids)
    assert layer.check_status() == 6  # MOE_ERR_DEVICE_INPUT
    clamped = np.clip(ids.cpu().numpy(), 0, E - 1)
    rc, ro, rp, ri = oracle.permute(clamped, E)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(inv.cpu().numpy(), ri)
    # the next clean call clears the status word
    layer.permute(inputs.random_topk_ids(T, E, k, seed=4, device=DEV))
    assert layer.check_status() == 0
    layer.close()


def test_bad_token_ids_in_hash_routing_are_reported():
    w = dataclasses.replace(W.V4PRO_HASH_T16384, T=32, d=128, d_ff=128, name="hash_small")
    inp = inputs.make_layer_inputs(w, device=DEV)
    inp.token_ids[3] = w.hash_vocab + 10
    layer = binding.MoELayer(w, inp)
    ids, wts = layer.route(inp.x, inp.token_ids)
    assert layer.check_status() == 6
    tid = inp.tid2eid.cpu().numpy()
    assert ids[3].cpu().tolist() == tid[w.hash_vocab - 1].tolist()   # clamped to the last row
    layer.close()


def test_batch_invariance_within_a_kernel_family():
    """A token's output does not depend on which other tokens share the batch (prefill path:
    no split-K, fixed reduction order)."""
    w = dataclasses.replace(W.V4FLASH_T8192, T=300, name="bi_T300")
    inp = inputs.make_layer_inputs(w, seed=9, device=DEV)
    layer = binding.MoELayer(w, inp)
    y_full = layer.forward(inp.x).clone()
    y_part = layer.forward(inp.x[:200].contiguous()).clone()
    torch.cuda.synchronize()
    assert torch.equal(y_full[:200].view(torch.int16), y_part.view(torch.int16))
    layer.close()
