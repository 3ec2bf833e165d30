"""moe_permute_noalloc: the dispatch permutation for callers that cannot allocate device
memory, such as a plugin inside a host framework that owns all device memory through its own
allocator, or a latency-critical loop where cudaMalloc (which can synchronise the device) is
not allowed.  It must give exactly the oracle's dispatch (integer results, so bit for bit), and
what moe_permute gives, on consecutive calls that share the library's fixed scratch array; at
the array's limit (131072 assignments over 512 experts plus a shared expert, the case its fixed
offsets are sized for) and at a decode-sized batch; refuse batches larger than the array
covers; and report an out-of-range expert id through moe_permute_noalloc_status."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from routed_expert_swiglu_gb300 import binding, build, inputs, workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load()


def _outputs(T, E, k):
    z = lambda n: torch.full((n,), -1, dtype=torch.int32, device=DEV)  # noqa: E731
    return z(E), z(E + 1), z(T * k), z(T * k)


def _layer(E, k, n_shared, max_tokens):
    w = dataclasses.replace(W.V4FLASH_T64, T=1, E=E, k=k, n_shared=n_shared, d=128, d_ff=128)
    return binding.MoELayer(w, inputs.make_layer_inputs(w, device=DEV), max_tokens=max_tokens)


def _check_against_oracle_and_workspace_path(layer, T, E, k, ids):
    got = _outputs(T, E, k)
    binding.moe_permute_noalloc(layer.plan, T, ids, *got)
    assert binding.moe_permute_noalloc_status() == binding.MOE_OK
    ref = oracle.permute(ids.cpu().numpy(), E)
    for a, b in zip(got, ref):
        assert np.array_equal(a.cpu().numpy(), b)
    for a, b in zip(got, layer.permute(ids)):
        assert torch.equal(a, b)


def test_noalloc_permute_matches_oracle_on_consecutive_calls():
    E, k = 384, 6
    layer = _layer(E, k, 0, 22000)
    # a large skewed batch, then a smaller one: the second call starts from the first one's
    # leftovers in the shared scratch array
    for T, skew, seed in ((4099, 0.0, 1), (777, 3.0, 2), (64, 0.0, 4)):
        ids = inputs.random_topk_ids(T, E, k, seed=seed, device=DEV, skew=skew)
        _check_against_oracle_and_workspace_path(layer, T, E, k, ids)
    # beyond the fixed scratch: 22000 * 6 = 132000 > 131072 assignments
    big = inputs.random_topk_ids(22000, E, k, seed=3, device=DEV)
    with pytest.raises(binding.MoEError) as ei:
        binding.moe_permute_noalloc(layer.plan, 22000, big, *_outputs(22000, E, k))
    assert ei.value.status == 2  # MOE_ERR_UNSUPPORTED
    layer.close()


def test_noalloc_permute_at_the_scratch_limit():
    """Exactly 131072 assignments (16384 tokens x top-8) over 512 experts with a shared expert:
    the most per-chunk histograms, groups and row tiles the fixed array holds."""
    E, k, T = 512, 8, 16384
    layer = _layer(E, k, 1, T)
    for seed, skew in ((5, 0.0), (6, 2.0)):
        ids = inputs.random_topk_ids(T, E, k, seed=seed, device=DEV, skew=skew)
        _check_against_oracle_and_workspace_path(layer, T, E, k, ids)
    layer.close()


def test_noalloc_permute_reports_out_of_range_ids():
    """An id equal to E is clamped to E - 1 (as moe_permute does) and flagged; the next clean
    call clears the flag."""
    E, k, T = 64, 4, 100
    layer = _layer(E, k, 0, T)
    ids = inputs.random_topk_ids(T, E, k, seed=8, device=DEV)
    bad = ids.clone()
    bad[3, 1] = E
    got = _outputs(T, E, k)
    binding.moe_permute_noalloc(layer.plan, T, bad, *got)
    assert binding.moe_permute_noalloc_status() == 6  # MOE_ERR_DEVICE_INPUT
    clamped = bad.clamp(max=E - 1)
    ref = oracle.permute(clamped.cpu().numpy(), E)
    for a, b in zip(got, ref):
        assert np.array_equal(a.cpu().numpy(), b)
    _check_against_oracle_and_workspace_path(layer, T, E, k, ids)
    layer.close()
