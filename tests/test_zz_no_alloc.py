"""moe_permute_noalloc: the dispatch permutation for callers that cannot allocate device
memory, such as a plugin inside a host framework that owns all device memory through its own
allocator, or a latency-critical loop where cudaMalloc (which can synchronise the device) is
not allowed.  It must give exactly what moe_permute gives (integer results, so bit for bit)
on consecutive calls that share the library's fixed scratch array, and refuse batches larger
than that array covers."""
import dataclasses

import pytest
import torch

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


def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    E, k = 384, 6
    w = dataclasses.replace(W.V4FLASH_T64, T=1, E=E, k=k, d=128, d_ff=128)
    inp = inputs.make_layer_inputs(w, device=DEV)
    layer = binding.MoELayer(w, inp, max_tokens=22000)
    # a large skewed batch, then a smaller one: the second call starts from the first one's
    # leftovers in the shared scratch array
    for T, skew, seed in ((4099, 0.0, 1), (777, 3.0, 2)):
        ids = inputs.random_topk_ids(T, E, k, seed=seed, device=DEV, skew=skew)
        ref = layer.permute(ids)
        got = _outputs(T, E, k)
        binding.moe_permute_noalloc(layer.plan, T, ids, *got)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    # beyond the fixed scratch: 22000 * 6 = 132000 > 131072 assignments
    big = inputs.random_topk_ids(22000, E, k, seed=3, device=DEV)
    with pytest.raises(binding.MoEError) as ei:
        binding.moe_permute_noalloc(layer.plan, 22000, big, *_outputs(22000, E, k))
    assert ei.value.status == 2  # MOE_ERR_UNSUPPORTED
    layer.close()
