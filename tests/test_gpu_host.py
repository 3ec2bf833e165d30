"""The host-buffer entry point (moe_forward_host) on the GPU: consecutive calls enqueued
without synchronisation (their input copies run on the plan's side stream and alternate
between two staging slots; page-locked outputs are written by the combine directly, pageable
ones through a staged copy), interleaved with a device-buffer call of another batch size on
the same workspace and stream, must each return exactly the device-path result for their
input."""
import dataclasses

import pytest
import torch

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


HASH_SMALL = dataclasses.replace(W.V4PRO_HASH_T16384, d=1024, d_ff=512, E=64, name="hash_small_T16384")


@pytest.mark.parametrize("base", [W.V4FLASH_T64, HASH_SMALL], ids=lambda w: w.name)
def test_host_calls_match_device_calls(base):
    T = 300
    w = dataclasses.replace(base, T=T, name=f"{base.name.rsplit('_T', 1)[0]}_T{T}")
    inp = inputs.make_layer_inputs(w, seed=11, device=DEV)
    layer = binding.MoELayer(w, inp)
    sizes = [T, 300, 64, 277, 300]          # prefill, prefill, decode, ragged prefill, prefill
    xs = [inputs.make_layer_inputs(w, seed=20 + i, device=DEV, T=n).x for i, n in enumerate(sizes)]
    toks = [None if inp.token_ids is None else
            torch.randint(0, w.hash_vocab, (n,), generator=torch.Generator().manual_seed(i), dtype=torch.int32)
            for i, n in enumerate(sizes)]
    # device-path results, one call at a time
    ref = []
    for x, tk in zip(xs, toks):
        y = layer.forward(x, None if tk is None else tk.to(DEV)).clone()
        torch.cuda.synchronize()
        ref.append(y.cpu())
    other_x = inputs.make_layer_inputs(w, seed=40, device=DEV, T=100).x
    other_tok = None if inp.token_ids is None else inp.token_ids[:100].contiguous()
    other_ref = layer.forward(other_x, other_tok).clone().cpu()
    torch.cuda.synchronize()
    # host-buffer calls back to back, with a device call of another size in between
    # page-locked buffers (the result is written into them directly), except call 3, whose
    # pageable buffers take the staged-copy path
    pin = lambda t, i: t if i == 3 else t.pin_memory()
    xh = [pin(x.cpu(), i) for i, x in enumerate(xs)]
    th = [None if tk is None else pin(tk, i) for i, tk in enumerate(toks)]
    yh = [pin(torch.empty((n, w.d), dtype=torch.bfloat16), i) for i, n in enumerate(sizes)]
    assert not yh[3].is_pinned() and yh[0].is_pinned()
    stream = torch.cuda.current_stream()
    other_out = torch.empty((100, w.d), dtype=torch.bfloat16, device=DEV)
    for i, n in enumerate(sizes):
        binding.moe_forward_host(layer.plan, n, xh[i], th[i], inp.w_r, inp.bias, inp.w13, inp.w2, inp.w13_sh,
                                 inp.w2_sh, yh[i], layer.ws, stream)
        if i == 1:
            binding.moe_forward(layer.plan, 100, other_x, other_tok, inp.w_r, inp.bias, inp.w13, inp.w2,
                                inp.w13_sh, inp.w2_sh, other_out, layer.ws, stream)
    torch.cuda.synchronize()
    other_host = other_out.cpu()
    assert layer.check_status() == 0
    for i in range(len(sizes)):
        assert torch.equal(yh[i].view(torch.int16), ref[i].view(torch.int16)), f"call {i} (T={sizes[i]})"
    assert torch.equal(other_host.view(torch.int16), other_ref.view(torch.int16))
    layer.close()
