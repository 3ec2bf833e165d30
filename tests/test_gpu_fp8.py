"""FP8 (E4M3) expert weights on the GPU, through the C ABI, against the oracle: the quantiser's
codes and tile exponents bit for bit (partial tiles, an all-zero tile, magnitudes over many
binades), and the layer with FP8 weights against the oracle's layer on its own dequantised
weights (the oracle quantises the bf16 weights itself), at decode and prefill batch sizes.
Shapes with d and d_ff multiples of 128 run the codes straight into the tensor cores (16-, 32-
and 64-row tiles all appear below); the others (toy, ragged) run the widening kernels."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_weights as F
from routed_expert_swiglu_gb300 import binding, inputs, workloads as W

from parity_util import check_output, check_routing, oracle_routing, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_swiglu_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("shape", [(3, 256, 384), (2, 200, 192), (1, 64, 4096), (5, 128, 64)])
def test_quantiser_bit_exact(shape):
    g = torch.Generator().manual_seed(sum(shape))
    w = torch.randn(shape, generator=g) * torch.exp(torch.randn(shape[:-1] + (1,), generator=g) * 3)
    w = w.to(torch.bfloat16)
    if shape[1] > 128 and shape[2] > 128:
        w[0, 128:, :128] = 0                                    # an all-zero tile
    codes, exps = binding.quantize_fp8(w.to(DEV))
    torch.cuda.synchronize()
    rc, re = F.quantize_fp8_tiles(w.double().numpy())
    assert np.array_equal(exps.cpu().numpy().astype(np.int64), re)
    assert np.array_equal(codes.cpu().numpy(), rc)


class OracleFp8Fetcher:
    """Expert weights as the oracle's own FP8 round trip of the bf16 weights (per expert, lazily)."""

    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    @staticmethod
    def _rt(w):
        codes, exps = F.quantize_fp8_tiles(to64(w))
        return F.dequantize_fp8_tiles(codes, exps)

    def __call__(self, e):
        if e not in self.cache:
            self.cache[e] = (self._rt(self.inp.w13[e]), self._rt(self.inp.w2[e]))
        return self.cache[e]

    def shared(self):
        if self.inp.w13_sh is None:
            return None
        return self._rt(self.inp.w13_sh), self._rt(self.inp.w2_sh)


def small(w, T, **kw):
    return dataclasses.replace(w, T=T, name=f"{w.name.rsplit('_T', 1)[0]}_T{T}", **kw)


# Batches that route more than 48 rows to an expert on average run the block-scaled CTA-pair
# kernels (codes and tile scales into the 2-SM MMA, E4M3-piece activations; d, d_ff multiples of
# 128: v3_E32_T400, tall_T1500 with two 224-row tiles per expert) or, for other shapes, the
# CTA-pair kernels that widen the codes to bf16 in shared memory (toy_T333, ragged_T400); smaller
# ones (up to 64 tokens, or at most 48 rows per expert: ragged_T150, v3_T96, edges_T80) stream the
# weights through the single-CTA kernels: the direct 8-bit MMA (d, d_ff multiples of 128) or, for
# other shapes, the single-CTA widening kernels.
CASES = [
    W.TOY,                                                                  # single-CTA kernels
    small(W.TOY, 333),                                                      # CTA-pair widening
    W.Workload("mid_T64", T=64, d=512, d_ff=256, E=16, k=4, n_shared=1, score=W.SCORE_SIGMOID, use_bias=True),
    W.Workload("ragged_T150", T=150, d=320, d_ff=192, E=12, k=3, n_shared=1, score=W.SCORE_SOFTMAX),
    W.Workload("ragged_T400", T=400, d=320, d_ff=192, E=12, k=3, n_shared=1, score=W.SCORE_SOFTMAX),
    small(W.V3_T4096, 400, E=32, n_groups=8, topk_groups=4, group_topk=2, d=1024, d_ff=256),
    # decode with d, d_ff not multiples of 128: single-CTA widening kernels
    W.Workload("ragged_T48", T=48, d=320, d_ff=192, E=12, k=3, n_shared=1, score=W.SCORE_SOFTMAX),
    # decode with 64-row direct-MMA tiles (T k > 24 E)
    W.Workload("deep_T64", T=64, d=256, d_ff=256, E=16, k=8, n_shared=0, score=W.SCORE_SOFTMAX),
    small(W.V3_T4096, 96, E=32, n_groups=8, topk_groups=4, group_topk=2, d=1024, d_ff=256),
    small(W.V4FLASH_T64, 64, E=16),                                         # V4-Flash dims, 16 experts
    small(W.V4PRO_HASH_T16384, 40, E=24, d=1024, d_ff=384),
    # direct-MMA path with 16-row tiles (2 mean rows per expert; the shared expert's 64 rows span
    # four tiles), and a prefill batch with two 224-row tiles per expert (the second ragged)
    W.Workload("wide_T64", T=64, d=512, d_ff=256, E=64, k=2, n_shared=1, score=W.SCORE_SQRT_SOFTPLUS,
               use_bias=True),
    W.Workload("tall_T1500", T=1500, d=256, d_ff=256, E=8, k=2, n_shared=1, score=W.SCORE_SOFTMAX),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_layer_vs_oracle(w):
    inp = inputs.make_layer_inputs(w, seed=21, device=DEV)
    layer = binding.MoELayer(w, inp)
    q = layer.quantize_fp8()
    y = layer.forward_fp8(inp.x, q, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    same = np.ones(w.T, bool)  # every token: the oracle is fed the GPU's ids
    fetch = OracleFp8Fetcher(inp)
    tok = np.nonzero(same)[0]
    ref = oracle.forward(to64(inp.x), gids, ref_w, fetch, fetch.shared(), tokens=tok)
    e, n = check_output(y.double().cpu().numpy()[tok], ref, label=w.name)
    print(f"{w.name} (fp8 weights): max elementwise {e:.2e}, normwise {n:.2e}")
    layer.close()


@pytest.mark.parametrize("T", [80, 300])  # 30 rows per expert: single-CTA kernels; 112.5: CTA pairs
def test_fp8_layer_with_zero_subnormal_and_tiny_scale_codes(T):
    """Weights with exact zeros, values that quantise to subnormal codes, and one expert scaled
    down to a tile exponent below -120: every code class of the converter, against the oracle."""
    w = W.Workload(f"edges_T{T}", T=T, d=256, d_ff=128, E=8, k=3, n_shared=1, score=W.SCORE_SOFTMAX)
    inp = inputs.make_layer_inputs(w, seed=23, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    for t in (inp.w13, inp.w2, inp.w13_sh, inp.w2_sh):
        u = torch.rand(t.shape, generator=g, device=DEV)
        t[u < 0.05] = 0
        tiny = (u >= 0.05) & (u < 0.10)
        t[tiny] = (t[tiny].float() * 2.0 ** -14).to(torch.bfloat16)
    inp.w2[2] = (inp.w2[2].float() * 1e-36).to(torch.bfloat16)
    inp.w13[5] = (inp.w13[5].float() * 1e-36).to(torch.bfloat16)
    layer = binding.MoELayer(w, inp)
    q = layer.quantize_fp8()
    e2 = q["w2"][1].cpu().numpy()
    assert e2[2].max() < -120 and (q["w13"][0].cpu().numpy() & 0x78 == 0).any()
    y = layer.forward_fp8(inp.x, q, None)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    same = np.ones(w.T, bool)  # every token: the oracle is fed the GPU's ids
    fetch = OracleFp8Fetcher(inp)
    tok = np.nonzero(same)[0]
    ref = oracle.forward(to64(inp.x), gids, ref_w, fetch, fetch.shared(), tokens=tok)
    check_output(y.double().cpu().numpy()[tok], ref, label=w.name)
    layer.close()


def test_fp8_layer_with_wide_activation_range():
    """Activation rows whose entries span 2^-20 .. 2^6 of their typical size (the E4M3 pieces
    share one power-of-two scale per row, so small entries sit near the pieces' subnormal
    floor), plus a row scaled by 2^-60, an all-zero row and a row with one entry 2^10 larger
    than the rest: the FP8 layer against the oracle on the same inputs."""
    w = W.Workload("range_T48", T=48, d=512, d_ff=256, E=8, k=2, n_shared=1, score=W.SCORE_SOFTMAX)
    inp = inputs.make_layer_inputs(w, seed=29, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(7)
    expo = torch.randint(-20, 7, inp.x.shape, generator=g, device=DEV).float()
    inp.x.copy_((inp.x.float() * torch.exp2(expo)).to(torch.bfloat16))
    inp.x[3] = (inp.x[3].float() * 2.0 ** -60).to(torch.bfloat16)
    inp.x[5] = 0
    inp.x[7, 11] = (inp.x[7, 11].float() * 2.0 ** 10).to(torch.bfloat16)
    layer = binding.MoELayer(w, inp)
    q = layer.quantize_fp8()
    y = layer.forward_fp8(inp.x, q, None)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    same = np.ones(w.T, bool)  # every token: the oracle is fed the GPU's ids
    fetch = OracleFp8Fetcher(inp)
    tok = np.nonzero(same)[0]
    ref = oracle.forward(to64(inp.x), gids, ref_w, fetch, fetch.shared(), tokens=tok)
    got = y.double().cpu().numpy()[tok]
    e, n = check_output(got, ref, label=w.name)
    print(f"{w.name} (fp8 weights): max elementwise {e:.2e}, normwise {n:.2e}")
    if 5 in tok:
        assert np.array_equal(got[list(tok).index(5)], ref[list(tok).index(5)])  # zero row: exactly 0
    layer.close()


# Full sizes, in the launch configuration bench.py times for FP8 weights (its decode and prefill legs):
# routing against the oracle on every token, the output on a few sampled tokens (the oracle
# quantises and dequantises every expert those tokens touch, a few seconds each).
FULL_FP8 = [(W.V4FLASH_T64, 4), (W.MIXTRAL_T16, 2), (W.V4FLASH_T8192, 32)]


@pytest.mark.slow
@pytest.mark.parametrize("w,sample", FULL_FP8, ids=lambda v: getattr(v, "name", str(v)))
def test_fp8_full_size_layer(w, sample):
    inp = inputs.make_layer_inputs(w, seed=0, device=DEV)
    layer = binding.MoELayer(w, inp)
    q = layer.quantize_fp8()
    y = layer.forward_fp8(inp.x, q, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    same = np.ones(w.T, bool)  # every token: the oracle is fed the GPU's ids
    rng = np.random.default_rng(4321)
    cand = np.nonzero(same)[0]
    tok = np.sort(rng.choice(cand, size=min(sample, cand.size), replace=False))
    fetch = OracleFp8Fetcher(inp)
    ref = oracle.forward(to64(inp.x), gids, ref_w, fetch, fetch.shared(), tokens=tok)
    e, n = check_output(y.double().cpu().numpy()[tok], ref, label=w.name)
    print(f"{w.name} full size (fp8 weights), sample of {tok.size}: max elementwise {e:.2e}, normwise {n:.2e}")
    layer.close()
    del layer, inp, y, v, q
    torch.cuda.empty_cache()
