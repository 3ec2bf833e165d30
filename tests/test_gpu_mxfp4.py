"""MXFP4 (E2M1, 1 x 32 sub-block scales) expert weights on the GPU, through the C ABI, against
the oracle: the quantiser's codes and sub-block exponents bit for bit (partial tiles, zero
sub-blocks and tiles, sub-block ranges wide enough to trigger the headroom raise), the lossless
conversion to FP8 tiles bit for bit on the oracle's own codes, and the layer run on the
converted weights against the oracle's layer on its own MXFP4 round trip of the weights."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_weights as F8
from oracle import mxfp4_weights as M
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


def pack(codes):
    """The library's storage of E2M1 codes: two per byte, code 2i of a row in the low nibble of
    byte i (the order in which the block-scaled MMA reads packed E2M1)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def weights(shape, seed):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(shape, generator=g)
    # per-sub-block magnitudes over ~24 binades, so that some tiles span more than the headroom
    blk = torch.randint(-18, 6, shape[:-1] + (shape[-1] // 32, 1), generator=g).float()
    return (w * torch.exp2(blk).repeat_interleave(32, dim=-1).reshape(shape)).to(torch.bfloat16)


@pytest.mark.parametrize("shape", [(3, 256, 384), (2, 200, 192), (1, 64, 4096), (4, 128, 96)])
def test_quantiser_bit_exact(shape):
    w = weights(shape, sum(shape))
    if shape[1] > 128 and shape[2] > 128:
        w[0, 128:, :128] = 0                                     # an all-zero tile
    w[-1, 3, 32:64] = 0                                          # an all-zero sub-block
    codes, exps = binding.quantize_mxfp4(w.to(DEV))
    torch.cuda.synchronize()
    rc, re = M.quantize_mxfp4(w.double().numpy())
    assert np.array_equal(exps.cpu().numpy().astype(np.int64), re)
    assert np.array_equal(codes.cpu().numpy(), pack(rc))
    assert (re.max() - re.min()) > M.HEADROOM                     # the raise was exercised


@pytest.mark.parametrize("shape", [(3, 256, 384), (2, 200, 192)])
def test_conversion_bit_exact(shape):
    rc, re = M.quantize_mxfp4(weights(shape, 7 + sum(shape)).double().numpy())
    want_c, want_e = M.mxfp4_to_fp8(rc, re)
    q8, e8 = binding.mxfp4_to_fp8(torch.from_numpy(pack(rc)).to(DEV),
                                  torch.from_numpy(re.astype(np.int8)).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(e8.cpu().numpy().astype(np.int64), want_e)
    assert np.array_equal(q8.cpu().numpy(), want_c)
    # and the FP8 form holds exactly the MXFP4 values
    assert np.array_equal(F8.dequantize_fp8_tiles(q8.cpu().numpy(), e8.cpu().numpy()), M.dequantize_mxfp4(rc, re))


class OracleMxfp4Fetcher:
    """Expert weights as the oracle's own MXFP4 round trip of the bf16 weights (lazily)."""

    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    @staticmethod
    def _rt(w):
        return M.dequantize_mxfp4(*M.quantize_mxfp4(to64(w)))

    def __call__(self, e):
        if e not in self.cache:
            self.cache[e] = (self._rt(self.inp.w13[e]), self._rt(self.inp.w2[e]))
        return self.cache[e]

    def shared(self):
        if self.inp.w13_sh is None:
            return None
        return self._rt(self.inp.w13_sh), self._rt(self.inp.w2_sh)


CASES = [
    W.TOY,                                                                  # widening FP8 kernels
    W.Workload("mid_T64", T=64, d=512, d_ff=256, E=16, k=4, n_shared=1, score=W.SCORE_SIGMOID, use_bias=True),
    W.Workload("ragged_T150", T=150, d=320, d_ff=192, E=12, k=3, n_shared=1, score=W.SCORE_SOFTMAX),
    W.Workload("wide_T64", T=64, d=512, d_ff=256, E=64, k=2, n_shared=1, score=W.SCORE_SQRT_SOFTPLUS,
               use_bias=True),
]


def run_layer(w, seed, sample=None):
    inp = inputs.make_layer_inputs(w, seed=seed, device=DEV)
    layer = binding.MoELayer(w, inp)
    q8 = layer.mxfp4_to_fp8(layer.quantize_mxfp4())
    y = layer.forward_fp8(inp.x, q8, inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    same = np.ones(w.T, bool)  # every token: the oracle is fed the GPU's ids
    tok = np.nonzero(same)[0]
    if sample is not None:
        tok = np.sort(np.random.default_rng(99).choice(tok, size=min(sample, tok.size), replace=False))
    fetch = OracleMxfp4Fetcher(inp)
    ref = oracle.forward(to64(inp.x), gids, ref_w, fetch, fetch.shared(), tokens=tok)
    e, n = check_output(y.double().cpu().numpy()[tok], ref, label=w.name)
    print(f"{w.name} (mxfp4 weights): max elementwise {e:.2e}, normwise {n:.2e}")
    layer.close()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_mxfp4_layer_vs_oracle(w):
    run_layer(w, seed=31)


@pytest.mark.slow
def test_mxfp4_full_size_layer():
    """The V4-Flash T=64 layer at full size, output on two sampled tokens."""
    run_layer(W.V4FLASH_T64, seed=0, sample=2)


# Native MXFP4 weights (the stored codes and sub-block scales fed to the block-scaled MMA):
# shapes with d and d_ff multiples of 128; batches that take 16-, 32- and 64-row token tiles.
NATIVE = [
    W.Workload("mid_T64", T=64, d=512, d_ff=256, E=16, k=4, n_shared=1, score=W.SCORE_SIGMOID, use_bias=True),
    W.Workload("wide_T64", T=64, d=512, d_ff=256, E=64, k=2, n_shared=1, score=W.SCORE_SQRT_SOFTPLUS,
               use_bias=True),
    W.Workload("noshared_T40", T=40, d=384, d_ff=384, E=12, k=3, n_shared=0, score=W.SCORE_SOFTMAX),
    W.Workload("v4flash_E16_T64", T=64, d=4096, d_ff=2048, E=16, k=6, n_shared=1, score=W.SCORE_SQRT_SOFTPLUS,
               use_bias=True),
    # decode with 64-row token tiles (32 rows per expert on average)
    W.Workload("deep_T64", T=64, d=256, d_ff=384, E=4, k=2, n_shared=1, score=W.SCORE_SOFTMAX),
    # a larger batch at 37.5 rows per expert: still the weight-streaming kernels (64-row tiles,
    # the shared expert's 200 rows in four, the last ragged)
    W.Workload("stream_T200", T=200, d=384, d_ff=256, E=16, k=3, n_shared=1, score=W.SCORE_SOFTMAX),
    # more than 48 rows per expert: the block-scaled CTA-pair kernels (224-row token tiles), one ragged tile per
    # expert, and two per expert (about 256 rows each; d = 384: the down projection's second
    # 256-feature block lies half past the matrix)
    W.Workload("tall_T300", T=300, d=256, d_ff=256, E=8, k=2, n_shared=1, score=W.SCORE_SOFTMAX),
    W.Workload("tall_T512", T=512, d=384, d_ff=256, E=8, k=4, n_shared=1, score=W.SCORE_SIGMOID, use_bias=True),
]


def run_native(w, seed, sample=None):
    inp = inputs.make_layer_inputs(w, seed=seed, device=DEV)
    layer = binding.MoELayer(w, inp)
    q4 = layer.quantize_mxfp4()
    y = layer.forward_mxfp4(inp.x, q4, inp.token_ids)
    assert layer.check_status() == 0
    y_conv = layer.forward_fp8(inp.x, layer.mxfp4_to_fp8(q4), inp.token_ids)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    same = np.ones(w.T, bool)  # every token: the oracle is fed the GPU's ids
    tok = np.nonzero(same)[0]
    if sample is not None:
        tok = np.sort(np.random.default_rng(98).choice(tok, size=min(sample, tok.size), replace=False))
    fetch = OracleMxfp4Fetcher(inp)
    ref = oracle.forward(to64(inp.x), gids, ref_w, fetch, fetch.shared(), tokens=tok)
    e, n = check_output(y.double().cpu().numpy()[tok], ref, label=w.name)
    diff = (y.float() - y_conv.float()).abs().max().item()
    print(f"{w.name} (native mxfp4): max elementwise {e:.2e}, normwise {n:.2e}; "
          f"max |native - converted fp8 path| {diff:.2e}")
    # the FP8 path on the converted weights computes the same layer (exact conversion) with other
    # partial sums: the two agree within the same tolerance
    check_output(y.double().cpu().numpy(), y_conv.double().cpu().numpy(), label=f"{w.name} native vs converted")
    layer.close()


@pytest.mark.parametrize("w", NATIVE, ids=lambda w: w.name)
def test_native_mxfp4_layer_vs_oracle(w):
    run_native(w, seed=37)


@pytest.mark.slow
@pytest.mark.parametrize("w,sample", [(W.V4FLASH_T64, 2), (W.V4FLASH_T8192, 6)], ids=lambda v: getattr(v, "name", str(v)))
def test_native_mxfp4_full_size_layer(w, sample):
    """Full size in the launch configurations the benchmark times: the decode kernels at T=64,
    the block-scaled CTA-pair kernels at T=8192."""
    run_native(w, seed=0, sample=sample)


def test_native_mxfp4_needs_128_multiples():
    inp = inputs.make_layer_inputs(W.TOY, seed=1, device=DEV)
    layer = binding.MoELayer(W.TOY, inp)
    q = layer.quantize_mxfp4()
    with pytest.raises(binding.MoEError) as ei:
        layer.forward_mxfp4(inp.x, q)
    assert binding.STATUS_NAMES[ei.value.status] == "MOE_ERR_UNSUPPORTED"
    layer.close()
