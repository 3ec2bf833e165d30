"""Bounded pipeline waits, exercised without faulting or hanging the GPU.

A test build of the library (MOE_TEST_UNSET_WAIT=1, MOE_WAIT_LIMIT_NS = 1 ms) makes the epilogue
warps of every grouped-GEMM launch (the tensor-core router GEMM above 64 tokens, single-CTA and
CTA-pair bf16 expert GEMMs, the FP8 and block-scaled MXFP4 decode GEMMs and the block-scaled
CTA-pair FP8 / MXFP4 GEMMs) first wait on a barrier phase that nothing completes.  Each such launch must give up after the limit,
stop its roles, wait out the quiet period in which the copies and MMAs issued before the abort
land, release its Tensor Memory, and report MOE_ERR_TIMEOUT through moe_check_status.  The test
build runs in a child process; afterwards this process runs the normal library on the same GPU
and its output must still match the oracle."""
import os
import subprocess
import sys

import pytest
import torch

from routed_expert_swiglu_gb300 import binding, build, inputs, workloads as W

from parity_util import check_output, check_routing, oracle_output, oracle_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MOE_ERR_TIMEOUT = 7

CHILD = """
import sys
sys.path.insert(0, {root!r})
from routed_expert_swiglu_gb300 import binding, inputs, workloads as W
binding.load({lib!r})
for w in (W.TOY, W.TOY.with_T(333), W.TOY.with_T(1)):
    inp = inputs.make_layer_inputs(w, seed=0, device="cuda:0")
    layer = binding.MoELayer(w, inp)
    layer.forward(inp.x)
    print("status", w.name, layer.check_status(), flush=True)
    layer.close()
# weight formats on the block-scaled kernels (d, d_ff multiples of 128): decode and prefill sizes
f = W.Workload("fmt_T32", T=32, d=256, d_ff=256, E=8, k=2, n_shared=1, score=W.SCORE_SOFTMAX)
for w in (f, f.with_T(300)):
    inp = inputs.make_layer_inputs(w, seed=0, device="cuda:0")
    layer = binding.MoELayer(w, inp)
    layer.forward_fp8(inp.x, layer.quantize_fp8())
    print("status", w.name + "_fp8", layer.check_status(), flush=True)
    layer.forward_mxfp4(inp.x, layer.quantize_mxfp4())
    print("status", w.name + "_mxfp4", layer.check_status(), flush=True)
    layer.close()
"""


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load()


def test_a_wait_that_runs_out_reports_timeout_and_leaves_the_gpu_usable():
    pkg = os.path.join(ROOT, "routed_expert_swiglu_gb300")
    lib = build.build(extra_flags=["-DMOE_TEST_UNSET_WAIT=1", "-DMOE_WAIT_LIMIT_NS=1000000ull"],
                      lib_path=os.path.join(pkg, "libmoe_gb300_unset_wait.so"),
                      build_dir=os.path.join(pkg, "_build_unset_wait"))
    out = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, lib=lib)], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    got = [ln.split() for ln in out.stdout.splitlines() if ln.startswith("status")]
    assert len(got) == 7, out.stdout
    for _, name, st in got:
        assert int(st) == MOE_ERR_TIMEOUT, f"{name}: status {st}, expected MOE_ERR_TIMEOUT"
    # the normal library on the same GPU afterwards
    w = W.TOY.with_T(333)
    inp = inputs.make_layer_inputs(w, seed=5, device=DEV)
    layer = binding.MoELayer(w, inp)
    y = layer.forward(inp.x)
    assert layer.check_status() == 0
    v = layer.views(w.T)
    gids = v["topk_ids"].cpu().numpy()
    ref_w, _ = check_routing(w, gids, v["topk_w"].cpu().numpy(), oracle_routing(w, inp))
    check_output(y.double().cpu().numpy(), oracle_output(inp, gids, ref_w), label=w.name)
    layer.close()
