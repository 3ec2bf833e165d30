"""The debug-bounds build (MOE_DEBUG_BOUNDS=1): internal row indices of the dispatch (scatter
rows, gathered token rows, token-major destination rows, the rows the E4M3 pieces of x are
written to), the grouped GEMMs' output rows (bf16, FP8 and MXFP4 weights) and the combine's rows
are checked before use, and a failed check is reported as MOE_ERR_INTERNAL
instead of addressing memory out of range.  On valid inputs no check may fire and the layer's
output must equal the default build's bit for bit (the checks only guard accesses).  The build
runs in a child process; this process runs the default library on the same inputs."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from routed_expert_swiglu_gb300 import binding, build, inputs, workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# bf16 layers, and a layer with d, d_ff multiples of 128 on FP8 and MXFP4 weights: decode kernels
# (T = 40), the block-scaled CTA-pair kernels (T = 300), and the token-major split of x (T = 1100)
CASES = ["toy_T64", "toy_T333", "v4flash_T300", "v3_T200", "fmt_T40:fp8", "fmt_T300:fp8", "fmt_T1100:fp8",
         "fmt_T40:mxfp4", "fmt_T300:mxfp4"]
FMT = W.Workload("fmt_T40", T=40, d=256, d_ff=256, E=8, k=2, n_shared=1, score=W.SCORE_SOFTMAX)

CHILD = """
import sys
import numpy as np
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
from routed_expert_swiglu_gb300 import binding
binding.load({lib!r})
import test_gpu_debug_bounds as t
out = {{}}
for name in t.CASES:
    y, st = t.run_case(name)
    out[name] = y
    print("status", name, st, flush=True)
np.savez({npz!r}, **out)
"""


def workload(name):
    base, T = name.split(":")[0].rsplit("_T", 1)
    w = {"toy": W.TOY, "v4flash": W.V4FLASH_T8192, "v3": W.V3_T4096, "fmt": FMT}[base]
    return w.with_T(int(T))


def run_case(name):
    """The layer's forward on seeded inputs: (output as int16 bit patterns, status)."""
    w = workload(name)
    fmt = name.split(":")[1] if ":" in name else "bf16"
    inp = inputs.make_layer_inputs(w, seed=11, device=DEV)
    layer = binding.MoELayer(w, inp)
    if fmt == "fp8":
        y = layer.forward_fp8(inp.x, layer.quantize_fp8(), inp.token_ids)
    elif fmt == "mxfp4":
        y = layer.forward_mxfp4(inp.x, layer.quantize_mxfp4(), inp.token_ids)
    else:
        y = layer.forward(inp.x, inp.token_ids)
    st = layer.check_status()
    bits = y.view(torch.int16).cpu().numpy()
    layer.close()
    return bits, st


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load()


def test_debug_bounds_build_matches_the_default_build(tmp_path):
    pkg = os.path.join(ROOT, "routed_expert_swiglu_gb300")
    lib = build.build(extra_flags=["-DMOE_DEBUG_BOUNDS=1"], lib_path=os.path.join(pkg, "libmoe_gb300_debug_bounds.so"),
                      build_dir=os.path.join(pkg, "_build_debug_bounds"))
    npz = str(tmp_path / "debug_bounds.npz")
    child = CHILD.format(root=ROOT, tests=os.path.dirname(os.path.abspath(__file__)), lib=lib, npz=npz)
    out = subprocess.run([sys.executable, "-c", child], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    got = [ln.split() for ln in out.stdout.splitlines() if ln.startswith("status")]
    assert [g[1] for g in got] == CASES, out.stdout
    assert all(int(g[2]) == 0 for g in got), out.stdout
    dbg = np.load(npz)
    for name in CASES:
        ref, st = run_case(name)
        assert st == 0
        assert np.array_equal(dbg[name], ref), f"{name}: debug-bounds build output differs"
