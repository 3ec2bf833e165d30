"""Build the CUDA library in-tree: one nvcc process per translation unit (in parallel), then a
shared-library link.  Target: sm_103a only.  Output: routed_expert_swiglu_gb300/libmoe_gb300.so.

    python -m routed_expert_swiglu_gb300.build [--verbose-ptxas]
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmoe_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = ["moe_api.cu", "grouped_gemm.cu", "fp8_gemm.cu", "bs_pair_gemm.cu", "routing.cu", "permute.cu", "combine.cu", "permute_noalloc.cu",
           "bias_update.cu", "fp8_quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{os.path.join(ROOT, 'include')}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the MoE library")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "moe.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose_ptxas: bool = False, force: bool = False, extra_flags=(), lib_path: str = LIB_PATH,
          build_dir: str = BUILD_DIR) -> str:
    """Compile every translation unit for sm_103a and link the shared library; returns its path.
    `extra_flags` (e.g. -DMOE_TN_PREFILL=256) select compile-time kernel variants; give such a
    build its own `lib_path` and `build_dir`."""
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or _stale(o, s):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o]
            if verbose_ptxas:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    outs = []
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
                if res.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
                outs.append(res.stderr)
    objs = [os.path.join(build_dir, s.replace(".cu", ".o")) for s in SOURCES]
    if jobs or not os.path.exists(lib_path):
        tmp = lib_path + ".tmp"
        res = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    if verbose_ptxas:
        sys.stderr.write("".join(outs))
    return lib_path


if __name__ == "__main__":
    print(build(verbose_ptxas="--verbose-ptxas" in sys.argv, force="--force" in sys.argv))
