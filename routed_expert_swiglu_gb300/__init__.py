"""Single-GPU Mixture-of-Experts SwiGLU FFN layer forward for GB300 (sm_103a).

The compute path is the CUDA library built from csrc/ (C ABI in include/moe.h); `binding`
is its thin ctypes binding.  `workloads` and `inputs` describe and draw synthetic layers;
`cost` holds the FLOP / byte model used for roofline reporting.
"""
from . import cost, inputs, workloads  # noqa: F401

__all__ = ["binding", "build", "cost", "inputs", "workloads"]
