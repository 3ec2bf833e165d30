"""Work model of the MoE layer: FLOPs, algorithmic bytes and the roofline time.

* One SwiGLU FFN costs 3*d*d_ff parameters and 6*d*d_ff FLOPs per token ("MoE compute and
  communication", section 二.1); a token runs k routed experts plus the shared ones
  (section 二.2), and the router adds 2*d*E FLOPs per token.
* Algorithmic bytes are the bytes a perfect kernel must move: every activated expert's
  weights once (w13 + w2 = 3*d*d_ff bf16 values), the router weight, x in, y out, and the
  routing result (ids int32 + weights fp32).  Dispatch/intermediate buffers are not
  algorithmic.
* Expected activated experts under uniform independent routing of B tokens:
  E*(1 - (1 - k/E)^B) (same page, section 四.1).
"""
from __future__ import annotations

from .workloads import Workload

BF16 = 2


def expert_params(d: int, d_ff: int) -> int:
    return 3 * d * d_ff


def ffn_flops_per_token(d: int, d_ff: int) -> int:
    return 6 * d * d_ff


def expected_active_experts(E: int, k: int, B: int) -> float:
    return E * (1.0 - (1.0 - k / E) ** B)


def layer_flops(w: Workload, T: int | None = None) -> int:
    """Router GEMM + (k + n_shared) SwiGLU FFNs per token."""
    T = w.T if T is None else T
    return T * (w.k + w.n_shared) * ffn_flops_per_token(w.d, w.d_ff) + 2 * T * w.d * w.E


def expert_gemm_flops(w: Workload, T: int | None = None) -> int:
    """FLOPs of the grouped gate/up + down GEMMs (routed and shared), without the router."""
    T = w.T if T is None else T
    return T * (w.k + w.n_shared) * ffn_flops_per_token(w.d, w.d_ff)


def layer_bytes(w: Workload, active_experts: float, T: int | None = None) -> float:
    """Algorithmic HBM bytes of one layer forward."""
    T = w.T if T is None else T
    weights = (active_experts + w.n_shared) * expert_params(w.d, w.d_ff) * BF16
    router = w.E * w.d * BF16
    acts = 2 * T * w.d * BF16
    routing = T * w.k * 8
    hashing = (T * 4 + T * w.k * 4) if w.hash_vocab else 0
    return weights + router + acts + routing + hashing


def expert_gemm_bytes(w: Workload, active_experts: float, T: int | None = None) -> float:
    """Algorithmic HBM bytes of the two grouped GEMMs: every activated expert's weights (and the
    shared expert's) once, the token rows in and the layer's rows out."""
    T = w.T if T is None else T
    return (active_experts + w.n_shared) * expert_params(w.d, w.d_ff) * BF16 + 2 * T * w.d * BF16


def roofline_seconds(flops: float, nbytes: float, peak_tflops: float, peak_gbs: float) -> float:
    """max(compute time, memory time) at the given peaks."""
    return max(flops / (peak_tflops * 1e12), nbytes / (peak_gbs * 1e9))
