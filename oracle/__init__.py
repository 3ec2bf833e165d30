"""CPU oracle for the MoE SwiGLU layer forward.

Test infrastructure only: the tests, the package smoke check and the benchmark's CPU
baseline leg are its only users.  It shares no code with the CUDA path.
"""
from .moe_oracle import (DENOM_MIN, SCORES, affinity, bias_update, forward, gate_weights, group_scores,
                         permute, round_to_bf16, route, router_logits, selection_keys, sigmoid, silu,
                         softmax, softplus, sqrt_softplus, swiglu_expert)
from . import fp8_weights  # noqa: E402,F401
from . import mxfp4_weights  # noqa: E402,F401
