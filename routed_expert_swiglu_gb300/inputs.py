"""Seeded synthetic inputs for the MoE layer.

This module only draws random numbers and lays them out; it holds none of the layer's
arithmetic.  Both the CUDA path and the CPU oracle consume what it produces.

Recipe (seed s; tensor i is drawn from its own generator seeded s*100 + i, in the order
x, W_r, w13, w2, w13_sh, w2_sh, bias, tid2eid, token_ids, zipf permutation):
  * x ~ N(0, 1); weights ~ N(0, 0.02^2), or N(0, 1/fan_in) for the toy layer;
    every float tensor is drawn in fp32 and rounded to nearest-even bf16.
  * bias ~ N(0, 0.01^2) fp32 when the workload uses a selection bias.
  * tid2eid[v] = k distinct expert ids (a random permutation's first k entries);
    token_ids ~ U[0, vocab).
  * Zipf skew: expert e gets a logit offset -s*ln(1 + pi(e)), pi a seeded permutation.
    It is realised through the layer's own inputs: x[:, d-1] = 1 and W_r[e, d-1] = offset_e
    (bf16), so the router computes it like any other logit term.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

from .workloads import Workload

_IDX = {"x": 0, "w_r": 1, "w13": 2, "w2": 3, "w13_sh": 4, "w2_sh": 5, "bias": 6,
        "tid2eid": 7, "token_ids": 8, "zipf": 9}


@dataclasses.dataclass
class LayerInputs:
    x: torch.Tensor                      # [T, d] bf16
    w_r: torch.Tensor                    # [E, d] bf16
    w13: torch.Tensor                    # [E, 2*d_ff, d] bf16 (gate rows, then up rows)
    w2: torch.Tensor                     # [E, d, d_ff] bf16
    w13_sh: Optional[torch.Tensor]       # [2*d_ff, d] bf16
    w2_sh: Optional[torch.Tensor]        # [d, d_ff] bf16
    bias: Optional[torch.Tensor]         # [E] fp32
    tid2eid: Optional[torch.Tensor]      # [vocab, k] int32
    token_ids: Optional[torch.Tensor]    # [T] int32


def _gen(device, seed: int, idx: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100 + idx)
    return g


def _normal_bf16(shape, std: float, g: torch.Generator, device, chunk_rows: int = 0):
    """N(0, std^2) drawn in fp32 then rounded to bf16; optionally drawn in chunks along
    dim 0 (same generator, consecutive draws) to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if chunk_rows <= 0 or shape[0] <= chunk_rows:
        out.copy_((torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std))
        return out
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        sub = (r1 - r0,) + tuple(shape[1:])
        out[r0:r1].copy_(torch.randn(sub, generator=g, device=device, dtype=torch.float32) * std)
    return out


def make_layer_inputs(w: Workload, seed: int = 0, device="cpu", T: Optional[int] = None) -> LayerInputs:
    """Draw every input of workload `w` on `device`.  `T` overrides the token count."""
    T = w.T if T is None else T
    d, f, E, k = w.d, w.d_ff, w.E, w.k
    if w.init == "fan_in":
        std_in, std_ff = 1.0 / math.sqrt(d), 1.0 / math.sqrt(f)
        std_r = std_in
    else:
        std_in = std_ff = std_r = 0.02
    x = _normal_bf16((T, d), 1.0, _gen(device, seed, _IDX["x"]), device)
    w_r = _normal_bf16((E, d), std_r, _gen(device, seed, _IDX["w_r"]), device)
    # Expert weights are drawn one expert at a time to bound the fp32 temporary.
    w13 = _normal_bf16((E, 2 * f, d), std_in, _gen(device, seed, _IDX["w13"]), device, chunk_rows=8)
    w2 = _normal_bf16((E, d, f), std_ff, _gen(device, seed, _IDX["w2"]), device, chunk_rows=8)
    w13_sh = w2_sh = None
    if w.n_shared:
        w13_sh = _normal_bf16((2 * f, d), std_in, _gen(device, seed, _IDX["w13_sh"]), device)
        w2_sh = _normal_bf16((d, f), std_ff, _gen(device, seed, _IDX["w2_sh"]), device)
    bias = None
    if w.use_bias:
        bias = torch.randn((E,), generator=_gen(device, seed, _IDX["bias"]), device=device,
                           dtype=torch.float32) * 0.01
    tid2eid = token_ids = None
    if w.hash_vocab:
        r = torch.rand((w.hash_vocab, E), generator=_gen(device, seed, _IDX["tid2eid"]),
                       device=device)
        tid2eid = r.argsort(dim=1)[:, :k].to(torch.int32).contiguous()
        token_ids = torch.randint(0, w.hash_vocab, (T,), generator=_gen(device, seed, _IDX["token_ids"]),
                                  device=device, dtype=torch.int64).to(torch.int32)
    if w.zipf_s > 0:
        perm = torch.randperm(E, generator=_gen(device, seed, _IDX["zipf"]), device=device)
        offset = -w.zipf_s * torch.log1p(perm.to(torch.float64))
        x[:, d - 1] = 1.0
        w_r[:, d - 1] = offset.to(torch.float32).to(torch.bfloat16)
    return LayerInputs(x, w_r, w13, w2, w13_sh, w2_sh, bias, tid2eid, token_ids)


def random_topk_ids(T: int, E: int, k: int, seed: int = 0, device="cpu", skew: float = 0.0) -> torch.Tensor:
    """[T, k] int32 of k distinct expert ids per token.  With skew > 0 the choice is
    biased towards low expert ids (Gumbel top-k over -skew*ln(1+e)), giving hot experts."""
    g = _gen(device, seed, 50)
    u = torch.rand((T, E), generator=g, device=device).clamp_min(1e-12)
    gumbel = -torch.log(-torch.log(u))
    if skew > 0:
        gumbel = gumbel - skew * torch.log1p(torch.arange(E, device=device, dtype=torch.float32))
    return gumbel.topk(k, dim=1).indices.to(torch.int32).contiguous()
