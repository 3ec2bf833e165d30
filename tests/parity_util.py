"""Helpers shared by the GPU parity tests: oracle evaluation on GPU-resident inputs and the
comparison rules.

Tolerances (fixed for this layer): layer output max|gpu - oracle| / (|oracle| + 1e-2) <= 2e-2
and normwise relative error <= 5e-3; gate weights <= 1e-3 absolute; integer results exact.
Routing: a token whose oracle selection margin (k-th vs (k+1)-th key, and last kept vs first
dropped group) exceeds 1e-3 must get exactly the oracle's SET of experts; their listed order
must match too where every gap between consecutive selected keys exceeds 1e-3 (nearly equal
keys may be listed either way).  Gate weights are compared per expert id.  A token inside
the selection margin may get any valid selection, and its output is compared only when its
set equals the oracle's.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_ELEM_TOL = 2e-2
OUT_ELEM_FLOOR = 1e-2
OUT_NORM_TOL = 5e-3
WEIGHT_TOL = 1e-3
MARGIN = 1e-3


def to64(t):
    """Device tensor -> fp64 numpy (copied in its own dtype, widened on the host; exact)."""
    return None if t is None else t.detach().cpu().to(torch.float64).numpy()


class ExpertFetcher:
    """Expert weights pulled from the device one expert at a time as fp64 (exact: bf16 -> fp64)."""

    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    def __call__(self, e):
        if e not in self.cache:
            if len(self.cache) > 8:
                self.cache.clear()
            self.cache[e] = (to64(self.inp.w13[e]), to64(self.inp.w2[e]))
        return self.cache[e]

    def shared(self):
        if self.inp.w13_sh is None:
            return None
        return to64(self.inp.w13_sh), to64(self.inp.w2_sh)


def oracle_route(w, inp, with_order=False):
    logits = oracle.router_logits(to64(inp.x), to64(inp.w_r))
    tid2eid = None if inp.tid2eid is None else inp.tid2eid.cpu().numpy()
    token_ids = None if inp.token_ids is None else inp.token_ids.cpu().numpy()
    ids, wts, margin, order_margin = oracle.route(
        logits, w.k, w.score, bias=to64(inp.bias), n_groups=w.n_groups, topk_groups=w.topk_groups,
        group_topk=w.group_topk, token_ids=token_ids, tid2eid=tid2eid, return_order_margin=True)
    if with_order:
        return logits, ids, wts, margin, order_margin
    return logits, ids, wts, margin


def check_routing(w, gpu_ids, gpu_w, ids, wts, margin, order_margin=None, inp=None):
    """Returns the boolean mask of tokens whose GPU expert set equals the oracle's."""
    gpu_ids = np.asarray(gpu_ids)
    gpu_w = np.asarray(gpu_w, np.float64)
    k = gpu_ids.shape[1]
    safe = margin > MARGIN
    g_order = np.argsort(gpu_ids, axis=1, kind="stable")
    o_order = np.argsort(ids, axis=1, kind="stable")
    g_sorted = np.take_along_axis(gpu_ids, g_order, axis=1)
    o_sorted = np.take_along_axis(ids, o_order, axis=1)
    same_set = (g_sorted == o_sorted).all(axis=1)
    bad = np.nonzero(~same_set & safe)[0]
    assert bad.size == 0, f"{bad.size} margin-safe tokens routed to a different expert set, e.g. token " \
                          f"{bad[:5]}: gpu {gpu_ids[bad[:1]]} oracle {ids[bad[:1]]}"
    if order_margin is not None:
        order_safe = safe & (order_margin > MARGIN)
        bad = np.nonzero(order_safe & (gpu_ids != ids).any(axis=1))[0]
        assert bad.size == 0, f"{bad.size} tokens list their experts in a different order although every " \
                              f"gap exceeds the margin, e.g. token {bad[:5]}"
    if same_set.any():
        gw = np.take_along_axis(gpu_w, g_order, axis=1)[same_set]
        ow = np.take_along_axis(wts, o_order, axis=1)[same_set]
        err = np.abs(gw - ow).max()
        assert err <= WEIGHT_TOL, f"gate weights differ by {err:.3e}"
    # tokens inside the margin with another selection: it must still be a valid one
    for t in np.nonzero(~same_set)[0]:
        assert len(set(gpu_ids[t].tolist())) == k, f"token {t}: repeated expert"
        assert ((gpu_ids[t] >= 0) & (gpu_ids[t] < w.E)).all()
    return same_set


def check_output(got, ref, rows=None, label=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    elem = np.abs(got - ref) / (np.abs(ref) + OUT_ELEM_FLOOR)
    norm = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    i = np.unravel_index(np.argmax(elem), elem.shape)
    assert elem.max() <= OUT_ELEM_TOL, f"{label}: max elementwise {elem.max():.3e} at {i}: gpu {got[i]} oracle {ref[i]}"
    assert norm <= OUT_NORM_TOL, f"{label}: normwise {norm:.3e}"
    return float(elem.max()), float(norm)
