"""Helpers shared by the GPU parity tests: oracle evaluation on GPU-resident inputs and the
comparison rules.

Tolerances (fixed for this layer): layer output max|gpu - oracle| / (|oracle| + 1e-2) <= 2e-2
and normwise relative error <= 5e-3; gate weights <= 1e-3 absolute; integer results exact.

Routing (margin 1e-3, keys and group scores from the fp64 oracle):
  * a token whose selection margin (k-th vs (k+1)-th key, and last kept vs first dropped group
    score) exceeds the margin gets exactly the oracle's set of experts;
  * where, in addition, every gap between consecutive selected keys exceeds the margin, the
    listed ids equal the oracle's bit for bit, order included (hash routing: always);
  * every token lists its experts in descending key order to within the margin;
  * a token inside the selection margin may get another selection, which must be a valid one
    to within the margin: distinct ids in range, the touched groups among those the oracle could
    have kept, and no expert it could have taken (in a touched or surely kept group) ahead of a
    chosen one by more than the margin;
  * the gate weights of every token equal the oracle's weights for the GPU's ids (<= 1e-3), and
    the layer output is compared with the oracle fed the GPU's ids, so the tokens inside the
    margin are checked like the rest.
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


class OracleRouting:
    """The oracle's routing of a layer's inputs, with what the checks need: logits, selection
    keys (before group masking), group scores, ids, weights and the two margins."""

    def __init__(self, w, inp):
        self.logits = oracle.router_logits(to64(inp.x), to64(inp.w_r))
        self.bias = to64(inp.bias)
        self.hashed = inp.tid2eid is not None
        tid2eid = None if inp.tid2eid is None else inp.tid2eid.cpu().numpy()
        token_ids = None if inp.token_ids is None else inp.token_ids.cpu().numpy()
        self.ids, self.wts, self.margin, self.order_margin = oracle.route(
            self.logits, w.k, w.score, bias=self.bias, n_groups=w.n_groups, topk_groups=w.topk_groups,
            group_topk=w.group_topk, token_ids=token_ids, tid2eid=tid2eid, return_order_margin=True)
        self.keys = oracle.selection_keys(self.logits, w.score, self.bias)
        self.gscore = (oracle.group_scores(self.keys, w.n_groups, w.group_topk) if w.n_groups else None)

    def weights_for(self, w, ids):
        """The oracle's gate weights of the given selection."""
        return oracle.gate_weights(self.logits, ids, w.score)


def oracle_routing(w, inp) -> OracleRouting:
    return OracleRouting(w, inp)


def oracle_route(w, inp, with_order=False):
    r = OracleRouting(w, inp)
    if with_order:
        return r.logits, r.ids, r.wts, r.margin, r.order_margin
    return r.logits, r.ids, r.wts, r.margin


def _valid_near_tie(w, R, t, chosen):
    """A selection of token t that differs from the oracle's is valid to within MARGIN: the groups
    it touches could have been kept, and no expert the token could have taken beats a chosen one by
    more than MARGIN."""
    key = R.keys[t]
    E = key.shape[0]
    if R.gscore is not None:
        gsz = E // w.n_groups
        gs = R.gscore[t]
        srt = np.sort(gs)[::-1]
        touched = sorted(set(int(e) // gsz for e in chosen))
        assert len(touched) <= w.topk_groups, f"token {t}: experts span {len(touched)} groups"
        thr = srt[w.topk_groups - 1]
        assert all(gs[g] >= thr - MARGIN for g in touched), f"token {t}: a touched group could not be kept"
        sure = [g for g in range(w.n_groups)
                if w.topk_groups < w.n_groups and gs[g] > srt[w.topk_groups] + MARGIN]
        cand = [e for g in sorted(set(touched) | set(sure)) for e in range(g * gsz, (g + 1) * gsz)]
    else:
        cand = range(E)
    others = np.array([key[e] for e in cand if e not in set(chosen.tolist())])
    lo = min(key[e] for e in chosen)
    assert others.size == 0 or others.max() <= lo + MARGIN, \
        f"token {t}: an unchosen expert's key beats a chosen one by {others.max() - lo:.3e}"


def check_routing(w, gpu_ids, gpu_w, R: OracleRouting):
    """Checks the GPU's routing against the oracle's (rules in the module docstring).  Returns
    (the oracle's weights for the GPU's ids, the number of tokens routed to another set)."""
    gpu_ids = np.asarray(gpu_ids)
    gpu_w = np.asarray(gpu_w, np.float64)
    T, k = gpu_ids.shape
    assert ((gpu_ids >= 0) & (gpu_ids < w.E)).all(), "expert id out of range"
    assert (np.sort(gpu_ids, axis=1)[:, 1:] != np.sort(gpu_ids, axis=1)[:, :-1]).all(), "repeated expert"
    ids = R.ids
    safe = R.margin > MARGIN
    same_set = (np.sort(gpu_ids, axis=1) == np.sort(ids, axis=1)).all(axis=1)
    bad = np.nonzero(~same_set & safe)[0]
    assert bad.size == 0, f"{bad.size} margin-safe tokens routed to a different expert set, e.g. token " \
                          f"{bad[:5]}: gpu {gpu_ids[bad[:1]]} oracle {ids[bad[:1]]}"
    exact = safe & (R.order_margin > MARGIN)
    bad = np.nonzero(exact & (gpu_ids != ids).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} margin-safe tokens list other ids or another order although every " \
                          f"gap exceeds the margin, e.g. token {bad[:5]}: gpu {gpu_ids[bad[:1]]} oracle {ids[bad[:1]]}"
    if not R.hashed:
        gk = np.take_along_axis(R.keys, gpu_ids.astype(np.int64), axis=1)
        drop = (gk[:, 1:] - gk[:, :-1]).max(axis=1) if k > 1 else np.zeros(T)
        bad = np.nonzero(drop > MARGIN)[0]
        assert bad.size == 0, f"{bad.size} tokens list their experts out of key order, e.g. token {bad[:5]}"
        for t in np.nonzero(~same_set)[0]:
            _valid_near_tie(w, R, t, gpu_ids[t])
    ref_w = R.weights_for(w, gpu_ids)
    err = np.abs(gpu_w - ref_w).max()
    assert err <= WEIGHT_TOL, f"gate weights differ by {err:.3e}"
    return ref_w, int((~same_set).sum())


def oracle_output(inp, gpu_ids, ref_w, tokens=None, fetch=None):
    """The oracle's layer output fed the GPU's expert ids and the oracle's weights for them, on
    `tokens` (default: all)."""
    fetch = fetch or ExpertFetcher(inp)
    return oracle.forward(to64(inp.x), gpu_ids, ref_w, fetch, fetch.shared(), tokens=tokens)


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
