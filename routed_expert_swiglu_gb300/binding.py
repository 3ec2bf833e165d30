"""Thin Python binding of the C ABI in include/moe.h (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA library.  Functions keep
the C names; tensors are torch tensors on the current CUDA device (their data pointers are
passed through) and calls are enqueued on torch's current stream unless `stream` is given.
Loading fails loudly when the library has not been built: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import workloads as W

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
                4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_INPUT", 7: "MOE_ERR_TIMEOUT",
                8: "MOE_ERR_INTERNAL"}
SCORE_CODES = {W.SCORE_SOFTMAX_TOPK: 0, W.SCORE_SOFTMAX: 1, W.SCORE_SIGMOID: 2, W.SCORE_SQRT_SOFTPLUS: 3}

# Every symbol include/moe.h declares.
EXPORTED = ("moe_plan_create", "moe_plan_destroy", "moe_workspace_bytes", "moe_route", "moe_permute",
            "moe_forward", "moe_forward_routed", "moe_forward_host", "moe_check_status",
            "moe_workspace_views", "moe_forward_stage_count", "moe_plan_set_events",
            "moe_forward_launch_count", "moe_status_string", "moe_permute_noalloc", "moe_permute_noalloc_status",
            "moe_update_bias", "moe_quantize_fp8", "moe_forward_fp8", "moe_quantize_mxfp4", "moe_mxfp4_to_fp8",
            "moe_forward_mxfp4")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("score", ctypes.c_int32), ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("group_topk", ctypes.c_int32), ("tid2eid", ctypes.c_void_p), ("vocab", ctypes.c_int32)]


class moe_ws_views(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_ids", "topk_w", "logits", "counts", "offsets", "perm_tok", "inv", "h", "o")]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"MoE CUDA library not built ({path}); run routed_expert_swiglu_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, S, V = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
    sig = {
        "moe_plan_create": ([ctypes.POINTER(moe_config), ctypes.POINTER(P)], I),
        "moe_plan_destroy": ([P], I),
        "moe_workspace_bytes": ([P, I], S),
        "moe_route": ([P, I, V, V, V, V, V, V, V, V, S, V], I),
        "moe_permute": ([P, I, V, V, V, V, V, V, S, V], I),
        "moe_forward": ([P, I, V, V, V, V, V, V, V, V, V, V, S, V], I),
        "moe_forward_routed": ([P, I, V, V, V, V, V, V, V, V, V, S, V], I),
        "moe_forward_host": ([P, I, V, V, V, V, V, V, V, V, V, V, S, V], I),
        "moe_check_status": ([P, V, V], I),
        "moe_workspace_views": ([P, I, V, ctypes.POINTER(moe_ws_views)], I),
        "moe_forward_stage_count": ([], I),
        "moe_plan_set_events": ([P, V, I], I),
        "moe_forward_launch_count": ([P, I], I),
        "moe_status_string": ([I], ctypes.c_char_p),
        "moe_permute_noalloc": ([P, I, V, V, V, V, V, V], I),
        "moe_permute_noalloc_status": ([V], I),
        "moe_update_bias": ([P, I, V, V, ctypes.c_float, V], I),
        "moe_quantize_fp8": ([V, I, I, I, V, V, V], I),
        "moe_forward_fp8": ([P, I, V, V, V, V, V, V, V, V, V, V, V, V, V, V, S, V], I),
        "moe_quantize_mxfp4": ([V, I, I, I, V, V, V], I),
        "moe_mxfp4_to_fp8": ([V, V, I, I, I, V, V, V], I),
        "moe_forward_mxfp4": ([P, I] + [V] * 14 + [S, V], I),
    }
    for name, (argt, rest) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = argt
        fn.restype = rest
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, where: str):
    if st != MOE_OK:
        raise MoEError(st, where)


def config_for(w: W.Workload, max_tokens: Optional[int] = None, tid2eid: Optional[torch.Tensor] = None) -> moe_config:
    c = moe_config()
    c.d, c.d_ff, c.n_experts, c.top_k, c.n_shared = w.d, w.d_ff, w.E, w.k, w.n_shared
    c.max_tokens = max_tokens or w.T
    c.score = SCORE_CODES[w.score]
    c.n_groups, c.topk_groups, c.group_topk = w.n_groups, w.topk_groups, w.group_topk
    c.tid2eid = None if tid2eid is None else tid2eid.data_ptr()
    c.vocab = w.hash_vocab if tid2eid is not None else 0
    return c


# ----------------------------------------------------------------------------- C names

def moe_plan_create(cfg: moe_config) -> ctypes.c_void_p:
    lib = load()
    plan = ctypes.c_void_p()
    _check(lib.moe_plan_create(ctypes.byref(cfg), ctypes.byref(plan)), "moe_plan_create")
    return plan


def moe_plan_destroy(plan) -> None:
    load().moe_plan_destroy(plan)


def moe_workspace_bytes(plan, T: int) -> int:
    return int(load().moe_workspace_bytes(plan, T))


def moe_route(plan, T, x, token_ids, w_r, bias, topk_ids, topk_w, logits, ws, stream=None):
    _check(load().moe_route(plan, T, _ptr(x), _ptr(token_ids), _ptr(w_r), _ptr(bias), _ptr(topk_ids),
                            _ptr(topk_w), _ptr(logits), _ptr(ws), ws.numel() * ws.element_size(),
                            _stream(stream)), "moe_route")


def moe_permute(plan, T, topk_ids, counts, offsets, perm_tok, inv, ws, stream=None):
    _check(load().moe_permute(plan, T, _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(perm_tok), _ptr(inv),
                              _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_permute")


def moe_permute_noalloc(plan, T, topk_ids, counts, offsets, perm_tok, inv, stream=None):
    """moe_permute without a workspace, for callers that may not allocate device memory (the
    library keeps a fixed scratch array on each device; T * top_k <= 131072)."""
    _check(load().moe_permute_noalloc(plan, T, _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(perm_tok),
                                      _ptr(inv), _stream(stream)), "moe_permute_noalloc")


def moe_permute_noalloc_status(stream=None):
    """Status code of the latest moe_permute_noalloc call on the current device (synchronises
    the stream): MOE_OK, or MOE_ERR_DEVICE_INPUT if it met an expert id outside [0, E)."""
    return int(load().moe_permute_noalloc_status(_stream(stream)))


def moe_update_bias(plan, T, counts, bias, gamma=0.001, stream=None):
    """In-place aux-loss-free bias step from the per-expert loads of a T-token step."""
    _check(load().moe_update_bias(plan, T, _ptr(counts), _ptr(bias), ctypes.c_float(gamma), _stream(stream)),
           "moe_update_bias")


def moe_forward(plan, T, x, token_ids, w_r, bias, w13, w2, w13_sh, w2_sh, out, ws, stream=None):
    _check(load().moe_forward(plan, T, _ptr(x), _ptr(token_ids), _ptr(w_r), _ptr(bias), _ptr(w13), _ptr(w2),
                              _ptr(w13_sh), _ptr(w2_sh), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "moe_forward")


def moe_quantize_fp8(w, codes, exps, stream=None):
    """E4M3 codes [n, rows, K] (uint8) and 128 x 128 tile exponents [n, ceil(rows/128),
    ceil(K/128)] (int8) of bf16 weight matrices w [n, rows, K] (or [rows, K])."""
    n, rows, K = (1,) + tuple(w.shape) if w.dim() == 2 else tuple(w.shape)
    _check(load().moe_quantize_fp8(_ptr(w), n, rows, K, _ptr(codes), _ptr(exps), _stream(stream)),
           "moe_quantize_fp8")


def quantize_fp8(w, stream=None):
    """Allocate and fill the FP8 codes and tile exponents of bf16 weights w [.., rows, K]."""
    rows, K = w.shape[-2:]
    codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    exps = torch.empty(tuple(w.shape[:-2]) + (-(-rows // 128), -(-K // 128)), dtype=torch.int8, device=w.device)
    moe_quantize_fp8(w, codes, exps, stream)
    return codes, exps


def quantize_mxfp4(w, stream=None):
    """MXFP4 codes [.., rows, K/2] (uint8, two per byte) and 1 x 32 sub-block exponents
    [.., rows, K/32] (int8) of bf16 weights w [.., rows, K]."""
    rows, K = w.shape[-2:]
    n = 1
    for v in w.shape[:-2]:
        n *= v
    codes = torch.empty(tuple(w.shape[:-1]) + (K // 2,), dtype=torch.uint8, device=w.device)
    exps = torch.empty(tuple(w.shape[:-1]) + (K // 32,), dtype=torch.int8, device=w.device)
    _check(load().moe_quantize_mxfp4(_ptr(w), n, rows, K, _ptr(codes), _ptr(exps), _stream(stream)),
           "moe_quantize_mxfp4")
    return codes, exps


def mxfp4_to_fp8(codes, exps, stream=None):
    """The FP8 codes [.., rows, K] and 128 x 128 tile exponents of MXFP4 weights (lossless)."""
    rows, K = codes.shape[-2], codes.shape[-1] * 2
    n = 1
    for v in codes.shape[:-2]:
        n *= v
    q8 = torch.empty(tuple(codes.shape[:-1]) + (K,), dtype=torch.uint8, device=codes.device)
    e8 = torch.empty(tuple(codes.shape[:-2]) + (-(-rows // 128), -(-K // 128)), dtype=torch.int8,
                     device=codes.device)
    _check(load().moe_mxfp4_to_fp8(_ptr(codes), _ptr(exps), n, rows, K, _ptr(q8), _ptr(e8), _stream(stream)),
           "moe_mxfp4_to_fp8")
    return q8, e8


def moe_forward_mxfp4(plan, T, x, token_ids, w_r, bias, w13, w2, w13_sh, w2_sh, out, ws, stream=None):
    """w13, w2, w13_sh, w2_sh: (codes, sub-block exponents) pairs as quantize_mxfp4 returns them
    (shared: None without a shared expert)."""
    def pair(q):
        return (None, None) if q is None else (_ptr(q[0]), _ptr(q[1]))
    args = [*pair(w13), *pair(w2), *pair(w13_sh), *pair(w2_sh)]
    _check(load().moe_forward_mxfp4(plan, T, _ptr(x), _ptr(token_ids), _ptr(w_r), _ptr(bias), *args, _ptr(out),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_forward_mxfp4")


def moe_forward_fp8(plan, T, x, token_ids, w_r, bias, q13, e13, q2, e2, q13_sh, e13_sh, q2_sh, e2_sh, out, ws,
                    stream=None):
    _check(load().moe_forward_fp8(plan, T, _ptr(x), _ptr(token_ids), _ptr(w_r), _ptr(bias), _ptr(q13), _ptr(e13),
                                  _ptr(q2), _ptr(e2), _ptr(q13_sh), _ptr(e13_sh), _ptr(q2_sh), _ptr(e2_sh),
                                  _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_forward_fp8")


def moe_forward_routed(plan, T, x, topk_ids, topk_w, w13, w2, w13_sh, w2_sh, out, ws, stream=None):
    _check(load().moe_forward_routed(plan, T, _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w13), _ptr(w2),
                                     _ptr(w13_sh), _ptr(w2_sh), _ptr(out), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)), "moe_forward_routed")


def moe_forward_host(plan, T, x_host, token_ids_host, w_r, bias, w13, w2, w13_sh, w2_sh, out_host, ws, stream=None):
    _check(load().moe_forward_host(plan, T, _ptr(x_host), _ptr(token_ids_host), _ptr(w_r), _ptr(bias), _ptr(w13),
                                   _ptr(w2), _ptr(w13_sh), _ptr(w2_sh), _ptr(out_host), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)), "moe_forward_host")


def moe_check_status(plan, ws, stream=None) -> int:
    return int(load().moe_check_status(plan, _ptr(ws), _stream(stream)))


def moe_workspace_views(plan, T, ws) -> moe_ws_views:
    v = moe_ws_views()
    _check(load().moe_workspace_views(plan, T, _ptr(ws), ctypes.byref(v)), "moe_workspace_views")
    return v


def moe_forward_stage_count() -> int:
    return int(load().moe_forward_stage_count())


def moe_plan_set_events(plan, events) -> None:
    """events: list of torch.cuda.Event (already recorded once so that they exist) or None."""
    if not events:
        _check(load().moe_plan_set_events(plan, None, 0), "moe_plan_set_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().moe_plan_set_events(plan, arr, len(events)), "moe_plan_set_events")
    return arr  # the caller keeps it alive while the plan uses it


def moe_forward_launch_count(plan, T) -> int:
    return int(load().moe_forward_launch_count(plan, T))


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


# ----------------------------------------------------------------------------- helpers

class MoELayer:
    """A plan plus a workspace sized for `max_tokens`, bound to one set of layer weights."""

    def __init__(self, w: W.Workload, inputs, max_tokens: Optional[int] = None, device=None):
        self.w = w
        self.inputs = inputs
        self.device = device or inputs.x.device
        self.max_tokens = max_tokens or w.T
        self.cfg = config_for(w, self.max_tokens, inputs.tid2eid)
        self.plan = moe_plan_create(self.cfg)
        nbytes = moe_workspace_bytes(self.plan, self.max_tokens)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self._events_arr = None

    def close(self):
        if self.plan is not None:
            moe_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ws_slice(self, ptr: int, numel: int, dtype) -> torch.Tensor:
        base = self.ws.data_ptr()
        off = int(ptr) - base
        esz = torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + numel * esz].view(dtype)

    def forward(self, x, token_ids=None, out=None, stream=None):
        T = x.shape[0]
        inp = self.inputs
        if out is None:
            out = torch.empty((T, self.w.d), dtype=torch.bfloat16, device=self.device)
        moe_forward(self.plan, T, x, token_ids, inp.w_r, inp.bias, inp.w13, inp.w2, inp.w13_sh, inp.w2_sh, out,
                    self.ws, stream)
        return out

    def quantize_fp8(self, stream=None):
        """FP8 codes and tile exponents of this layer's expert weights (routed and shared)."""
        inp = self.inputs
        q = {"w13": quantize_fp8(inp.w13, stream), "w2": quantize_fp8(inp.w2, stream)}
        if inp.w13_sh is not None:
            q["w13_sh"] = quantize_fp8(inp.w13_sh, stream)
            q["w2_sh"] = quantize_fp8(inp.w2_sh, stream)
        return q

    def quantize_mxfp4(self, stream=None):
        """MXFP4 codes and sub-block exponents of this layer's expert weights."""
        inp = self.inputs
        q = {"w13": quantize_mxfp4(inp.w13, stream), "w2": quantize_mxfp4(inp.w2, stream)}
        if inp.w13_sh is not None:
            q["w13_sh"] = quantize_mxfp4(inp.w13_sh, stream)
            q["w2_sh"] = quantize_mxfp4(inp.w2_sh, stream)
        return q

    @staticmethod
    def mxfp4_to_fp8(q4, stream=None):
        """The FP8 form (for forward_fp8) of MXFP4 weights from quantize_mxfp4."""
        return {k: mxfp4_to_fp8(c, e, stream) for k, (c, e) in q4.items()}

    def forward_mxfp4(self, x, q, token_ids=None, out=None, stream=None):
        """The layer on native MXFP4 expert weights q (from quantize_mxfp4)."""
        T = x.shape[0]
        inp = self.inputs
        if out is None:
            out = torch.empty((T, self.w.d), dtype=torch.bfloat16, device=self.device)
        moe_forward_mxfp4(self.plan, T, x, token_ids, inp.w_r, inp.bias, q["w13"], q["w2"], q.get("w13_sh"),
                          q.get("w2_sh"), out, self.ws, stream)
        return out

    def forward_fp8(self, x, q, token_ids=None, out=None, stream=None):
        """The layer with FP8 expert weights q (from quantize_fp8)."""
        T = x.shape[0]
        inp = self.inputs
        if out is None:
            out = torch.empty((T, self.w.d), dtype=torch.bfloat16, device=self.device)
        sh = q.get("w13_sh"), q.get("w2_sh")
        moe_forward_fp8(self.plan, T, x, token_ids, inp.w_r, inp.bias, q["w13"][0], q["w13"][1], q["w2"][0],
                        q["w2"][1], None if sh[0] is None else sh[0][0], None if sh[0] is None else sh[0][1],
                        None if sh[1] is None else sh[1][0], None if sh[1] is None else sh[1][1], out, self.ws,
                        stream)
        return out

    def forward_routed(self, x, topk_ids, topk_w, out=None, stream=None):
        T = x.shape[0]
        inp = self.inputs
        if out is None:
            out = torch.empty((T, self.w.d), dtype=torch.bfloat16, device=self.device)
        moe_forward_routed(self.plan, T, x, topk_ids, topk_w, inp.w13, inp.w2, inp.w13_sh, inp.w2_sh, out,
                           self.ws, stream)
        return out

    def route(self, x, token_ids=None, with_logits=False, stream=None):
        T = x.shape[0]
        ids = torch.empty((T, self.w.k), dtype=torch.int32, device=self.device)
        wts = torch.empty((T, self.w.k), dtype=torch.float32, device=self.device)
        logits = torch.empty((T, self.w.E), dtype=torch.float32, device=self.device) if with_logits else None
        moe_route(self.plan, T, x, token_ids, self.inputs.w_r, self.inputs.bias, ids, wts, logits, self.ws, stream)
        return (ids, wts, logits) if with_logits else (ids, wts)

    def permute(self, topk_ids, stream=None):
        T = topk_ids.shape[0]
        E, N = self.w.E, T * self.w.k
        dev = self.device
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(N, dtype=torch.int32, device=dev)
        inv = torch.empty(N, dtype=torch.int32, device=dev)
        moe_permute(self.plan, T, topk_ids, counts, offsets, perm, inv, self.ws, stream)
        return counts, offsets, perm, inv

    def views(self, T: int) -> dict:
        """Workspace intermediates of the last forward with T tokens, as tensor views."""
        v = moe_workspace_views(self.plan, T, self.ws)
        w = self.w
        N = T * w.k
        rows_h = N + w.n_shared * T
        return {
            "topk_ids": self._ws_slice(v.topk_ids, T * w.k, torch.int32).view(T, w.k),
            "topk_w": self._ws_slice(v.topk_w, T * w.k, torch.float32).view(T, w.k),
            "logits": self._ws_slice(v.logits, T * w.E, torch.float32).view(T, w.E),
            "counts": self._ws_slice(v.counts, w.E, torch.int32),
            "offsets": self._ws_slice(v.offsets, w.E + 1, torch.int32),
            "perm_tok": self._ws_slice(v.perm_tok, N, torch.int32),
            "inv": self._ws_slice(v.inv, N, torch.int32),
            "h": self._ws_slice(v.h, rows_h * w.d_ff, torch.bfloat16).view(rows_h, w.d_ff),
            "o": self._ws_slice(v.o, rows_h * w.d, torch.float32).view(rows_h, w.d),
        }

    def check_status(self, stream=None) -> int:
        return moe_check_status(self.plan, self.ws, stream)

    def set_events(self, events):
        self._events_arr = moe_plan_set_events(self.plan, events)
