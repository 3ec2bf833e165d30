"""The C-ABI library builds for sm_103a, loads without a GPU, exports every symbol the header
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from routed_expert_swiglu_gb300 import binding, build, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status|size_t|int32_t|const char\*)\s+(moe_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    declared = header_functions()
    assert len(declared) >= 14
    assert sorted(binding.EXPORTED) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_no_libcuda_link_dependency():
    out = os.popen(f"ldd {binding.LIB_PATH}").read()
    assert "libcuda.so" not in out and "libtorch" not in out


def _cfg(**kw):
    c = binding.config_for(W.V4FLASH_T64)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,code", [
    ("d", 100, 2), ("d_ff", 0, 1), ("n_experts", 600, 2), ("top_k", 9, 2), ("top_k", 0, 1),
    ("n_shared", 2, 2), ("score", 7, 1), ("max_tokens", 0, 1), ("n_groups", 3, 1),
])
def test_plan_create_rejects_bad_config(lib, field, value, code):
    plan = ctypes.c_void_p()
    st = lib.moe_plan_create(ctypes.byref(_cfg(**{field: value})), ctypes.byref(plan))
    assert st == code and not plan.value


def test_group_config_rules(lib):
    plan = ctypes.c_void_p()
    ok = _cfg(n_groups=8, topk_groups=4, group_topk=2)
    assert lib.moe_plan_create(ctypes.byref(ok), ctypes.byref(plan)) == 0
    lib.moe_plan_destroy(plan)
    for bad in (dict(n_groups=8, topk_groups=9, group_topk=2), dict(n_groups=8, topk_groups=4, group_topk=40),
                dict(n_groups=64, topk_groups=4, group_topk=2)):
        assert lib.moe_plan_create(ctypes.byref(_cfg(**bad)), ctypes.byref(plan)) != 0


def test_host_validation_without_gpu(lib):
    plan = binding.moe_plan_create(_cfg(max_tokens=64))
    need = lib.moe_workspace_bytes(plan, 64)
    assert need > 0 and lib.moe_workspace_bytes(plan, 65) == 0 and lib.moe_workspace_bytes(plan, -1) == 0
    assert lib.moe_workspace_bytes(plan, 0) > 0
    buf = ctypes.create_string_buffer(need + 4096)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    ws = ctypes.c_void_p(base)
    p16 = ctypes.c_void_p(base)  # any aligned non-null address: validation fails before use
    nul = None
    # T out of range, workspace too small, misaligned workspace, null pointers
    assert lib.moe_forward(plan, 65, p16, nul, p16, nul, p16, p16, p16, p16, p16, ws, need, nul) == 1
    assert lib.moe_forward(plan, 64, p16, nul, p16, nul, p16, p16, p16, p16, p16, ws, need - 1, nul) == 4
    assert lib.moe_forward(plan, 64, p16, nul, p16, nul, p16, p16, p16, p16, p16, ctypes.c_void_p(base + 16),
                           need, nul) == 3
    assert lib.moe_forward(plan, 64, nul, nul, p16, nul, p16, p16, p16, p16, p16, ws, need, nul) == 1
    assert lib.moe_forward(plan, 64, p16, nul, p16, nul, p16, p16, nul, p16, p16, ws, need, nul) == 1  # shared
    assert lib.moe_forward(plan, 64, ctypes.c_void_p(base + 8), nul, p16, nul, p16, p16, p16, p16, p16, ws, need,
                           nul) == 3
    assert lib.moe_route(plan, 64, p16, nul, p16, nul, nul, p16, nul, ws, need, nul) == 1
    assert lib.moe_permute(plan, 64, nul, nul, nul, nul, nul, ws, need, nul) == 1
    # T = 0 is a valid no-op: returns before any CUDA call
    assert lib.moe_forward(plan, 0, nul, nul, nul, nul, nul, nul, nul, nul, nul, nul, 0, nul) == 0
    assert lib.moe_plan_set_events(plan, None, 0) == 0
    assert lib.moe_plan_set_events(plan, p16, 3) == 1
    # 384 assignments (one 1024-assignment chunk) run the dispatch's three index steps as one
    # launch: 7
    assert lib.moe_forward_launch_count(plan, 64) == 7
    assert lib.moe_status_string(4) == b"workspace too small"
    binding.moe_plan_destroy(plan)
    big = binding.moe_plan_create(_cfg(max_tokens=8192))
    assert lib.moe_forward_launch_count(big, 8192) == 9 and lib.moe_forward_launch_count(big, 170) == 7
    assert lib.moe_forward_launch_count(big, 65) == 7
    binding.moe_plan_destroy(big)
    # at most 64 tokens over at most 64 experts the router and top-k are one launch: 6
    big = binding.moe_plan_create(_cfg(max_tokens=8192, n_experts=64))
    assert lib.moe_forward_launch_count(big, 64) == 6 and lib.moe_forward_launch_count(big, 65) == 7
    assert lib.moe_forward_launch_count(big, 171) == 9
    binding.moe_plan_destroy(big)


def test_hash_plan_requires_token_ids(lib):
    import torch
    tid = torch.zeros((16, 6), dtype=torch.int32)
    c = binding.config_for(W.V4PRO_HASH_T16384, max_tokens=8, tid2eid=tid)
    plan = binding.moe_plan_create(c)
    need = lib.moe_workspace_bytes(plan, 8)
    buf = ctypes.create_string_buffer(need + 512)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    assert lib.moe_route(plan, 8, p, None, p, None, p, p, None, p, need, None) == 1
    binding.moe_plan_destroy(plan)


def test_weight_format_validation_without_gpu(lib):
    """FP8 / MXFP4 entry points reject bad shapes, null and misaligned pointers on the host."""
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p16, nul = ctypes.c_void_p(base), None
    # quantisers: K a multiple of 32 (MXFP4), positive sizes, non-null, aligned
    assert lib.moe_quantize_mxfp4(p16, 1, 128, 100, p16, p16, nul) == 1
    assert lib.moe_quantize_mxfp4(nul, 1, 128, 128, p16, p16, nul) == 1
    assert lib.moe_quantize_mxfp4(ctypes.c_void_p(base + 2), 1, 128, 128, p16, p16, nul) == 3
    assert lib.moe_quantize_mxfp4(p16, 1, 128, 128, ctypes.c_void_p(base + 8), p16, nul) == 3
    assert lib.moe_quantize_fp8(p16, 1, 0, 128, p16, p16, nul) == 1
    assert lib.moe_quantize_fp8(ctypes.c_void_p(base + 1), 1, 128, 128, p16, p16, nul) == 3
    # conversion: tile exponents required, FP8 codes optional, K a multiple of 32
    assert lib.moe_mxfp4_to_fp8(p16, p16, 1, 128, 128, p16, nul, nul) == 1
    assert lib.moe_mxfp4_to_fp8(p16, p16, 1, 128, 96 + 8, p16, p16, nul) == 1
    assert lib.moe_mxfp4_to_fp8(p16, p16, 1, 128, 128, ctypes.c_void_p(base + 4), p16, nul) == 3
    # the native MXFP4 forward: arguments, exponent alignment, and the shape rule
    plan = binding.moe_plan_create(_cfg(max_tokens=64))
    need = lib.moe_workspace_bytes(plan, 64)
    ws_buf = ctypes.create_string_buffer(need + 4096)
    ws = ctypes.c_void_p((ctypes.addressof(ws_buf) + 255) // 256 * 256)
    w = [p16] * 8                                       # (codes, sub-block exponents) x 4; base is 256-aligned
    assert lib.moe_forward_mxfp4(plan, 65, p16, nul, p16, nul, *w, p16, ws, need, nul) == 1
    bad = list(w)
    bad[1] = nul                                        # s13
    assert lib.moe_forward_mxfp4(plan, 64, p16, nul, p16, nul, *bad, p16, ws, need, nul) == 1
    bad = list(w)
    bad[1] = ctypes.c_void_p(base + 2)                  # s13 not 4-byte aligned
    assert lib.moe_forward_mxfp4(plan, 64, p16, nul, p16, nul, *bad, p16, ws, need, nul) == 3
    bad = list(w)
    bad[2] = ctypes.c_void_p(base + 16)                 # c2 16-byte but not 32-byte aligned
    assert lib.moe_forward_mxfp4(plan, 64, p16, nul, p16, nul, *bad, p16, ws, need, nul) == 3
    bad = list(w)
    bad[4] = nul                                        # shared codes of a layer with a shared expert
    assert lib.moe_forward_mxfp4(plan, 64, p16, nul, p16, nul, *bad, p16, ws, need, nul) == 1
    assert lib.moe_forward_fp8(plan, 64, p16, nul, p16, nul, p16, nul, p16, p16, p16, p16, p16, p16, p16, ws,
                               need, nul) == 1         # e13 null
    binding.moe_plan_destroy(plan)
    toy = binding.moe_plan_create(binding.config_for(W.TOY, max_tokens=64))   # d_ff = 64
    need = lib.moe_workspace_bytes(toy, 64)
    ws_buf = ctypes.create_string_buffer(need + 4096)
    ws = ctypes.c_void_p((ctypes.addressof(ws_buf) + 255) // 256 * 256)
    assert lib.moe_forward_mxfp4(toy, 64, p16, nul, p16, nul, *w, p16, ws, need, nul) == 2
    binding.moe_plan_destroy(toy)
