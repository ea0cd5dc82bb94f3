"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_w4a16.h")


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from w4a16_mixture_experts_sigmoid_gb300 import build as build_mod
    build_mod.build()
    from w4a16_mixture_experts_sigmoid_gb300 import binding
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    from w4a16_mixture_experts_sigmoid_gb300 import binding
    assert sorted(binding.SIGNATURES) == names


def test_status_strings(lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    for code in range(8):
        assert B.moe_status_string(code) and B.moe_status_string(code) != "unknown status"
    assert B.moe_status_string(99) == "unknown status"


def test_workspace_size(lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    d = B.dims(384, 8, 7168, 2048)
    ws = B.moe_workspace_size(d, 64)
    Tk = 64 * 8
    # at least x_perm + h + y of the routed rows
    assert ws >= Tk * 7168 * 2 * 2 + Tk * 2048 * 2
    assert B.moe_workspace_size(d, 64, 2048) > ws
    assert B.moe_workspace_size(B.dims(384, 8, 7168, 2040), 64) == 0        # I not a multiple of 32
    assert B.moe_workspace_size(B.dims(2000, 8, 7168, 2048), 64) == 0       # E > 1024
    assert B.moe_workspace_size(B.dims(8, 9, 256, 128), 4) == 0             # k > E
    assert B.moe_workspace_size(B.dims(8, 2, 256, 128, 64), 4) == 0         # group != 32
    assert B.moe_workspace_size(d, -1) == 0


def test_arguments_rejected_before_any_launch(lib):
    from w4a16_mixture_experts_sigmoid_gb300 import binding as B
    L = lib
    assert L.moe_route(None, 4, 8, 2, None, None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_route(16, -1, 8, 2, 16, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_route(16, 4, 8, 9, 16, 16, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route(16, 4, 2000, 2, 16, 16, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route(16, 0, 8, 2, 16, 16, None) == B.MOE_OK                     # T == 0: no-op
    assert L.moe_sigmoid_scores(None, 4, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_permute(16, 4, 8, 2, 16, 16, 16, 16, 64, None, 16, 4096, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_permute(16, 4, 8, 2, 16, 16, 16, None, 0, None, 16, 16, 0, None) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    d = B.dims(8, 2, 256, 128)
    w = B.moe_weights_t(16, 16, 16, 16, None, None, 0)
    byref = ctypes.byref
    assert L.moe_w4a16_grouped_gemm(7, d, byref(w), 16, 4, 16, 16, 16, 4096, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_w4a16_grouped_gemm(0, B.dims(8, 2, 250, 128), byref(w), 16, 4, 16, 16, 16, 4096, 0, None) == \
        B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_w4a16_grouped_gemm(0, d, None, 16, 4, 16, 16, 16, 4096, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_w4a16_grouped_gemm(0, d, byref(w), 16, 4, 16, 16, 16, 8, 0, None) == \
        B.MOE_ERR_WORKSPACE_TOO_SMALL
    # natural-order rows on the tensor-core path need room to rewrite them: 256 + R*K*2 bytes
    assert L.moe_w4a16_grouped_gemm(0, d, byref(w), 16, 4, 16, 16, 16, 256 + 8 * 256 * 2 - 16, 0, None) == \
        B.MOE_ERR_WORKSPACE_TOO_SMALL
    bad = B.moe_weights_t(16, 16, 16 + 4, 16, None, None, 0)                  # misaligned pointer
    assert L.moe_w4a16_grouped_gemm(0, d, byref(bad), 16, 4, 16, 16, 16, 4096, 0, None) == B.MOE_ERR_INVALID_ARG
    half_shared = B.moe_weights_t(16, 16, 16, 16, 16, None, 64)
    assert L.moe_forward(d, byref(half_shared), 16, 16, 4, 16, 16, 1 << 30, 0, None) == B.MOE_ERR_INVALID_ARG
    odd_shared = B.moe_weights_t(16, 16, 16, 16, 16, 16, 96)
    assert L.moe_forward(d, byref(odd_shared), 16, 16, 4, 16, 16, 1 << 30, 0, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_forward(d, byref(w), 16, 16, 4, 16, 16, 64, 0, None) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_forward(d, byref(w), 16, 16, 1 << 24, 16, 16, 1 << 40, 0, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_shared_expert(d, byref(w), 16, 4, 16, 16, 1 << 30, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(None, 16, 16, 4, 2, 256, None, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(16, 16, 16, 4, 2, 250, None, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine_f32(None, 16, 16, 4, 2, 256, None, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine_f32(16, 16, 16, 4, 2, 250, None, 16, None) == B.MOE_ERR_INVALID_ARG
    # router projection: shape rules and null pointers, before any launch
    assert L.moe_router_logits(16, 16, 4, 384, 7000, 16, 16, 1 << 20, 0, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_router_logits(None, 16, 4, 384, 7168, 16, 16, 1 << 20, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_router_logits(16, 16, 4, 384, 7168, None, 16, 1 << 20, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_router_logits(16, 16, 4, 384, 7168, 16, 16, 16, 0, None) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_router_logits(16, 16, 0, 384, 7168, 16, 16, 0, 0, None) == B.MOE_OK
    assert L.moe_route_project(16, 16, 4, 384, 7168, 400, 16, 16, 16, 16, 1 << 20, 0, None) == \
        B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_router_workspace_size(64, 384, 7168) > L.moe_router_workspace_size(512, 384, 7168) > 0
    # offloaded bank: null tensors and a missing offsets array are refused before anything else
    hw = B.moe_weights_t(None, None, None, None, None, None, 0)
    dw = B.moe_weights_t(16, 16, 16, 16, None, None, 0)
    assert L.moe_stage_experts(B.dims(8, 2, 256, 128), byref(hw), 16, byref(dw), None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_stage_experts(B.dims(8, 2, 256, 128), byref(dw), None, byref(dw), None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward_offload(B.dims(8, 2, 256, 128), byref(dw), byref(hw), 16, 16, 4, 16, 16, 1 << 20, 0,
                                 None) == B.MOE_ERR_INVALID_ARG
    d2 = B.dims(384, 8, 7168, 2048)
    assert L.moe_workspace_size(d2, 64, 0, B.MOE_FLAG_ROUTER_PROJECT) > L.moe_workspace_size(d2, 64, 0, 0)
    assert L.moe_check_status(None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_debug_expire_wait(None, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward_host(d, byref(w), None, 16, 4, 16, 16, 1 << 30, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_rmsnorm(None, 4, 256, 1e-6, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_rmsnorm(16, 4, 250, 1e-6, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_rmsnorm(16, 4, 256, -1.0, 16, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_rmsnorm(16, 0, 256, 1e-6, 16, None) == B.MOE_OK                # T == 0: no-op
    two = (B.moe_weights_t * 2)(w, w)
    lg = (ctypes.c_void_p * 2)(16, 16)
    assert L.moe_stack_forward(d, two, 0, lg, 16, 4, 1e-6, 16, 16, 1 << 30, 0, None) == B.MOE_ERR_INVALID_ARG
    mixed = (B.moe_weights_t * 2)(w, B.moe_weights_t(16, 16, 16, 16, 16, 16, 64))   # shared_I differs
    assert L.moe_stack_forward(d, mixed, 2, lg, 16, 4, 1e-6, 16, 16, 1 << 30, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_stack_forward(d, two, 2, (ctypes.c_void_p * 2)(16, None), 16, 4, 1e-6, 16, 16, 1 << 30, 0,
                               None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_stack_forward(d, two, 2, lg, 16, 4, 1e-6, 16, 16, 4096, 0, None) == \
        B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_stack_workspace_size(d, 4, 0, 0) == L.moe_workspace_size(d, 4, 0, 0) + 3 * 2048
    assert L.moe_launch_count() == 0                                           # nothing launched
