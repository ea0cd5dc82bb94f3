"""ctypes binding of libmoe_w4a16.so: the C ABI of include/moe_w4a16.h, same names.

Argument marshalling only: tensors become device pointers, the stream
defaults to PyTorch's current stream, and a non-zero status raises MoeError.
Every step of the layer runs in the library's CUDA kernels; there is no
other implementation behind these functions, and loading fails loudly if the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, POINTER, Structure, c_char_p, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_w4a16.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_DEVICE_BOUNDS = 6
MOE_ERR_UNSUPPORTED_DEVICE = 7

MOE_GEMM_GATEUP_SILU = 0
MOE_GEMM_DOWN = 1

MOE_FLAG_GEMM_SIMT = 0x1
MOE_FLAG_A_SMEM = 0x2
MOE_FLAG_ROWS_MMA_ORDER = 0x4
MOE_FLAG_OUT_F32 = 0x8
MOE_FLAG_GEMM_PAIR = 0x10
MOE_FLAG_ROUTER_PROJECT = 0x20
MOE_PERMUTE_STATIC_SCRATCH_BYTES = 1 << 20


def MOE_FLAG_TOKENS_PER_TILE(n: int) -> int:
    return (int(n) & 0xFF) << 8


class moe_dims_t(Structure):
    _fields_ = [("E", c_int32), ("top_k", c_int32), ("H", c_int32), ("I", c_int32), ("group", c_int32)]


class moe_weights_t(Structure):
    _fields_ = [("w13_packed", c_void_p), ("w13_scale", c_void_p), ("w2_packed", c_void_p),
                ("w2_scale", c_void_p), ("shared_wgu", c_void_p), ("shared_wd", c_void_p),
                ("shared_I", c_int32)]


class moe_weights_fp4_t(Structure):
    _fields_ = [("w13_packed", c_void_p), ("w13_scale", c_void_p), ("w13_gscale", c_void_p),
                ("w2_packed", c_void_p), ("w2_scale", c_void_p), ("w2_gscale", c_void_p),
                ("shared_wgu", c_void_p), ("shared_wd", c_void_p), ("shared_I", c_int32)]


# name -> (restype, argtypes); every symbol include/moe_w4a16.h declares
SIGNATURES = {
    "moe_status_string": (c_char_p, [c_int32]),
    "moe_workspace_size": (c_size_t, [moe_dims_t, c_int32, c_int32, c_uint32]),
    "moe_route": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "moe_sigmoid_scores": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p]),
    "moe_router_workspace_size": (c_size_t, [c_int32, c_int32, c_int32]),
    "moe_router_logits": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_size_t,
                                    c_uint32, c_void_p]),
    "moe_route_project": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_fp4_grouped_gemm": (c_int32, [c_int32, moe_dims_t, POINTER(moe_weights_fp4_t), c_void_p, c_int32,
                                       c_void_p, c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_forward_fp4": (c_int32, [moe_dims_t, POINTER(moe_weights_fp4_t), c_void_p, c_void_p, c_int32, c_void_p,
                                  c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_stage_experts": (c_int32, [moe_dims_t, POINTER(moe_weights_t), c_void_p, POINTER(moe_weights_t), c_void_p]),
    "moe_forward_offload": (c_int32, [moe_dims_t, POINTER(moe_weights_t), POINTER(moe_weights_t), c_void_p, c_void_p,
                                      c_int32, c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_forward_project": (c_int32, [moe_dims_t, POINTER(moe_weights_t), c_void_p, c_void_p, c_int32, c_void_p,
                                      c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_permute": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_permute_static_scratch": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_int32, c_void_p, c_void_p, c_uint32, c_void_p]),
    "moe_w4a16_grouped_gemm": (c_int32, [c_int32, moe_dims_t, POINTER(moe_weights_t), c_void_p, c_int32,
                                         c_void_p, c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_shared_expert": (c_int32, [moe_dims_t, POINTER(moe_weights_t), c_void_p, c_int32, c_void_p,
                                    c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_combine": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p,
                              c_void_p, c_void_p]),
    "moe_combine_f32": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                  c_void_p, c_void_p]),
    "moe_forward": (c_int32, [moe_dims_t, POINTER(moe_weights_t), c_void_p, c_void_p, c_int32, c_void_p,
                              c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_host_staging_size": (c_size_t, [moe_dims_t, c_int32]),
    "moe_forward_host": (c_int32, [moe_dims_t, POINTER(moe_weights_t), c_void_p, c_void_p, c_int32,
                                   c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_rmsnorm": (c_int32, [c_void_p, c_int32, c_int32, c_float, c_void_p, c_void_p]),
    "moe_stack_workspace_size": (c_size_t, [moe_dims_t, c_int32, c_int32, c_uint32]),
    "moe_stack_forward": (c_int32, [moe_dims_t, POINTER(moe_weights_t), c_int32, POINTER(c_void_p), c_void_p,
                                    c_int32, c_float, c_void_p, c_void_p, c_size_t, c_uint32, c_void_p]),
    "moe_check_status": (c_int32, [c_void_p, c_void_p]),
    "moe_launch_count": (c_uint64, []),
    "moe_debug_expire_wait": (c_int32, [c_void_p, c_int64, c_void_p]),
}

_lib = None


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = int(code)
        super().__init__(f"{what}: {moe_status_string(code)} (status {code})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _dptr(t):
    if t is not None and not isinstance(t, int) and not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return _ptr(t)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)


def dims(E: int, top_k: int, H: int, I: int, group: int = 32) -> moe_dims_t:
    return moe_dims_t(E, top_k, H, I, group)


def weights(w13, s13, w2, s2, shared_wgu=None, shared_wd=None) -> moe_weights_t:
    shared_I = 0 if shared_wd is None else int(shared_wd.shape[1])
    return moe_weights_t(_dptr(w13), _dptr(s13), _dptr(w2), _dptr(s2), _dptr(shared_wgu), _dptr(shared_wd),
                         shared_I)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


# ---------------------------------------------------------------------------
# the entry points
# ---------------------------------------------------------------------------

def moe_status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


def moe_workspace_size(d: moe_dims_t, T: int, shared_I: int = 0, flags: int = 0) -> int:
    return int(load().moe_workspace_size(d, T, shared_I, flags))


def moe_host_staging_size(d: moe_dims_t, T: int) -> int:
    return int(load().moe_host_staging_size(d, T))


def moe_route(logits, T: int, E: int, k: int, topk_ids, topk_w, stream=None) -> None:
    _check(load().moe_route(_dptr(logits), T, E, k, _dptr(topk_ids), _dptr(topk_w), _stream(stream)), "moe_route")


def moe_router_workspace_size(T: int, E: int, H: int) -> int:
    return int(load().moe_router_workspace_size(T, E, H))


def moe_router_logits(x, w_gate, T: int, E: int, H: int, logits, ws, flags: int = 0, stream=None) -> None:
    _check(load().moe_router_logits(_dptr(x), _dptr(w_gate), T, E, H, _dptr(logits), _dptr(ws), _nbytes(ws), flags,
                                    _stream(stream)), "moe_router_logits")


def moe_route_project(x, w_gate, T: int, E: int, H: int, k: int, logits, topk_ids, topk_w, ws, flags: int = 0,
                      stream=None) -> None:
    _check(load().moe_route_project(_dptr(x), _dptr(w_gate), T, E, H, k, _dptr(logits), _dptr(topk_ids),
                                    _dptr(topk_w), _dptr(ws), _nbytes(ws), flags, _stream(stream)),
           "moe_route_project")


def host_weights(w13, s13, w2, s2) -> moe_weights_t:
    """moe_weights_t of a routed bank in page-locked host memory (pinned CPU tensors): the library
    reads it over the host link (moe_stage_experts, moe_forward_offload)."""
    for t in (w13, s13, w2, s2):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("a host bank is made of pinned CPU tensors")
    return moe_weights_t(_ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), None, None, 0)


def moe_stage_experts(d: moe_dims_t, host_w: moe_weights_t, expert_offsets, dev_w: moe_weights_t,
                      stream=None) -> None:
    _check(load().moe_stage_experts(d, ctypes.byref(host_w), _dptr(expert_offsets), ctypes.byref(dev_w),
                                    _stream(stream)), "moe_stage_experts")


def moe_forward_offload(d: moe_dims_t, host_w: moe_weights_t, dev_w: moe_weights_t, x, logits, T: int, out, ws,
                        flags: int = 0, stream=None) -> None:
    _check(load().moe_forward_offload(d, ctypes.byref(host_w), ctypes.byref(dev_w), _dptr(x), _dptr(logits), T,
                                      _dptr(out), _dptr(ws), _nbytes(ws), flags, _stream(stream)),
           "moe_forward_offload")


def weights_fp4(w13, s13, g13, w2, s2, g2, sh_gu=None, sh_d=None) -> moe_weights_fp4_t:
    """moe_weights_fp4_t of device tensors (scales uint8, matrix scales fp32 [E])."""
    Is = 0 if sh_d is None else int(sh_d.shape[1])
    return moe_weights_fp4_t(_dptr(w13), _dptr(s13), _dptr(g13), _dptr(w2), _dptr(s2), _dptr(g2), _dptr(sh_gu),
                             _dptr(sh_d), Is)


def moe_fp4_grouped_gemm(op: int, d: moe_dims_t, w: moe_weights_fp4_t, a_rows, T: int, expert_offsets, out_rows,
                         ws, flags: int = 0, stream=None) -> None:
    _check(load().moe_fp4_grouped_gemm(op, d, ctypes.byref(w), _dptr(a_rows), T, _dptr(expert_offsets),
                                       _dptr(out_rows), _dptr(ws), _nbytes(ws), flags, _stream(stream)),
           "moe_fp4_grouped_gemm")


def moe_forward_fp4(d: moe_dims_t, w: moe_weights_fp4_t, x, logits, T: int, out, ws, flags: int = 0,
                    stream=None) -> None:
    _check(load().moe_forward_fp4(d, ctypes.byref(w), _dptr(x), _dptr(logits), T, _dptr(out), _dptr(ws), _nbytes(ws),
                                  flags, _stream(stream)), "moe_forward_fp4")


def moe_forward_project(d: moe_dims_t, w: moe_weights_t, w_gate, x, T: int, out, ws, flags: int = 0,
                        stream=None) -> None:
    _check(load().moe_forward_project(d, ctypes.byref(w), _dptr(w_gate), _dptr(x), T, _dptr(out), _dptr(ws),
                                      _nbytes(ws), flags, _stream(stream)), "moe_forward_project")


def moe_sigmoid_scores(logits, n: int, scores, stream=None) -> None:
    _check(load().moe_sigmoid_scores(_dptr(logits), n, _dptr(scores), _stream(stream)), "moe_sigmoid_scores")


def moe_permute(topk_ids, T: int, E: int, k: int, expert_offsets, sorted_token_ids, inv_perm, x, H: int,
                x_perm, ws, flags: int = 0, stream=None) -> None:
    _check(load().moe_permute(_dptr(topk_ids), T, E, k, _dptr(expert_offsets), _dptr(sorted_token_ids),
                              _dptr(inv_perm), _dptr(x), H, _dptr(x_perm), _dptr(ws), _nbytes(ws), flags,
                              _stream(stream)), "moe_permute")


def moe_permute_static_scratch(topk_ids, T: int, E: int, k: int, expert_offsets, sorted_token_ids, inv_perm, x,
                               H: int, x_perm, status, flags: int = 0, stream=None) -> None:
    """moe_permute with the library's own fixed histogram scratch: no workspace, nothing allocated."""
    _check(load().moe_permute_static_scratch(_dptr(topk_ids), T, E, k, _dptr(expert_offsets),
                                             _dptr(sorted_token_ids), _dptr(inv_perm), _dptr(x), H, _dptr(x_perm),
                                             _dptr(status), flags, _stream(stream)), "moe_permute_static_scratch")


def moe_w4a16_grouped_gemm(op: int, d: moe_dims_t, w: moe_weights_t, a_rows, T: int, expert_offsets, out_rows,
                           ws, flags: int = 0, stream=None) -> None:
    _check(load().moe_w4a16_grouped_gemm(op, d, ctypes.byref(w), _dptr(a_rows), T, _dptr(expert_offsets),
                                         _dptr(out_rows), _dptr(ws), _nbytes(ws), flags, _stream(stream)),
           "moe_w4a16_grouped_gemm")


def moe_shared_expert(d: moe_dims_t, w: moe_weights_t, x, T: int, out, ws, flags: int = 0, stream=None) -> None:
    _check(load().moe_shared_expert(d, ctypes.byref(w), _dptr(x), T, _dptr(out), _dptr(ws), _nbytes(ws), flags,
                                    _stream(stream)), "moe_shared_expert")


def moe_combine(y_rows, inv_perm, topk_w, T: int, k: int, H: int, addend, out, stream=None) -> None:
    _check(load().moe_combine(_dptr(y_rows), _dptr(inv_perm), _dptr(topk_w), T, k, H, _dptr(addend), _dptr(out),
                              _stream(stream)), "moe_combine")


def moe_combine_f32(y_rows, inv_perm, topk_w, T: int, k: int, H: int, addend, out, stream=None) -> None:
    _check(load().moe_combine_f32(_dptr(y_rows), _dptr(inv_perm), _dptr(topk_w), T, k, H, _dptr(addend), _dptr(out),
                                  _stream(stream)), "moe_combine_f32")


def moe_forward(d: moe_dims_t, w: moe_weights_t, x, logits, T: int, out, ws, flags: int = 0, stream=None) -> None:
    _check(load().moe_forward(d, ctypes.byref(w), _dptr(x), _dptr(logits), T, _dptr(out), _dptr(ws), _nbytes(ws),
                              flags, _stream(stream)), "moe_forward")


def moe_forward_host(d: moe_dims_t, w: moe_weights_t, x_host, logits_host, T: int, out_host, ws, flags: int = 0,
                     stream=None) -> None:
    """x_host, logits_host, out_host: CPU tensors (pinned for asynchronous copies)."""
    for t in (x_host, logits_host, out_host):
        if t.is_cuda:
            raise ValueError("moe_forward_host takes host tensors")
    _check(load().moe_forward_host(d, ctypes.byref(w), _ptr(x_host), _ptr(logits_host), T, _ptr(out_host),
                                   _dptr(ws), _nbytes(ws), flags, _stream(stream)), "moe_forward_host")


def moe_rmsnorm(x, T: int, H: int, eps: float, out, stream=None) -> None:
    _check(load().moe_rmsnorm(_dptr(x), T, H, eps, _dptr(out), _stream(stream)), "moe_rmsnorm")


def moe_stack_workspace_size(d: moe_dims_t, T: int, shared_I: int = 0, flags: int = 0) -> int:
    return int(load().moe_stack_workspace_size(d, T, shared_I, flags))


def moe_stack_forward(d: moe_dims_t, layers, logits, x, T: int, eps: float, out, ws, flags: int = 0,
                      stream=None) -> None:
    """layers: list of moe_weights_t; logits: list of device tensors fp32 [T][E], one per layer."""
    L = len(layers)
    if len(logits) != L:
        raise ValueError("one logits tensor per layer")
    arr = (moe_weights_t * L)(*layers)
    lp = (c_void_p * L)(*[_dptr(t) for t in logits])
    _check(load().moe_stack_forward(d, arr, L, lp, _dptr(x), T, eps, _dptr(out), _dptr(ws), _nbytes(ws), flags,
                                    _stream(stream)), "moe_stack_forward")


def moe_check_status(ws, stream=None) -> int:
    """Synchronise, read and reset the device status word; returns the code (0 = no error)."""
    return int(load().moe_check_status(_dptr(ws), _stream(stream)))


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


def moe_debug_expire_wait(ws, timeout_ns: int, stream=None) -> None:
    _check(load().moe_debug_expire_wait(_dptr(ws), timeout_ns, _stream(stream)), "moe_debug_expire_wait")
