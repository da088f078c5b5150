"""ctypes binding of ``libmoe_b300.so`` (the C ABI in include/moe_b300.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Functions take torch tensors (device memory owned by the
caller) and launch on the current torch CUDA stream unless ``stream`` is
given.  There is no CPU fallback: if the library is missing, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_F32, MOE_BF16, MOE_FP8 = 0, 1, 2
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
          6: "MOE_ERR_DEVICE_CHECK"}

EXPORTED = ("moe_workspace_size", "moe_pack_weights", "moe_route",
            "moe_permute", "moe_expert_ffn", "moe_combine", "moe_update_bias",
            "moe_get_device_error", "moe_status_string",
            "moe_last_error_detail", "moe_last_launch_count",
            "moe_route_noalloc", "moe_selftest_wait_timeout",
            "moe_route_grouped", "moe_fp8_weight_bytes",
            "moe_pack_weights_fp8", "moe_x_perm_bytes", "moe_expert_ffn_part",
            "moe_backward_workspace_size", "moe_backward",
            "moe_expert_ffn_train")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int),
                ("n_routed", ctypes.c_int), ("top_k", ctypes.c_int),
                ("n_shared", ctypes.c_int), ("d_ff", ctypes.c_int),
                ("dtype", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m mixture_experts_layer_gemms_b300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z, V = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    SP = ctypes.POINTER(MoeShape)
    sig = {
        "moe_workspace_size": [SP, ctypes.POINTER(ctypes.c_size_t)],
        "moe_pack_weights": [SP, P, P, P, P, P, P, P, P, V],
        "moe_route": [SP, P, P, P, P, P, P, P, Z, V],
        "moe_permute": [SP, P, P, P, P, P, P, P, P, Z, V],
        "moe_expert_ffn": [SP, P, P, P, P, P, P, P, P, P, P, Z, V],
        "moe_combine": [SP, P, P, P, P, P, P, I, V],
        "moe_update_bias": [I, P, ctypes.c_longlong, ctypes.c_float, P, V],
        "moe_get_device_error": [V],
        "moe_status_string": [I],
        "moe_last_error_detail": [],
        "moe_last_launch_count": [],
        "moe_route_noalloc": [SP, P, P, P, P, P, P, V],
        "moe_selftest_wait_timeout": [ctypes.c_uint, V],
        "moe_route_grouped": [SP, I, I, P, P, P, P, P, P, P, Z, V],
        "moe_fp8_weight_bytes": [SP, I, ctypes.POINTER(ctypes.c_size_t)],
        "moe_pack_weights_fp8": [SP, P, P, P, P, P, P, P, P, P, P, V],
        "moe_x_perm_bytes": [SP, ctypes.POINTER(ctypes.c_size_t)],
        "moe_expert_ffn_part": [SP, I, P, P, P, P, P, P, P, P, P, P, Z, V],
        "moe_backward_workspace_size": [SP, ctypes.POINTER(ctypes.c_size_t)],
        "moe_backward": [SP] + [P] * 22 + [I, P, Z, V],
        "moe_expert_ffn_train": [SP] + [P] * 12 + [Z, V],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_last_error_detail.restype = ctypes.c_char_p
    return lib


LIB = _load()


def _check(status: int, where: str) -> None:
    if status != 0:
        detail = LIB.moe_last_error_detail().decode(errors="replace")
        raise MoEError(status, where, detail)


def last_launch_count() -> int:
    """Kernel launches issued by the previous successful call."""
    return int(LIB.moe_last_launch_count())


def make_shape(T, d, n_routed, top_k, n_shared, d_ff, dtype) -> MoeShape:
    if isinstance(dtype, torch.dtype):
        dt = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}[dtype]
    else:
        dt = {"f32": MOE_F32, "bf16": MOE_BF16, "fp8": MOE_FP8}.get(dtype,
                                                                 dtype)
    return MoeShape(int(T), int(d), int(n_routed), int(top_k), int(n_shared),
                    int(d_ff), int(dt))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def workspace_size(shape: MoeShape) -> int:
    n = ctypes.c_size_t(0)
    _check(LIB.moe_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
           "moe_workspace_size")
    return int(n.value)


def pack_weights(shape, w_gate, w_up, ws_gate, ws_up, ws_down, w_gu_packed,
                 ws_gu_packed, ws_down_packed, stream=None) -> None:
    _check(LIB.moe_pack_weights(ctypes.byref(shape), _ptr(w_gate), _ptr(w_up),
                                _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down),
                                _ptr(w_gu_packed), _ptr(ws_gu_packed),
                                _ptr(ws_down_packed), _stream(stream)),
           "moe_pack_weights")


def fp8_weight_bytes(shape, which: int) -> int:
    """Bytes of a packed e4m3 weight buffer (0 routed gate/up, 1 routed
    down, 2 shared gate/up, 3 shared down)."""
    n = ctypes.c_size_t(0)
    _check(LIB.moe_fp8_weight_bytes(ctypes.byref(shape), int(which),
                                    ctypes.byref(n)), "moe_fp8_weight_bytes")
    return int(n.value)


def x_perm_bytes(shape) -> int:
    n = ctypes.c_size_t(0)
    _check(LIB.moe_x_perm_bytes(ctypes.byref(shape), ctypes.byref(n)),
           "moe_x_perm_bytes")
    return int(n.value)


def pack_weights_fp8(shape, w_gate, w_up, w_down, ws_gate, ws_up, ws_down,
                     w_gu8, w_down8, ws_gu8, ws_down8, stream=None) -> None:
    _check(LIB.moe_pack_weights_fp8(
        ctypes.byref(shape), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
        _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), _ptr(w_gu8), _ptr(w_down8),
        _ptr(ws_gu8), _ptr(ws_down8), _stream(stream)), "moe_pack_weights_fp8")


def route(shape, u, centroids, bias, topk_idx, topk_gate, counts, workspace,
          stream=None) -> None:
    _check(LIB.moe_route(ctypes.byref(shape), _ptr(u), _ptr(centroids),
                         _ptr(bias), _ptr(topk_idx), _ptr(topk_gate),
                         _ptr(counts), _ptr(workspace),
                         workspace.numel() * workspace.element_size(),
                         _stream(stream)), "moe_route")


def route_grouped(shape, n_groups, topk_groups, u, centroids, bias, topk_idx,
                  topk_gate, counts, workspace, stream=None) -> None:
    """moe_route restricted to each token's topk_groups best expert groups."""
    _check(LIB.moe_route_grouped(ctypes.byref(shape), int(n_groups),
                                 int(topk_groups), _ptr(u), _ptr(centroids),
                                 _ptr(bias), _ptr(topk_idx), _ptr(topk_gate),
                                 _ptr(counts), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "moe_route_grouped")


def route_noalloc(shape, u, centroids, bias, topk_idx, topk_gate, counts,
                  stream=None) -> None:
    """moe_route without a workspace (library-owned 1 MiB scratch); see
    include/moe_b300.h for who needs it and its limits."""
    _check(LIB.moe_route_noalloc(ctypes.byref(shape), _ptr(u),
                                 _ptr(centroids), _ptr(bias), _ptr(topk_idx),
                                 _ptr(topk_gate), _ptr(counts),
                                 _stream(stream)), "moe_route_noalloc")


def permute(shape, u, topk_idx, counts, offsets, perm, inv, x_perm, workspace,
            stream=None) -> None:
    _check(LIB.moe_permute(ctypes.byref(shape), _ptr(u), _ptr(topk_idx),
                           _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                           _ptr(x_perm), _ptr(workspace),
                           workspace.numel() * workspace.element_size(),
                           _stream(stream)), "moe_permute")


def expert_ffn(shape, x_perm, offsets, w_gu_packed, w_down, u, ws_gu_packed,
               ws_down_packed, y_perm, y_shared, workspace, stream=None) -> None:
    _check(LIB.moe_expert_ffn(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets),
                              _ptr(w_gu_packed), _ptr(w_down), _ptr(u),
                              _ptr(ws_gu_packed), _ptr(ws_down_packed),
                              _ptr(y_perm), _ptr(y_shared), _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _stream(stream)), "moe_expert_ffn")


def expert_ffn_train(shape, x_perm, offsets, w_gu_packed, w_down, u,
                     ws_gu_packed, ws_down_packed, y_perm, y_shared, act,
                     act_shared, workspace, stream=None) -> None:
    """expert_ffn that also stores the gate/up pre-activations (fp16) in act
    [T*K, 2*d_ff] and act_shared [T, 2*S*d_ff] for backward()."""
    _check(LIB.moe_expert_ffn_train(
        ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(w_gu_packed),
        _ptr(w_down), _ptr(u), _ptr(ws_gu_packed), _ptr(ws_down_packed),
        _ptr(y_perm), _ptr(y_shared), _ptr(act), _ptr(act_shared),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "moe_expert_ffn_train")


def expert_ffn_part(shape, part, x_perm, offsets, w_gu_packed, w_down, u,
                    ws_gu_packed, ws_down_packed, y_perm, y_shared, workspace,
                    stream=None) -> None:
    """part 1: routed experts only; part 2: shared experts only (may run on
    another stream beside the routing, the permute and a part-1 call)."""
    _check(LIB.moe_expert_ffn_part(
        ctypes.byref(shape), int(part), _ptr(x_perm), _ptr(offsets),
        _ptr(w_gu_packed), _ptr(w_down), _ptr(u), _ptr(ws_gu_packed),
        _ptr(ws_down_packed), _ptr(y_perm), _ptr(y_shared), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "moe_expert_ffn_part")


def backward_workspace_size(shape: MoeShape) -> int:
    n = ctypes.c_size_t()
    _check(LIB.moe_backward_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return n.value


def backward(shape, dh, u, centroids, topk_idx, topk_gate, offsets, inv,
             y_perm, w_gu_packed, w_down, ws_gu_packed, ws_down_packed, du, dE,
             dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down, workspace,
             stream=None, act=None, act_shared=None) -> None:
    """Gradients of the layer for dh; the weight gradients' dtype (fp32 or
    bf16) is taken from dw_gate.  act / act_shared: the pre-activations of
    expert_ffn_train on the same batch (else they are recomputed)."""
    gd = MOE_BF16 if dw_gate.dtype == torch.bfloat16 else MOE_F32
    _check(LIB.moe_backward(
        ctypes.byref(shape), _ptr(dh), _ptr(u), _ptr(centroids),
        _ptr(topk_idx), _ptr(topk_gate), _ptr(offsets), _ptr(inv),
        _ptr(y_perm), _ptr(act), _ptr(act_shared), _ptr(w_gu_packed),
        _ptr(w_down), _ptr(ws_gu_packed),
        _ptr(ws_down_packed), _ptr(du), _ptr(dE), _ptr(dw_gate), _ptr(dw_up),
        _ptr(dw_down), _ptr(dws_gate), _ptr(dws_up), _ptr(dws_down), gd,
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "moe_backward")


def combine(shape, u, y_perm, y_shared, inv, topk_gate, h, stream=None) -> None:
    h_dt = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}[h.dtype]
    _check(LIB.moe_combine(ctypes.byref(shape), _ptr(u), _ptr(y_perm),
                           _ptr(y_shared), _ptr(inv), _ptr(topk_gate), _ptr(h),
                           h_dt, _stream(stream)), "moe_combine")


def update_bias(n_routed, counts, total_assign, gamma, bias,
                stream=None) -> None:
    _check(LIB.moe_update_bias(int(n_routed), _ptr(counts), int(total_assign),
                               float(gamma), _ptr(bias), _stream(stream)),
           "moe_update_bias")


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> None:
    """Launch a kernel whose bounded wait must give up (see the header)."""
    _check(LIB.moe_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "moe_selftest_wait_timeout")


def get_device_error(stream=None) -> None:
    _check(LIB.moe_get_device_error(_stream(stream)), "device")
