"""ctypes binding of libhylo_kl.so (include/hylo_kl.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no arithmetic of the
loss: it checks tensor dtypes/shapes/devices, passes raw device pointers, sizes and the
current CUDA stream, and raises HyloError on a non-OK status. There is no fallback: if the
shared library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhylo_kl.so")

STATUS = {
    0: "HYLO_OK",
    -1: "HYLO_ERR_NULL",
    -2: "HYLO_ERR_DIM",
    -3: "HYLO_ERR_ALIGN",
    -4: "HYLO_ERR_TAU",
    -5: "HYLO_ERR_WORKSPACE",
    -6: "HYLO_ERR_CUDA",
    -7: "HYLO_ERR_TIMEOUT",
    -8: "HYLO_ERR_ARCH",
}

EXPORTS = ("hylo_kl_workspace_bytes", "hylo_kl_forward", "hylo_kl_backward", "hylo_kl_sync_status",
           "hylo_kl_workspace_bytes_split", "hylo_kl_backward_split",
           "hylo_kl_last_error", "hylo_kl_forward_noalloc", "hylo_kl_selftest_wait_timeout",
           "hylo_fused_kl_logits", "hylo_ild_loss")


class HyloError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Loads the in-tree shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m hybrid_upcycling_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    i64, f32, vp, sz = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    L.hylo_kl_workspace_bytes.argtypes = [i64, i64, i64, i64, i64]
    L.hylo_kl_workspace_bytes.restype = sz
    L.hylo_kl_forward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, i64, vp, vp, vp, vp, vp, vp, sz, vp]
    L.hylo_kl_forward.restype = ctypes.c_int
    L.hylo_kl_backward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, i64, vp, vp, vp, f32, vp, vp, vp, sz, vp]
    L.hylo_kl_backward.restype = ctypes.c_int
    L.hylo_kl_workspace_bytes_split.argtypes = [i64, i64, i64, i64, i64]
    L.hylo_kl_workspace_bytes_split.restype = sz
    L.hylo_kl_backward_split.argtypes = list(L.hylo_kl_backward.argtypes)
    L.hylo_kl_backward_split.restype = ctypes.c_int
    L.hylo_kl_forward_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, i64, vp, vp, vp, vp, vp, vp]
    L.hylo_kl_forward_noalloc.restype = ctypes.c_int
    L.hylo_fused_kl_logits.argtypes = [vp, vp, i64, i64, i64, f32, f32, vp, vp, vp, vp, vp, vp]
    L.hylo_fused_kl_logits.restype = ctypes.c_int
    L.hylo_ild_loss.argtypes = [vp, vp, i64, i64, i64, f32, vp, vp, vp, vp]
    L.hylo_ild_loss.restype = ctypes.c_int
    L.hylo_kl_selftest_wait_timeout.argtypes = [ctypes.c_int, vp]
    L.hylo_kl_selftest_wait_timeout.restype = ctypes.c_int
    L.hylo_kl_sync_status.argtypes = [vp]
    L.hylo_kl_sync_status.restype = ctypes.c_int
    L.hylo_kl_last_error.argtypes = []
    L.hylo_kl_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int) -> None:
    if status != 0:
        msg = load().hylo_kl_last_error()
        raise HyloError(status, msg.decode() if msg else "")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dims(h_s, W_s, h_t, W_t):
    for name, t in (("h_s", h_s), ("W_s", W_s), ("h_t", h_t), ("W_t", W_t)):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D bfloat16 tensor")
    N, d_s = h_s.shape
    V = W_s.shape[0]
    d_t = h_t.shape[1]
    if h_t.shape[0] != N or W_s.shape[1] != d_s or tuple(W_t.shape) != (V, d_t):
        raise ValueError(f"shape mismatch: h_s {tuple(h_s.shape)} W_s {tuple(W_s.shape)} "
                         f"h_t {tuple(h_t.shape)} W_t {tuple(W_t.shape)}")
    return N, d_s, d_t, V


def hylo_kl_workspace_bytes(N: int, d_s: int, d_t: int, V: int, token_chunk: int = 4096) -> int:
    return int(load().hylo_kl_workspace_bytes(N, d_s, d_t, V, token_chunk))


def hylo_kl_forward(h_s, W_s, h_t, W_t, tau: float, token_chunk: int, kl, lse_s, lse_t, loss, workspace,
                    stream=None, lse_gap=None) -> None:
    """lse_gap (optional fp32 [N]) receives the precise lse_s - lse_t for hylo_kl_backward."""
    N, d_s, d_t, V = _dims(h_s, W_s, h_t, W_t)
    _check(load().hylo_kl_forward(_ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(W_t), N, d_s, d_t, V, float(tau),
                                  int(token_chunk), _ptr(kl), _ptr(lse_s), _ptr(lse_t), _ptr(lse_gap), _ptr(loss),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def hylo_kl_backward(h_s, W_s, h_t, W_t, tau: float, token_chunk: int, lse_s, lse_t, grad_scale: float, dh_s,
                     dW_s, workspace, stream=None, lse_gap=None) -> None:
    """lse_gap (optional) is the forward's precise lse_s - lse_t; None uses lse_s - lse_t."""
    N, d_s, d_t, V = _dims(h_s, W_s, h_t, W_t)
    _check(load().hylo_kl_backward(_ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(W_t), N, d_s, d_t, V, float(tau),
                                   int(token_chunk), _ptr(lse_s), _ptr(lse_t), _ptr(lse_gap), float(grad_scale),
                                   _ptr(dh_s), _ptr(dW_s), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)))


def hylo_kl_workspace_bytes_split(N: int, d_s: int, d_t: int, V: int, token_chunk: int = 4096) -> int:
    return int(load().hylo_kl_workspace_bytes_split(N, d_s, d_t, V, token_chunk))


def hylo_kl_backward_split(h_s, W_s, h_t, W_t, tau: float, token_chunk: int, lse_s, lse_t, grad_scale: float,
                           dh_s, dW_s, workspace, stream=None, lse_gap=None) -> None:
    """hylo_kl_backward with G kept as two bf16 terms (workspace: hylo_kl_workspace_bytes_split)."""
    N, d_s, d_t, V = _dims(h_s, W_s, h_t, W_t)
    _check(load().hylo_kl_backward_split(_ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(W_t), N, d_s, d_t, V, float(tau),
                                         int(token_chunk), _ptr(lse_s), _ptr(lse_t), _ptr(lse_gap), float(grad_scale),
                                         _ptr(dh_s), _ptr(dW_s), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))


def hylo_kl_forward_noalloc(h_s, W_s, h_t, W_t, tau: float, token_chunk: int, kl, lse_s, lse_t, loss,
                            stream=None, lse_gap=None) -> None:
    """hylo_kl_forward without a workspace: the library's built-in scratch is used instead."""
    N, d_s, d_t, V = _dims(h_s, W_s, h_t, W_t)
    _check(load().hylo_kl_forward_noalloc(_ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(W_t), N, d_s, d_t, V, float(tau),
                                          int(token_chunk), _ptr(kl), _ptr(lse_s), _ptr(lse_t), _ptr(lse_gap),
                                          _ptr(loss), _stream(stream)))


def hylo_fused_kl_logits(z_s, z_t, tau: float, grad_scale: float, kl, lse_s, lse_t, loss, dz_s=None,
                         stream=None) -> None:
    """Fused KL on bf16 logits z_s, z_t [N, V] (row stride = z.stride(0)); dz_s optional."""
    for name, t in (("z_s", z_s), ("z_t", z_t)):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name} must be a 2-D bfloat16 tensor with unit column stride")
    if z_s.shape != z_t.shape or z_s.stride(0) != z_t.stride(0):
        raise ValueError("z_s and z_t must have the same shape and row stride")
    if dz_s is not None and (dz_s.dtype != torch.bfloat16 or dz_s.shape != z_s.shape or dz_s.stride(0) != z_s.stride(0)):
        raise ValueError("dz_s must be bfloat16 with the shape and row stride of z_s")
    N, V = z_s.shape
    _check(load().hylo_fused_kl_logits(_ptr(z_s), _ptr(z_t), N, V, z_s.stride(0), float(tau), float(grad_scale),
                                       _ptr(kl), _ptr(lse_s), _ptr(lse_t), _ptr(loss), _ptr(dz_s), _stream(stream)))


def hylo_ild_loss(S, T, grad_scale: float, norms, loss, dS=None, stream=None) -> None:
    """Stage-I ILD loss on stacked bf16 tensors S, T [P, N, d]; dS optional."""
    for name, t in (("S", S), ("T", T)):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 3-D bfloat16 tensor")
    if S.shape != T.shape or (dS is not None and (dS.shape != S.shape or dS.dtype != torch.bfloat16
                                                  or not dS.is_contiguous())):
        raise ValueError("S, T (and dS) must have the same shape")
    P, N, d = S.shape
    _check(load().hylo_ild_loss(_ptr(S), _ptr(T), P, N, d, float(grad_scale), _ptr(norms), _ptr(loss), _ptr(dS),
                                _stream(stream)))


def hylo_kl_selftest_wait_timeout(limit_ms: int, stream=None) -> None:
    _check(load().hylo_kl_selftest_wait_timeout(int(limit_ms), _stream(stream)))


def hylo_kl_sync_status(stream=None) -> None:
    _check(load().hylo_kl_sync_status(_stream(stream)))


def hylo_kl_last_error() -> str:
    msg = load().hylo_kl_last_error()
    return msg.decode() if msg else ""
