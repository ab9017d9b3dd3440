"""User-facing PyTorch wrappers of the fused hidden-state KL loss and its two siblings.

``fused_hidden_state_kl(h_s, W_s, h_t, W_t, tau)`` is an autograd function: it returns the mean
KL(p_t || p_s) over all tokens (and the per-token values), and its backward gives d/dh_s and
d/dW_s in the inputs' dtype. ``kl_fwd_bwd(...)`` runs forward and backward in one call and
returns fp32 gradients (optionally into caller buffers), for trainers that keep fp32 gradient
accumulators. ``fused_logits_kl(z_s, z_t, tau)`` is the same loss on precomputed logits and
``ild_loss(S, T)`` the Stage-I layer-alignment loss, both autograd functions whose gradient is
formed in the forward launch. All run entirely in the sm_103a kernels of libhylo_kl.so through
the C ABI; PyTorch only allocates the outputs and the workspace. The teacher inputs receive no
gradient.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import torch

from . import _lib

# One workspace per (device, split flag), grown when a call needs more and shared by the
# forward and the backward of every call on that device (calls on one device run in stream
# order; callers that run calls concurrently on several streams pass their own workspaces to
# the C-ABI functions instead).
_WORKSPACES: Dict[Tuple[torch.device, bool], torch.Tensor] = {}


def workspace(N: int, d_s: int, d_t: int, V: int, token_chunk: int, device, split: bool = False) -> torch.Tensor:
    """A workspace of at least the bytes the library needs for these sizes (cached per device)."""
    query = _lib.hylo_kl_workspace_bytes_split if split else _lib.hylo_kl_workspace_bytes
    nbytes = query(N, d_s, d_t, V, token_chunk)
    if nbytes == 0:
        raise ValueError("invalid sizes for the fused hidden-state KL")
    device = torch.device(device)
    key = (device, split)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


def _forward(h_s, W_s, h_t, W_t, tau, token_chunk, split_g=False):
    N, d_s = h_s.shape
    V, d_t = W_t.shape
    ws = workspace(N, d_s, d_t, V, token_chunk, h_s.device, split=split_g)
    f = dict(dtype=torch.float32, device=h_s.device)
    kl, lse_s, lse_t, gap = (torch.empty(N, **f) for _ in range(4))
    loss = torch.empty(1, **f)
    _lib.hylo_kl_forward(h_s, W_s, h_t, W_t, tau, token_chunk, kl, lse_s, lse_t, loss, ws, lse_gap=gap)
    return loss, kl, lse_s, lse_t, gap, ws


def _backward(h_s, W_s, h_t, W_t, tau, token_chunk, lse_s, lse_t, gap, ws, grad_scale, dh_s, dW_s, split_g):
    bwd = _lib.hylo_kl_backward_split if split_g else _lib.hylo_kl_backward
    bwd(h_s, W_s, h_t, W_t, tau, token_chunk, lse_s, lse_t, grad_scale, dh_s, dW_s, ws, lse_gap=gap)


class FusedHiddenStateKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, h_s, W_s, h_t, W_t, tau: float = 1.0, token_chunk: int = 4096, split_g: bool = False):
        loss, kl, lse_s, lse_t, gap, _ = _forward(h_s, W_s, h_t, W_t, tau, token_chunk, split_g)
        ctx.save_for_backward(h_s, W_s, h_t, W_t, lse_s, lse_t, gap)
        ctx.tau, ctx.token_chunk, ctx.split_g = tau, token_chunk, split_g
        ctx.mark_non_differentiable(kl)
        return loss[0], kl

    @staticmethod
    def backward(ctx, g_loss, g_kl):
        h_s, W_s, h_t, W_t, lse_s, lse_t, gap = ctx.saved_tensors
        N, d_s = h_s.shape
        V, d_t = W_t.shape
        ws = workspace(N, d_s, d_t, V, ctx.token_chunk, h_s.device, split=ctx.split_g)
        f = dict(dtype=torch.float32, device=h_s.device)
        dh_s, dW_s = torch.empty(N, d_s, **f), torch.empty(V, d_s, **f)
        # The gradients for an upstream gradient of 1; the upstream value is applied on the
        # device below, fused with the conversion to the inputs' dtype (no host read of it).
        _backward(h_s, W_s, h_t, W_t, ctx.tau, ctx.token_chunk, lse_s, lse_t, gap, ws, 1.0, dh_s, dW_s, ctx.split_g)
        if g_loss is None:
            return dh_s.to(h_s.dtype), dW_s.to(W_s.dtype), None, None, None, None, None
        g = g_loss.to(torch.float32)
        out_h = torch.empty(N, d_s, dtype=h_s.dtype, device=h_s.device)
        out_W = torch.empty(V, d_s, dtype=W_s.dtype, device=W_s.device)
        torch.mul(dh_s, g, out=out_h)  # one pass: scale and convert
        torch.mul(dW_s, g, out=out_W)
        return out_h, out_W, None, None, None, None, None


def fused_hidden_state_kl(h_s, W_s, h_t, W_t, tau: float = 1.0, token_chunk: int = 4096, split_g: bool = False):
    """Mean KL(softmax(h_t W_t^T / tau) || softmax(h_s W_s^T / tau)) over tokens, and per-token KL.
    split_g: backward with G kept as two bf16 terms (hylo_kl_backward_split)."""
    return FusedHiddenStateKL.apply(h_s, W_s, h_t, W_t, tau, token_chunk, split_g)


def kl_fwd_bwd(h_s, W_s, h_t, W_t, tau: float = 1.0, token_chunk: int = 4096, grad_scale: float = 1.0,
               dh_s: Optional[torch.Tensor] = None, dW_s: Optional[torch.Tensor] = None, split_g: bool = False):
    """Forward and backward in one call, without autograd: returns (loss [1], kl [N], dh_s, dW_s)
    with fp32 gradients of grad_scale * loss. dh_s [N, d_s] / dW_s [V, d_s] (fp32, contiguous)
    may be given to receive the gradients (they are overwritten), e.g. a trainer's fp32 gradient
    buffers, so that no extra pass converts them."""
    loss, kl, lse_s, lse_t, gap, ws = _forward(h_s, W_s, h_t, W_t, tau, token_chunk, split_g)
    N, d_s = h_s.shape
    V = W_s.shape[0]
    f = dict(dtype=torch.float32, device=h_s.device)
    dh_s = torch.empty(N, d_s, **f) if dh_s is None else dh_s
    dW_s = torch.empty(V, d_s, **f) if dW_s is None else dW_s
    _backward(h_s, W_s, h_t, W_t, tau, token_chunk, lse_s, lse_t, gap, ws, grad_scale, dh_s, dW_s, split_g)
    return loss, kl, dh_s, dW_s


def _logits_rows(z: torch.Tensor) -> torch.Tensor:
    """z itself if its rows meet the C ABI's layout (unit column stride, row stride a multiple
    of 8 elements), else a copy into rows padded to a multiple of 8 (returned as a [N, V] view)."""
    N, V = z.shape
    if z.stride(1) == 1 and z.stride(0) >= V and z.stride(0) % 8 == 0:
        return z
    ld = (V + 7) // 8 * 8
    buf = torch.empty(N, ld, dtype=z.dtype, device=z.device)
    buf[:, :V] = z
    return buf[:, :V]


class FusedLogitsKL(torch.autograd.Function):
    """Mean KL(softmax(z_t / tau) || softmax(z_s / tau)) over the rows of precomputed bf16
    logits [N, V], through hylo_fused_kl_logits. The gradient with respect to z_s is formed in
    the same launch as the loss (when z_s needs one) and scaled by the upstream gradient in the
    backward; z_t (the teacher) receives none."""

    @staticmethod
    def forward(ctx, z_s, z_t, tau: float = 1.0):
        if z_s.shape != z_t.shape or z_s.dtype != torch.bfloat16 or z_t.dtype != torch.bfloat16:
            raise ValueError("z_s and z_t must be bfloat16 tensors of the same [N, V] shape")
        zs, zt = _logits_rows(z_s), _logits_rows(z_t)
        if zs.stride(0) != zt.stride(0):  # the ABI takes one row stride for both
            zs, zt = _logits_rows(zs.contiguous()), _logits_rows(zt.contiguous())
        N, V = zs.shape
        f = dict(dtype=torch.float32, device=zs.device)
        kl, lse_s, lse_t = (torch.empty(N, **f) for _ in range(3))
        loss = torch.empty(1, **f)
        dz = None
        if ctx.needs_input_grad[0]:
            dz = torch.empty(N, zs.stride(0), dtype=torch.bfloat16, device=zs.device)[:, :V]
        _lib.hylo_fused_kl_logits(zs, zt, tau, 1.0, kl, lse_s, lse_t, loss, dz)
        ctx.save_for_backward(dz if dz is not None else torch.empty(0, device=zs.device))
        ctx.has_dz = dz is not None
        ctx.mark_non_differentiable(kl)
        return loss[0], kl

    @staticmethod
    def backward(ctx, g_loss, g_kl):
        (dz,) = ctx.saved_tensors
        if not ctx.has_dz or g_loss is None:
            return None, None, None
        return dz * g_loss.to(torch.float32), None, None


def fused_logits_kl(z_s, z_t, tau: float = 1.0):
    """Mean KL(p_t || p_s) over rows of bf16 logits z_s, z_t [N, V], and the per-row KL; the
    student logits z_s receive the gradient (bf16)."""
    return FusedLogitsKL.apply(z_s, z_t, tau)


class ILDLoss(torch.autograd.Function):
    """Stage-I alignment loss sum_p mean_n ||S[p, n] - T[p, n]||_2 over stacked bf16 tensors
    [P, N, d], through hylo_ild_loss. The gradient with respect to S is formed in the same
    launch (when S needs one) and scaled by the upstream gradient in the backward; T (the
    teacher) receives none."""

    @staticmethod
    def forward(ctx, S, T):
        S, T = S.contiguous(), T.contiguous()
        P, N, d = S.shape
        f = dict(dtype=torch.float32, device=S.device)
        norms = torch.empty(P, N, **f)
        loss = torch.empty(1, **f)
        dS = torch.empty_like(S) if ctx.needs_input_grad[0] else None
        _lib.hylo_ild_loss(S, T, 1.0, norms, loss, dS)
        ctx.save_for_backward(dS if dS is not None else torch.empty(0, device=S.device))
        ctx.has_dS = dS is not None
        ctx.mark_non_differentiable(norms)
        return loss[0], norms

    @staticmethod
    def backward(ctx, g_loss, g_norms):
        (dS,) = ctx.saved_tensors
        if not ctx.has_dS or g_loss is None:
            return None, None
        return dS * g_loss.to(torch.float32), None


def ild_loss(S, T):
    """Stage-I ILD loss of student S against teacher T ([P, N, d] bf16) and the per-row norms
    [P, N]; S receives the gradient (bf16)."""
    return ILDLoss.apply(S, T)
