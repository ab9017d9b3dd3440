"""User-facing PyTorch wrappers of the fused hidden-state KL loss.

``fused_hidden_state_kl(h_s, W_s, h_t, W_t, tau)`` is an autograd function: it returns the mean
KL(p_t || p_s) over all tokens (and the per-token values), and its backward gives d/dh_s and
d/dW_s in the inputs' dtype. ``kl_fwd_bwd(...)`` runs forward and backward in one call and
returns fp32 gradients (optionally into caller buffers), for trainers that keep fp32 gradient
accumulators. Both run entirely in the sm_103a kernels of libhylo_kl.so through the C ABI;
PyTorch only allocates the outputs and the workspace. The teacher inputs (h_t, W_t) receive no
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
