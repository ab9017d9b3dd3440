"""User-facing PyTorch wrapper of the fused hidden-state KL loss.

``fused_hidden_state_kl(h_s, W_s, h_t, W_t, tau)`` returns the mean KL(p_t || p_s) over all
tokens (and the per-token values); its backward gives d/dh_s and d/dW_s. Both directions run
entirely in the sm_103a kernels of libhylo_kl.so via the C ABI; PyTorch only allocates the
outputs and the workspace. The teacher inputs (h_t, W_t) receive no gradient.
"""
from __future__ import annotations

import torch

from . import _lib


def _alloc_outputs(N: int, device):
    f = dict(dtype=torch.float32, device=device)
    return torch.empty(N, **f), torch.empty(N, **f), torch.empty(N, **f), torch.empty(N, **f), torch.empty(1, **f)


def workspace(N: int, d_s: int, d_t: int, V: int, token_chunk: int, device, split: bool = False) -> torch.Tensor:
    query = _lib.hylo_kl_workspace_bytes_split if split else _lib.hylo_kl_workspace_bytes
    nbytes = query(N, d_s, d_t, V, token_chunk)
    if nbytes == 0:
        raise ValueError("invalid sizes for the fused hidden-state KL")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


class FusedHiddenStateKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, h_s, W_s, h_t, W_t, tau: float = 1.0, token_chunk: int = 4096, split_g: bool = False):
        N, d_s = h_s.shape
        V, d_t = W_t.shape
        ws = workspace(N, d_s, d_t, V, token_chunk, h_s.device)
        kl, lse_s, lse_t, gap, loss = _alloc_outputs(N, h_s.device)
        _lib.hylo_kl_forward(h_s, W_s, h_t, W_t, tau, token_chunk, kl, lse_s, lse_t, loss, ws, lse_gap=gap)
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
        dh_s = torch.empty(N, d_s, dtype=torch.float32, device=h_s.device)
        dW_s = torch.empty(V, d_s, dtype=torch.float32, device=h_s.device)
        scale = 1.0 if g_loss is None else float(g_loss)  # one host read of the upstream scalar
        bwd = _lib.hylo_kl_backward_split if ctx.split_g else _lib.hylo_kl_backward
        bwd(h_s, W_s, h_t, W_t, ctx.tau, ctx.token_chunk, lse_s, lse_t, scale, dh_s, dW_s, ws, lse_gap=gap)
        return dh_s.to(h_s.dtype), dW_s.to(W_s.dtype), None, None, None, None, None


def fused_hidden_state_kl(h_s, W_s, h_t, W_t, tau: float = 1.0, token_chunk: int = 4096, split_g: bool = False):
    """Mean KL(softmax(h_t W_t^T / tau) || softmax(h_s W_s^T / tau)) over tokens, and per-token KL.
    split_g: backward with G kept as two bf16 terms (hylo_kl_backward_split)."""
    return FusedHiddenStateKL.apply(h_s, W_s, h_t, W_t, tau, token_chunk, split_g)
