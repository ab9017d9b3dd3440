"""Token-sharded (data-parallel) fused hidden-state KL over a torch.distributed process group.

Stage II of HyLo trains with FSDP on 8 GPUs (Long-Context Aware Upcycling digest, section
Experiments: FSDP full shard, bf16, 8 x MI300X; HyLo-Llama-8MLA8GDN-8K-SFT reading notes, Stage
II). For this loss that is a split of the tokens: every rank holds its own N_r tokens (h_s, h_t
rows) and the full LM heads W_s, W_t, and

  * each token's KL, log-sum-exps and dh_s row depend on that token's row alone (local);
  * the loss is the mean over all N = sum_r N_r tokens: L = sum_r N_r L_r / N, with L_r the mean
    of the rank's own tokens -- one all-reduce of a scalar;
  * G = (p_s - p_t) / (tau N) carries the GLOBAL N, so each rank runs its backward with
    grad_scale = upstream * N_r / N (the library normalises by the N it is given, N_r);
  * dW_s = G^T h_s is a sum over all tokens: the ranks' partial dW_s are summed with one
    all-reduce, or with one reduce-scatter that leaves each rank the rows of its vocabulary
    shard (the FSDP layout of the gradient).

``kl_fwd_bwd_sharded`` does exactly this around one call of the C ABI per rank; the kernels
are the single-GPU ones. The per-shard computation can be replaced (``compute=``) by any
function with the same contract, which is how the orchestration is tested on CPU ranks.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import torch
import torch.distributed as dist


@dataclass
class ShardResult:
    loss: torch.Tensor        # [1] float64: the global mean KL over all ranks' tokens
    kl: torch.Tensor          # [N_r] float32: this rank's per-token KL
    dh_s: torch.Tensor        # [N_r, d_s] float32: gradient of (upstream * loss) w.r.t. this rank's h_s
    dW_s: torch.Tensor        # [V, d_s] summed over ranks, or [rows, d_s] of this rank's vocabulary shard
    n_total: int              # tokens over all ranks
    vocab_rows: tuple         # (first, last + 1) vocabulary rows held in dW_s


# compute(h_s, W_s, h_t, W_t, tau, token_chunk, grad_scale) -> (loss_local [1], kl [N_r], dh_s, dW_s)
Compute = Callable[..., tuple]


class LibraryCompute:
    """One forward + backward of the shard through the C ABI (libhylo_kl.so) on the tensors'
    CUDA device. The workspace is kept between calls (grown when a call needs more). With
    `timing` set, each call appends three CUDA events recorded on the current stream (before
    the forward, between forward and backward, after the backward) to `marks`."""

    def __init__(self, timing: bool = False):
        self.ws: Optional[torch.Tensor] = None
        self.timing = timing
        self.marks = []

    def _mark(self):
        if not self.timing:
            return None
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    def __call__(self, h_s, W_s, h_t, W_t, tau, token_chunk, grad_scale):
        from . import _lib
        N, d_s = h_s.shape
        V, d_t = W_t.shape
        dev = h_s.device
        need = _lib.hylo_kl_workspace_bytes(N, d_s, d_t, V, token_chunk)
        if self.ws is None or self.ws.numel() < need or self.ws.device != dev:
            self.ws = torch.empty(need, dtype=torch.uint8, device=dev)
        f = dict(dtype=torch.float32, device=dev)
        kl, lse_s, lse_t, gap = (torch.empty(N, **f) for _ in range(4))
        loss = torch.empty(1, **f)
        dh_s, dW_s = torch.empty(N, d_s, **f), torch.empty(V, d_s, **f)
        e0 = self._mark()
        _lib.hylo_kl_forward(h_s, W_s, h_t, W_t, tau, token_chunk, kl, lse_s, lse_t, loss, self.ws, lse_gap=gap)
        e1 = self._mark()
        _lib.hylo_kl_backward(h_s, W_s, h_t, W_t, tau, token_chunk, lse_s, lse_t, grad_scale, dh_s, dW_s, self.ws,
                              lse_gap=gap)
        if self.timing:
            self.marks.append((e0, e1, self._mark()))
        return loss, kl, dh_s, dW_s


def vocab_shard(V: int, rank: int, world: int) -> tuple:
    """Rows [first, last) of the vocabulary held by `rank` after a reduce-scatter: ceil(V / world)
    rows per rank, the last ranks' shares cut at V (possibly empty)."""
    per = -(-V // world)
    return min(V, rank * per), min(V, (rank + 1) * per)


def kl_fwd_bwd_sharded(h_s, W_s, h_t, W_t, tau: float, token_chunk: int = 4096, group=None,
                       grad_reduce: str = "all_reduce", upstream: float = 1.0,
                       compute: Optional[Compute] = None, n_total: Optional[int] = None) -> ShardResult:
    """Forward + backward of the fused hidden-state KL for this rank's tokens, combined over the
    process group into the results of the unsharded loss (see the module docstring).

    h_s [N_r, d_s], h_t [N_r, d_t]: this rank's tokens (any N_r >= 1, ranks may differ);
    W_s [V, d_s], W_t [V, d_t]: the full LM heads, identical on every rank. grad_reduce:
    "all_reduce" (every rank gets the full dW_s) or "reduce_scatter" (each rank gets the rows
    vocab_shard(V, rank, world) of dW_s). upstream: d(outer)/dL, folded into grad_scale.
    n_total: the tokens of all ranks, if the caller knows it (otherwise one all-reduce of the
    token counts, read on the host). Collectives: the loss sum and dW_s (all-reduce, or
    reduce-scatter), on the tensors' device (NCCL for CUDA tensors, gloo for CPU tensors).
    """
    if grad_reduce not in ("all_reduce", "reduce_scatter"):
        raise ValueError("grad_reduce must be 'all_reduce' or 'reduce_scatter'")
    compute = compute if compute is not None else LibraryCompute()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    dev = h_s.device
    n_local = int(h_s.shape[0])
    if n_total is None:
        counts = torch.tensor([n_local], dtype=torch.int64, device=dev)
        dist.all_reduce(counts, group=group)
        n_total = int(counts.item())
    loss_local, kl, dh_s, dW_s = compute(h_s, W_s, h_t, W_t, tau, token_chunk, upstream * n_local / n_total)
    # sum_r N_r L_r in float64, then the global mean (stays on the device: no host read)
    loss = loss_local.to(torch.float64).reshape(1) * n_local
    dist.all_reduce(loss, group=group)
    loss = loss / n_total
    V, d_s = dW_s.shape
    if grad_reduce == "all_reduce" or world == 1:
        dist.all_reduce(dW_s, group=group)
        rows = (0, V)
    else:
        per = -(-V // world)
        if per * world != V:  # the collective wants equal shares: pad the vocabulary with zero rows
            padded = torch.zeros(per * world, d_s, dtype=dW_s.dtype, device=dev)
            padded[:V] = dW_s
        else:
            padded = dW_s
        out = torch.empty(per, d_s, dtype=dW_s.dtype, device=dev)
        dist.reduce_scatter_tensor(out, padded, group=group)
        rows = vocab_shard(V, rank, world)
        dW_s = out[: rows[1] - rows[0]]
    return ShardResult(loss=loss, kl=kl, dh_s=dh_s, dW_s=dW_s, n_total=n_total, vocab_rows=rows)
