"""Seeded synthetic inputs for the fused hidden-state KL loss.

This module only draws random tensors with the shapes and value distributions of the
workloads named below; it holds none of the loss arithmetic, so both the fp64 oracle and
the CUDA path can consume the same bf16 bits.

Workloads (all bf16, row-major; ``h`` = final hidden states, ``W`` = LM-head weights
laid out like ``nn.Linear.weight`` = [vocab, hidden]):

  tiny                 N=64,    d_s=64,   d_t=128,  V=512,    tau=1; h ~ N(0,1), W ~ N(0, 0.05^2)
  llama1b_8b_8k        N=8192,  d_s=2048, d_t=4096, V=128256, tau=1; RMS-normalised N(0,1) h,
                       W ~ N(0, 0.02^2)  (HyLo-Llama-1B student vs Llama-3.1-8B teacher, one 8K sequence)
  stage2_64k           N=65536, same shapes/distributions (one 64K sequence of Stage-II distillation)
  qwen17b_8b           N=16384 (2 x 8192), V=151936, tau=2, otherwise as llama1b_8b_8k
  llama3b_nearconv     N=65536, d_s=3072, d_t=4096, V=128256, tau=1; near-converged student:
                       h_t = RMSnorm(u P^T), u ~ N(0,1), P = Q of a QR of a 4096x3072 N(0,1) matrix,
                       W_t ~ N(0, 0.02^2), W_s = W_t P, h_s = h_t P + 0.01 * N(0,1)

The teacher is Llama-3.1-8B-sized (d_t=4096, V=128256) as in the Stage-II recipe of the
HyLo reading notes (kwkr.cn, "two-stage training recipe", Stage II) and the Experiments
section of the Long-Context Aware Upcycling digest (ftxj.github.io); no weights or data are
available, so these draws stand in for them with the real shapes.

Recipe: one ``torch.Generator`` on the target device seeded with ``1000 + config index``;
tensors are drawn in fp32 in a fixed order (h_s, W_s, h_t, W_t; for the near-converged
workload P, u, W_t, noise), RMS-normalised where stated (divide each row by
sqrt(mean(x^2)), no gain), then rounded once to bf16 (round-to-nearest-even).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    N: int
    d_s: int
    d_t: int
    V: int
    tau: float
    w_std: float
    rms_norm: bool
    near_converged: bool = False
    token_chunk: int = 4096

    @property
    def seed(self) -> int:
        return 1000 + self.index

    def flops_exec(self) -> float:
        """Tensor-core flops of one fwd+bwd with the logit recompute: 4 N V (2 d_s + d_t)."""
        return 4.0 * self.N * self.V * (2 * self.d_s + self.d_t)

    def flops_model(self) -> float:
        """Flops without the recompute: 2 N V (3 d_s + d_t)."""
        return 2.0 * self.N * self.V * (3 * self.d_s + self.d_t)

    def flops_fwd(self) -> float:
        return 2.0 * self.N * self.V * (self.d_s + self.d_t)

    def flops_bwd(self) -> float:
        """Backward: the logit recompute 2 N V (d_s + d_t) plus dh_s and dW_s, 4 N V d_s."""
        return 2.0 * self.N * self.V * (3 * self.d_s + self.d_t)

    def with_sizes(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("tiny", 0, 64, 64, 128, 512, 1.0, 0.05, False),
        Workload("llama1b_8b_8k", 1, 8192, 2048, 4096, 128256, 1.0, 0.02, True),
        Workload("stage2_64k", 2, 65536, 2048, 4096, 128256, 1.0, 0.02, True),
        Workload("qwen17b_8b", 3, 16384, 2048, 4096, 151936, 2.0, 0.02, True),
        Workload("llama3b_nearconv", 4, 65536, 3072, 4096, 128256, 1.0, 0.02, True, near_converged=True),
    )
}


def _rms_normalise(x: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt(torch.mean(x * x, dim=1, keepdim=True))


def _randn(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw (h_s, W_s, h_t, W_t) in bf16 on ``device`` for workload ``w``.

    The same call with the same device, seed and sizes returns the same bits.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    if not w.near_converged:
        h_s = _randn(gen, (w.N, w.d_s), device)
        W_s = _randn(gen, (w.V, w.d_s), device) * w.w_std
        h_t = _randn(gen, (w.N, w.d_t), device)
        W_t = _randn(gen, (w.V, w.d_t), device) * w.w_std
        if w.rms_norm:
            h_s = _rms_normalise(h_s)
            h_t = _rms_normalise(h_t)
    else:
        # P has orthonormal columns, so h_t (a row space of P^T) satisfies h_t P P^T = h_t and the
        # student logits differ from the teacher's only by the 0.01-scaled noise term.
        P, _ = torch.linalg.qr(_randn(gen, (w.d_t, w.d_s), device))
        u = _randn(gen, (w.N, w.d_s), device)
        h_t = _rms_normalise(u @ P.T)
        W_t = _randn(gen, (w.V, w.d_t), device) * w.w_std
        W_s = W_t @ P
        h_s = h_t @ P + 0.01 * _randn(gen, (w.N, w.d_s), device)
        del P, u
    out = {
        "h_s": h_s.to(torch.bfloat16).contiguous(),
        "W_s": W_s.to(torch.bfloat16).contiguous(),
        "h_t": h_t.to(torch.bfloat16).contiguous(),
        "W_t": W_t.to(torch.bfloat16).contiguous(),
    }
    return out


def make_logits(w: Workload, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Student and teacher logits [N, V] in bf16 with the spread the hidden-state workload
    produces: independent N(0, s^2) with s^2 = w_std^2 * d (RMS-normalised hidden states; for
    unnormalised N(0,1) hidden states the same), i.e. the logits z = h W^T would have. Near-
    converged workloads draw z_s = z_t + N(0, (0.01 w_std)^2 d_s). Seeded like make_inputs."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed((w.seed if seed is None else seed) + 7919)
    st = w.w_std * (w.d_t ** 0.5)
    z_t = _randn(gen, (w.N, w.V), device) * st
    if w.near_converged:
        z_s = z_t + _randn(gen, (w.N, w.V), device) * (0.01 * w.w_std * (w.d_s ** 0.5))
    else:
        z_s = _randn(gen, (w.N, w.V), device) * (w.w_std * (w.d_s ** 0.5))
    return {"z_s": z_s.to(torch.bfloat16), "z_t": z_t.to(torch.bfloat16)}


def to_f64_numpy(t: torch.Tensor):
    """Widen a bf16 tensor to a float64 numpy array (exact)."""
    return t.detach().to("cpu", torch.float64).numpy()
