"""fp64 CPU oracle of the fused hidden-state KL distillation loss.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of ``bench.py`` do. It
shares no code with the CUDA library (no kernels, headers, helpers or constants).

What it computes (the plain definition; no online merge, no blocking beyond the pages'
token chunk). Inputs are the bf16 tensors the GPU receives, widened exactly to float64.
For every token n, with tau the temperature:

    z_s = h_s[n] W_s^T,   z_t = h_t[n] W_t^T                       (full vocabulary, materialised)
    l_x = z_x / tau - logsumexp(z_x / tau)                          (log-softmax, max-shifted)
    KL_n = sum_v exp(l_t,v) (l_t,v - l_s,v)                         (KL(p_t || p_s))
    L = (1/N) sum_n KL_n                                            (kl_weight 1, no CE term)
    G[n, v] = grad_scale * (exp(l_s,v) - exp(l_t,v)) / (tau N)      (= dL/dz_s, exact)
    dh_s = G W_s,   dW_s = G^T h_s

Sources:
  * Long-Context Aware Upcycling digest (ftxj.github.io), section Method: Stage II fine-tunes
    the assembled hybrid end to end with KL distillation; the Fused Hidden-State KL skips the
    teacher LM head (the loss takes final hidden states and applies both LM-head projections),
    fuses softmax+KL, and runs a chunked KL with chunk=4096; section Key Ideas names the
    Fused KL / Fused Hidden-State KL memory stack.
  * HyLo-Llama-8MLA8GDN-8K-SFT reading notes (kwkr.cn), section two-stage training recipe,
    Stage II: the loss is the KL divergence between the student's and the teacher's
    next-token distributions, kl_weight 1.0, no cross-entropy, with a fused KL kernel so
    the full logit tensor is never materialised.

Readings where the pages are silent (they print no formula): forward KL(p_t || p_s) (the
usual distillation direction); logits divided by tau with no tau^2 factor; the loss is the
mean over all N tokens of all chunks; "chunk=4096" is a token chunk and results do not
depend on it; the teacher is frozen, so no teacher gradients.

Pins: every function here is checked in tests/test_oracle_pins.py against closed forms,
invariants, library special cases, brute force and finite differences (see that file).
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np


def lm_head_logits(h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z = h W^T: project final hidden states [n, d] through an LM head [V, d] (digest, Method:
    the hidden-state KL applies the LM-head projections inside the loss)."""
    return h @ W.T


def log_softmax(z: np.ndarray, tau: float) -> Tuple[np.ndarray, np.ndarray]:
    """Row-wise log softmax of z/tau and its log-sum-exp (max-shifted for range only)."""
    x = z / tau
    m = np.max(x, axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.sum(np.exp(x - m), axis=1))
    return x - lse[:, None], lse


def _chunks(N: int, token_chunk: int):
    token_chunk = max(1, int(token_chunk))
    for c0 in range(0, N, token_chunk):
        yield slice(c0, min(N, c0 + token_chunk))


def kl_forward(h_s, W_s, h_t, W_t, tau: float, token_chunk: int = 4096):
    """Per-token KL(p_t || p_s), both log-sum-exps, and the mean loss (digest, Method; reading
    notes, Stage II). Returns (kl[N], lse_s[N], lse_t[N], loss)."""
    N = h_s.shape[0]
    kl = np.zeros(N)
    lse_s = np.zeros(N)
    lse_t = np.zeros(N)
    for sl in _chunks(N, token_chunk):
        l_s, lse_s[sl] = log_softmax(lm_head_logits(h_s[sl], W_s), tau)
        l_t, lse_t[sl] = log_softmax(lm_head_logits(h_t[sl], W_t), tau)
        p_t = np.exp(l_t)
        kl[sl] = np.sum(p_t * (l_t - l_s), axis=1)
    loss = float(np.mean(kl)) if N > 0 else 0.0
    return kl, lse_s, lse_t, loss


def kl_grad_logits(h_s, W_s, h_t, W_t, tau: float, grad_scale: float, n_total: int):
    """G = dL/dz_s for a block of tokens of a loss averaged over ``n_total`` tokens."""
    l_s, _ = log_softmax(lm_head_logits(h_s, W_s), tau)
    l_t, _ = log_softmax(lm_head_logits(h_t, W_t), tau)
    return (np.exp(l_s) - np.exp(l_t)) * (grad_scale / (tau * n_total))


def kl_backward(h_s, W_s, h_t, W_t, tau: float, token_chunk: int = 4096, grad_scale: float = 1.0):
    """Gradients of grad_scale * L with respect to h_s and W_s (the student's final hidden
    states and LM head; the teacher is frozen). Returns (dh_s [N, d_s], dW_s [V, d_s])."""
    N = h_s.shape[0]
    dh_s = np.zeros(h_s.shape)
    dW_s = np.zeros(W_s.shape)
    for sl in _chunks(N, token_chunk):
        G = kl_grad_logits(h_s[sl], W_s, h_t[sl], W_t, tau, grad_scale, N)
        dh_s[sl] = G @ W_s
        dW_s += G.T @ h_s[sl]
    return dh_s, dW_s


def kl_rows(h_s, W_s, h_t, W_t, tau: float, rows: Sequence[int], grad_scale: float = 1.0,
            n_total: Optional[int] = None, token_chunk: int = 256):
    """KL_n, lse_s,n, lse_t,n and dh_s[n, :] for selected token rows only, each computed
    exactly as in kl_forward / kl_backward (every token's results depend on its own row
    alone, apart from the 1/N of the mean). Returns (kl, lse_s, lse_t, dh_rows)."""
    rows = np.asarray(rows, dtype=np.int64)
    n_total = h_s.shape[0] if n_total is None else n_total
    kl = np.zeros(len(rows))
    lse_s = np.zeros(len(rows))
    lse_t = np.zeros(len(rows))
    dh = np.zeros((len(rows), W_s.shape[1]))
    for sl in _chunks(len(rows), token_chunk):
        r = rows[sl]
        hs = np.asarray(h_s[r], dtype=np.float64)
        ht = np.asarray(h_t[r], dtype=np.float64)
        l_s, lse_s[sl] = log_softmax(lm_head_logits(hs, W_s), tau)
        l_t, lse_t[sl] = log_softmax(lm_head_logits(ht, W_t), tau)
        p_t = np.exp(l_t)
        kl[sl] = np.sum(p_t * (l_t - l_s), axis=1)
        G = (np.exp(l_s) - p_t) * (grad_scale / (tau * n_total))
        dh[sl] = G @ W_s
    return kl, lse_s, lse_t, dh



def kl_grad_vocab_rows(h_s, W_s, h_t, W_t, tau: float, vocab_rows: Sequence[int], lse_s, lse_t,
                       grad_scale: float = 1.0, n_total: Optional[int] = None, token_chunk: int = 4096):
    """Rows dW_s[v, :] of the student LM-head gradient for selected vocabulary rows v only,
    given every token's log-sum-exps over the full vocabulary (as kl_forward returns them):
    dW_s[v] = sum_n G[n, v] h_s[n] with G[n, v] = grad_scale (exp(z_s[n,v]/tau - lse_s[n]) -
    exp(z_t[n,v]/tau - lse_t[n])) / (tau N), the column v of the G of kl_backward (the softmax
    of each token needs the whole vocabulary only through its log-sum-exp).
    Returns dW rows [len(vocab_rows), d_s]."""
    rows = np.asarray(vocab_rows, dtype=np.int64)
    N = h_s.shape[0]
    n_total = N if n_total is None else n_total
    Ws = np.asarray(W_s[rows], dtype=np.float64)
    Wt = np.asarray(W_t[rows], dtype=np.float64)
    lse_s = np.asarray(lse_s, dtype=np.float64)
    lse_t = np.asarray(lse_t, dtype=np.float64)
    out = np.zeros((len(rows), W_s.shape[1]))
    for sl in _chunks(N, token_chunk):
        hs = np.asarray(h_s[sl], dtype=np.float64)
        zs = lm_head_logits(hs, Ws) / tau
        zt = lm_head_logits(np.asarray(h_t[sl], dtype=np.float64), Wt) / tau
        G = (np.exp(zs - lse_s[sl, None]) - np.exp(zt - lse_t[sl, None])) * (grad_scale / (tau * n_total))
        out += G.T @ hs
    return out


def kl_from_logits(z_s, z_t, tau: float, grad_scale: float = 1.0):
    """The same loss on given logits ("Fused KL" of the digest's Key Ideas, applied to logits
    that were already projected): per-token KL(p_t || p_s), both log-sum-exps, the mean loss,
    and G = d(grad_scale * L)/dz_s = grad_scale * (p_s - p_t) / (tau N).
    Returns (kl, lse_s, lse_t, loss, G)."""
    N = z_s.shape[0]
    l_s, lse_s = log_softmax(z_s, tau)
    l_t, lse_t = log_softmax(z_t, tau)
    p_t = np.exp(l_t)
    kl = np.sum(p_t * (l_t - l_s), axis=1)
    G = (np.exp(l_s) - p_t) * (grad_scale / (tau * N))
    return kl, lse_s, lse_t, (float(np.mean(kl)) if N > 0 else 0.0), G


def ild_loss(S, T, grad_scale: float = 1.0):
    """Stage-I Enhanced-ILD alignment loss (Long-Context Aware Upcycling digest, section Method:
    L_ILD = sum over layers of ||h_s - h_t||_2 + ||a_s - a_t||_2, hidden states and token-mixer
    outputs; the reading notes' Stage I aligns each new layer with the base model's internal
    representations). S and T stack the student and teacher tensors as [P, N, d] (P = one entry
    per layer and per kind, h or a). Reading of the printed formula: the Euclidean norm of each
    token's difference vector (not squared), averaged over the N tokens and summed over the P
    entries. Returns (norms [P, N], loss, grad) with grad = grad_scale * dL/dS =
    grad_scale * (S - T) / (N ||S - T||), taken as 0 where the difference is 0."""
    S = np.asarray(S, dtype=np.float64)
    T = np.asarray(T, dtype=np.float64)
    P, N, d = S.shape
    D = S - T
    norms = np.sqrt(np.sum(D * D, axis=2))
    loss = float(np.sum(norms) / N) if N > 0 else 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        scale = np.where(norms > 0, grad_scale / (N * norms), 0.0)
    grad = D * scale[:, :, None]
    return norms, loss, grad
