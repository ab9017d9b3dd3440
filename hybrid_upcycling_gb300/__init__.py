"""GB300-native (sm_103a) fused hidden-state KL distillation loss of HyLo's Stage II.

The compute lives in libhylo_kl.so (hand-written tcgen05/TMA kernels behind the C ABI of
include/hylo_kl.h). ``_lib`` binds that ABI one-to-one; ``kl`` wraps the three losses as PyTorch
autograd functions; ``synthetic`` draws the seeded benchmark inputs.
"""
from . import synthetic  # noqa: F401

__all__ = ["synthetic", "fused_hidden_state_kl", "fused_logits_kl", "ild_loss"]


def fused_hidden_state_kl(*args, **kwargs):
    from .kl import fused_hidden_state_kl as f
    return f(*args, **kwargs)


def fused_logits_kl(*args, **kwargs):
    from .kl import fused_logits_kl as f
    return f(*args, **kwargs)


def ild_loss(*args, **kwargs):
    from .kl import ild_loss as f
    return f(*args, **kwargs)
