"""GB300-native (sm_103a) fused hidden-state KL distillation loss of HyLo's Stage II.

The compute lives in libhylo_kl.so (hand-written tcgen05/TMA kernels behind the C ABI of
include/hylo_kl.h). ``_lib`` binds that ABI one-to-one; ``kl`` wraps it as a PyTorch autograd
function; ``synthetic`` draws the seeded benchmark inputs.
"""
from . import synthetic  # noqa: F401

__all__ = ["synthetic", "fused_hidden_state_kl"]


def fused_hidden_state_kl(*args, **kwargs):
    from .kl import fused_hidden_state_kl as f
    return f(*args, **kwargs)
