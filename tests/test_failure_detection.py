"""Failure detection without faulting a GPU.

Every pipeline wait in the kernels is time-limited: on expiry the kernel records a timeout in a
per-device status word, drains what it has in flight and returns. The GPU test forces a wait
to run out (a barrier nothing signals) and checks that the host reads HYLO_ERR_TIMEOUT, that
the status is cleared after the read, and that the device keeps working. The CPU test checks
the argument guard without a GPU.
"""
import pytest
import torch

from hybrid_upcycling_gb300 import _lib, build


def test_selftest_rejects_bad_limits_without_a_gpu():
    build.build()
    lib = _lib.load()
    assert lib.hylo_kl_selftest_wait_timeout(0, None) == -2
    assert lib.hylo_kl_selftest_wait_timeout(5000, None) == -2


@pytest.mark.gpu
def test_timed_out_wait_is_reported_and_device_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _lib.hylo_kl_sync_status()  # start from a clean status word
    _lib.hylo_kl_selftest_wait_timeout(20)
    with pytest.raises(_lib.HyloError) as err:
        _lib.hylo_kl_sync_status()
    assert err.value.status == -7  # HYLO_ERR_TIMEOUT
    assert "timed out" in str(err.value)
    _lib.hylo_kl_sync_status()  # cleared by the read
    # the context is still healthy: a real forward runs and is finite
    from hybrid_upcycling_gb300 import synthetic as syn
    w = syn.WORKLOADS["tiny"]
    x = syn.make_inputs(w, device="cuda")
    f = dict(dtype=torch.float32, device="cuda")
    ws = torch.empty(_lib.hylo_kl_workspace_bytes(w.N, w.d_s, w.d_t, w.V, 4096), dtype=torch.uint8, device="cuda")
    out = [torch.empty(w.N, **f), torch.empty(w.N, **f), torch.empty(w.N, **f), torch.empty(1, **f)]
    _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 1.0, 4096, *out, ws)
    _lib.hylo_kl_sync_status()
    assert torch.isfinite(out[3]).all() and out[3].item() > 0
