"""The forward entry point that allocates nothing (hylo_kl_forward_noalloc).

It exists for callers that cannot allocate device memory themselves, such as a plugin that
may only use the buffers its host framework gives it, or a step loop that must not call
cudaMalloc. Its scratch is a fixed array inside the library. This file is named so that
pytest collects it last; its GPU test passes alone in a fresh process and after the others.
"""
import numpy as np
import pytest
import torch

from hybrid_upcycling_gb300 import _lib, build, synthetic as syn

TOL_KL, TOL_LOSS, TOL_LSE = 1e-3, 1e-4, 2e-5
FAKE = 0x10000


def _noalloc(lib, N=16, d_s=64, d_t=128, V=100, ptr=FAKE, tau=1.0):
    return lib.hylo_kl_forward_noalloc(ptr, ptr, ptr, ptr, N, d_s, d_t, V, tau, 4096, ptr, ptr, ptr, None, ptr, None)


def test_noalloc_rejects_bad_arguments_without_touching_the_gpu():
    build.build()
    lib = _lib.load()
    assert _noalloc(lib, ptr=None) == -1
    assert _noalloc(lib, d_s=12) == -2
    assert _noalloc(lib, N=698998) == -2  # more tokens than the built-in scratch holds
    assert b"built-in scratch" in lib.hylo_kl_last_error()
    assert _noalloc(lib, ptr=FAKE + 4) == -3
    assert _noalloc(lib, tau=0.0) == -4


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    w = syn.WORKLOADS["llama1b_8b_8k"].with_sizes(N=3000, V=20000)
    x = syn.make_inputs(w, device="cuda")
    N = w.N
    f = dict(dtype=torch.float32, device="cuda")

    ws = torch.empty(_lib.hylo_kl_workspace_bytes(N, w.d_s, w.d_t, w.V, 4096), dtype=torch.uint8, device="cuda")
    ref = [torch.empty(N, **f), torch.empty(N, **f), torch.empty(N, **f), torch.empty(1, **f)]
    _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 4096, *ref, ws)
    _lib.hylo_kl_sync_status()
    r_kl, r_ls, r_lt, r_loss = (t.double().cpu().numpy() for t in ref)

    for call in range(2):  # the second call starts with the first call's leftovers in the scratch
        out = [torch.full((N,), float("nan"), **f) for _ in range(3)] + [torch.full((1,), float("nan"), **f)]
        _lib.hylo_kl_forward_noalloc(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 4096, *out)
        _lib.hylo_kl_sync_status()
        kl, ls, lt, loss = (t.double().cpu().numpy() for t in out)
        assert np.all(np.abs(kl - r_kl) <= TOL_KL * (1 + r_kl)), call
        assert abs(loss[0] - r_loss[0]) <= TOL_LOSS * abs(r_loss[0]), call
        assert np.all(np.abs(ls - r_ls) <= TOL_LSE * (1 + np.abs(r_ls))), call
        assert np.all(np.abs(lt - r_lt) <= TOL_LSE * (1 + np.abs(r_lt))), call


@pytest.mark.gpu
def test_noalloc_forward_at_its_token_limit():
    """N = 698997, the largest N the built-in array holds: the statistics fill it to its last
    statistics byte (fewer vocabulary segments than the workspace forward would use, so the
    results agree with it to fp32 summation order) and the launch paces its clusters with the
    counters at the array's tail. Checked against the workspace forward and, on 300 sampled
    rows including the last, against the fp64 oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    from oracle import kl_oracle as orc
    w = syn.Workload("limit", 0, 698997, 64, 64, 2000, 1.0, 0.1, False)
    x = syn.make_inputs(w, device="cuda", seed=5)
    N = w.N
    f = dict(dtype=torch.float32, device="cuda")
    ws = torch.empty(_lib.hylo_kl_workspace_bytes(N, w.d_s, w.d_t, w.V, 4096), dtype=torch.uint8, device="cuda")
    ref = [torch.empty(N, **f), torch.empty(N, **f), torch.empty(N, **f), torch.empty(1, **f)]
    _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 4096, *ref, ws)
    out = [torch.full((N,), float("nan"), **f) for _ in range(3)] + [torch.full((1,), float("nan"), **f)]
    _lib.hylo_kl_forward_noalloc(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 4096, *out)
    _lib.hylo_kl_sync_status()
    kl, ls, lt, loss = (t.double().cpu().numpy() for t in out)
    r_kl, r_loss = ref[0].double().cpu().numpy(), ref[3].item()
    assert np.all(np.isfinite(kl))
    assert np.all(np.abs(kl - r_kl) <= TOL_KL * (1 + r_kl))
    assert abs(loss[0] - r_loss) <= TOL_LOSS * abs(r_loss)
    rows = np.array(sorted({0, N - 1, N - 2} | set(np.random.default_rng(1).choice(N, 297, replace=False).tolist())))
    a = {k: x[k].double().cpu().numpy() for k in ("W_s", "W_t")}
    hs, ht = x["h_s"][torch.from_numpy(rows).cuda()].double().cpu().numpy(), x["h_t"][torch.from_numpy(rows).cuda()].double().cpu().numpy()
    o_kl, o_ls, o_lt, _ = orc.kl_rows(hs, a["W_s"], ht, a["W_t"], w.tau, np.arange(len(rows)))
    assert np.all(np.abs(kl[rows] - o_kl) <= TOL_KL * (1 + o_kl))
    assert np.all(np.abs(ls[rows] - o_ls) <= TOL_LSE * (1 + np.abs(o_ls)))
    assert np.all(np.abs(lt[rows] - o_lt) <= TOL_LSE * (1 + np.abs(o_lt)))
