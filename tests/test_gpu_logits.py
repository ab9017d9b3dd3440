"""GPU parity of the logits-input "Fused KL" (hylo_fused_kl_logits) against the fp64 oracle.

Tolerances: per token |dkl| <= 1e-3 (1 + kl), mean loss 1e-4 relative, lse 2e-5 (1 + |lse|) as
for the hidden-state path; dz_s is stored in bf16, whose rounding alone is at most 2^-8 of each
element and ~1.7e-3 rms over many elements, so ||d dz_s||_F <= 2e-3 ||dz_s||_F.
"""
import numpy as np
import pytest
import torch

from hybrid_upcycling_gb300 import _lib, build, synthetic as syn
from oracle import kl_oracle as orc

pytestmark = pytest.mark.gpu

TOL_KL, TOL_LOSS, TOL_GRAD, TOL_LSE = 1e-3, 1e-4, 2e-3, 2e-5


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return _lib.load()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run(z_s, z_t, tau, gs=1.0, grad=True, ld=None):
    N, V = z_s.shape
    if ld is not None and ld != V:  # place the logits in rows of stride ld
        zs_buf = torch.zeros(N, ld, dtype=torch.bfloat16, device="cuda")
        zt_buf = torch.zeros(N, ld, dtype=torch.bfloat16, device="cuda")
        zs_buf[:, :V] = z_s
        zt_buf[:, :V] = z_t
        z_s, z_t = zs_buf[:, :V], zt_buf[:, :V]
    f = dict(dtype=torch.float32, device="cuda")
    kl, ls, lt, loss = (torch.full((n,), float("nan"), **f) for n in (N, N, N, 1))
    dz = None
    if grad:
        dz = torch.full((N, z_s.stride(0)), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :V]
    _lib.hylo_fused_kl_logits(z_s, z_t, tau, gs, kl, ls, lt, loss, dz)
    _lib.hylo_kl_sync_status()
    return dict(kl=kl, lse_s=ls, lse_t=lt, loss=loss, dz=dz)


def check(z_s, z_t, tau, gs=1.0, ld=None, loss_abs=0.0):
    g = run(z_s, z_t, tau, gs, ld=ld)
    kl, ls, lt, loss, G = orc.kl_from_logits(f64(z_s), f64(z_t), tau, gs)
    gk = f64(g["kl"])
    assert np.all(np.abs(gk - kl) <= TOL_KL * (1 + kl)), np.max(np.abs(gk - kl))
    assert abs(g["loss"].item() - loss) <= TOL_LOSS * abs(loss) + loss_abs, (g["loss"].item(), loss)
    assert np.all(np.abs(f64(g["lse_s"]) - ls) <= TOL_LSE * (1 + np.abs(ls)))
    assert np.all(np.abs(f64(g["lse_t"]) - lt) <= TOL_LSE * (1 + np.abs(lt)))
    if np.linalg.norm(G) == 0:  # V = 1: p_s = p_t = 1; G is formed from a gap of fp32 sums, ~1e-7 off
        N = z_s.shape[0]
        assert np.max(np.abs(f64(g["dz"]))) <= 1e-6 * abs(gs) / (tau * N)
        return g
    err = np.linalg.norm(f64(g["dz"]) - G) / np.linalg.norm(G)
    assert err <= TOL_GRAD, err
    return g


def logits(N, V, seed, st=1.28, ss=0.9):
    gen = torch.Generator("cuda").manual_seed(seed)
    z_t = (torch.randn(N, V, generator=gen, device="cuda") * st).to(torch.bfloat16)
    z_s = (torch.randn(N, V, generator=gen, device="cuda") * ss).to(torch.bfloat16)
    return z_s, z_t


@pytest.mark.parametrize("N,V,tau,gs,ld", [
    (300, 1000, 0.7, 1.3, None),     # V not a multiple of 32
    (257, 4096, 1.0, 1.0, 4104),     # padded rows (ld > V)
    (64, 33000, 2.0, 0.5, None),     # more chunks than threads
    (1, 5, 1.0, 1.0, 8),             # tiny
    (17, 1, 1.0, 1.0, 8),            # V = 1
    (9, 200000, 1.0, 1.0, None),     # large vocabulary, partial last chunk
    (300, 131072, 1.0, 1.0, None),   # whole chunks only
])
def test_dense_parity(N, V, tau, gs, ld):
    z_s, z_t = logits(N, V, seed=N + V)
    check(z_s, z_t, tau, gs, ld=ld, loss_abs=1e-7)


@pytest.mark.parametrize("tau", [0.02, 50.0])
def test_extreme_temperatures(tau):
    """tau = 0.02: near one-hot distributions, and exp((m_s - m_t)/tau) overflows fp32 on most
    rows, so the statistics switch to the direct KL form (the 'far' rows); tau = 50: nearly
    uniform distributions and a tiny KL."""
    z_s, z_t = logits(200, 3000, seed=77)
    check(z_s, z_t, tau, 1.0, loss_abs=1e-9)


@pytest.mark.parametrize("V,grad", [(64, True), (64, False), (8, True), (1000, False)])
def test_many_short_rows(V, grad):
    """Thousands of rows of one chunk each: warps turn rows over fast and may run ahead of the
    row's merging warp by several rows, which the slot barriers (partials, row values) must
    hold back; every row against the oracle, with and without the gradient pass."""
    z_s, z_t = logits(6000, V, seed=V + 3)
    if grad:
        check(z_s, z_t, 1.0, 1.0, loss_abs=1e-9)
    else:
        g = run(z_s, z_t, 1.0, grad=False)
        kl, ls, lt, loss, _ = orc.kl_from_logits(f64(z_s), f64(z_t), 1.0)
        assert np.all(np.abs(f64(g["kl"]) - kl) <= TOL_KL * (1 + kl))
        assert np.all(np.abs(f64(g["lse_s"]) - ls) <= TOL_LSE * (1 + np.abs(ls)))
        assert abs(g["loss"].item() - loss) <= TOL_LOSS * loss


def test_forward_only_matches_and_writes_no_gradient():
    z_s, z_t = logits(100, 3000, seed=2)
    a = run(z_s, z_t, 1.0, grad=False)
    b = run(z_s, z_t, 1.0, grad=True)
    for k in ("kl", "lse_s", "lse_t", "loss"):
        assert torch.equal(a[k], b[k])


def test_near_identical_logits_mean_loss():
    """z_s = z_t + 1e-2-scale noise: KL ~ 1e-5 from two ~log V terms (cancellation-free form)."""
    w = syn.WORKLOADS["llama3b_nearconv"].with_sizes(N=200, V=20000)
    z = syn.make_logits(w, device="cuda")
    g = check(z["z_s"], z["z_t"], 1.0)
    assert g["loss"].item() < 1e-3


def test_one_outlier_word_gradient():
    """z_t = z_s except on one word: on every other word p_s and p_t differ only through the
    normalisers, by a factor exp(-(lse_s - lse_t)) with |lse_s - lse_t| ~ 1e-5, so dz_s there
    is p_t (exp(-gap) - 1). Checked on those words alone: a difference of two rounded
    probabilities (each ~1e-7 relative) would miss it by percents; the kernel forms p_t (2^D - 1)
    from the gap it derives from its own statistics."""
    z_s, _ = logits(400, 5000, seed=31, ss=1.1)
    z_t = z_s.clone()
    z_t[:, 7] = (z_t[:, 7].float() + 0.05).to(torch.bfloat16)
    g = check(z_s, z_t, 1.0, loss_abs=1e-9)
    assert 0 < g["loss"].item() < 1e-4
    *_, G = orc.kl_from_logits(f64(z_s), f64(z_t), 1.0)
    rest = np.ones(5000, dtype=bool)
    rest[7] = False
    err = np.linalg.norm(f64(g["dz"])[:, rest] - G[:, rest]) / np.linalg.norm(G[:, rest])
    print(f"normaliser-only words: dz rel err {err:.2e}")
    assert err <= TOL_GRAD, err


def test_hidden_state_and_logits_paths_agree():
    """The logits path on logits the hidden-state workload would produce: same statistics as
    the oracle at the same tolerances (a cross-check of the shared row statistics)."""
    w = syn.WORKLOADS["qwen17b_8b"].with_sizes(N=128, V=12000)
    z = syn.make_logits(w, device="cuda")
    check(z["z_s"], z["z_t"], w.tau, 1.0)


def test_full_size_logits_sampled():
    w = syn.WORKLOADS["llama1b_8b_8k"]
    z = syn.make_logits(w, device="cuda")
    g = run(z["z_s"], z["z_t"], w.tau)
    kl_g = g["kl"].double()
    assert torch.all(torch.isfinite(kl_g))
    assert abs(g["loss"].item() - kl_g.mean().item()) <= 1e-6 * kl_g.mean().item()
    rows = np.array(sorted({0, 1, w.N - 1, 4095, 4096} | set(np.random.default_rng(5).choice(w.N, 60, replace=False).tolist())))
    kl, ls, lt, _, G = orc.kl_from_logits(f64(z["z_s"][rows]), f64(z["z_t"][rows]), w.tau)
    G *= len(rows) / w.N  # the oracle's G above was normalised by the sample size
    gk = f64(g["kl"][rows])
    assert np.all(np.abs(gk - kl) <= TOL_KL * (1 + kl))
    assert np.all(np.abs(f64(g["lse_t"][rows]) - lt) <= TOL_LSE * (1 + np.abs(lt)))
    err = np.linalg.norm(f64(g["dz"][rows]) - G) / np.linalg.norm(G)
    print(f"logits full size: kl max err {np.max(np.abs(gk - kl)):.2e}, dz rows rel {err:.2e}")
    assert err <= TOL_GRAD


def test_autograd_wrapper_matches_oracle():
    """kl.fused_logits_kl as an autograd function on logits whose rows are not a multiple of 8
    (the wrapper pads them): loss, per-row KL and z_s.grad through loss.backward() (upstream 1:
    the kernel's single bf16 rounding), then upstream 2.5 (one more bf16 rounding, twice the
    bound); no gradient for z_t."""
    from hybrid_upcycling_gb300.kl import fused_logits_kl
    z_s, z_t = logits(130, 1001, seed=90)
    kl_r, _, _, loss_r, G = orc.kl_from_logits(f64(z_s), f64(z_t), 1.3)
    zs = z_s.clone().requires_grad_(True)
    loss, kl = fused_logits_kl(zs, z_t, 1.3)
    loss.backward()
    assert abs(loss.item() - loss_r) <= TOL_LOSS * loss_r
    assert np.all(np.abs(f64(kl) - kl_r) <= TOL_KL * (1 + kl_r))
    assert zs.grad.dtype == torch.bfloat16 and zs.grad.shape == z_s.shape
    assert np.linalg.norm(f64(zs.grad) - G) / np.linalg.norm(G) <= TOL_GRAD
    zs.grad = None
    loss, _ = fused_logits_kl(zs, z_t, 1.3)
    (2.5 * loss).backward()
    assert np.linalg.norm(f64(zs.grad) - 2.5 * G) / np.linalg.norm(2.5 * G) <= 2 * TOL_GRAD
    assert z_t.grad is None


def test_bench_configuration_against_the_oracle():
    """65536 x 128256 logits, the size bench.py --path logits times, with the workload's first
    U = 1024 rows repeated over all rows, so that the fp64 oracle evaluates only U distinct rows:
    every row's KL and the exact mean loss, dz_s on 512 rows spread over the range, and rows with
    equal inputs give equal bits."""
    w = syn.WORKLOADS["stage2_64k"]
    z = syn.make_logits(w.with_sizes(N=1024), device="cuda")
    U, N = 1024, w.N
    z_s = z["z_s"].repeat(N // U, 1).contiguous()
    z_t = z["z_t"].repeat(N // U, 1).contiguous()
    kl_u, _, _, loss_u, G_u = orc.kl_from_logits(f64(z["z_s"]), f64(z["z_t"]), w.tau)
    G_u *= U / N  # the oracle normalised by its own U rows; the kernel by all N
    g = run(z_s, z_t, w.tau)
    kl_ref = np.tile(kl_u, N // U)
    assert np.all(np.abs(f64(g["kl"]) - kl_ref) <= TOL_KL * (1 + kl_ref))
    assert abs(g["loss"].item() - loss_u) <= TOL_LOSS * loss_u
    rows = np.array(sorted({0, 1, U - 1, U, N - 1} | set(np.random.default_rng(3).choice(N, 507, replace=False).tolist())))
    r = torch.from_numpy(rows).cuda()
    err = np.linalg.norm(f64(g["dz"][r]) - G_u[rows % U]) / np.linalg.norm(G_u[rows % U])
    print(f"logits 65536 x 128256: dz rows rel {err:.2e}")
    assert err <= TOL_GRAD
    assert torch.equal(g["dz"][r], g["dz"][torch.from_numpy(rows % U).cuda()])
