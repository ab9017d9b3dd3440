"""GPU parity: the sm_103a library (through its C ABI) against the fp64 oracle.

Tolerances (stated for the fused hidden-state KL):
  per token   |kl_gpu - kl_ref| <= 1e-3 (1 + kl_ref)
  mean loss   |L_gpu - L_ref| <= 1e-4 |L_ref|
  gradients   ||g_gpu - g_ref||_F <= 2e-3 ||g_ref||_F   for dh_s and dW_s
  lse         |lse_gpu - lse_ref| <= 2e-5 (1 + |lse_ref|)   (fp32 logits and sums; derived)
Small shapes are compared densely; the full workload sizes on sampled tokens (the oracle
recomputes each sampled token over the whole vocabulary), on a dense full-vocabulary token
subset, and through invariants that hold at any size.
"""
import math
import os

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


def run(x, tau, token_chunk=4096, grad_scale=1.0, backward=True, stream=None, use_gap=True, split=False):
    dev = x["h_s"].device
    N, d_s = x["h_s"].shape
    V, d_t = x["W_t"].shape
    wsb = (_lib.hylo_kl_workspace_bytes_split if split else _lib.hylo_kl_workspace_bytes)(N, d_s, d_t, V, token_chunk)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    kl = torch.full((N,), float("nan"), device=dev)
    lse_s = torch.full((N,), float("nan"), device=dev)
    lse_t = torch.full((N,), float("nan"), device=dev)
    loss = torch.full((1,), float("nan"), device=dev)
    gap = torch.full((N,), float("nan"), device=dev) if use_gap else None
    _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], tau, token_chunk, kl, lse_s, lse_t, loss, ws,
                         stream=stream, lse_gap=gap)
    out = dict(kl=kl, lse_s=lse_s, lse_t=lse_t, loss=loss, gap=gap)
    if backward:
        dh = torch.full((N, d_s), float("nan"), device=dev)
        dW = torch.full((V, d_s), float("nan"), device=dev)
        bwd = _lib.hylo_kl_backward_split if split else _lib.hylo_kl_backward
        bwd(x["h_s"], x["W_s"], x["h_t"], x["W_t"], tau, token_chunk, lse_s, lse_t, grad_scale, dh, dW, ws,
            stream=stream, lse_gap=gap)
        out.update(dh=dh, dW=dW)
    _lib.hylo_kl_sync_status(stream)
    return out


def frob_rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_g_floor(hs, Ws, ht, Wt, tau, grad_scale, dh, dW):
    """Gradient errors of the exact G rounded once to bf16 (the backward's G precision)."""
    G = orc.kl_grad_logits(hs, Ws, ht, Wt, tau, grad_scale, hs.shape[0])
    Gb = torch.from_numpy(G).to(torch.bfloat16).double().numpy()
    return frob_rel(Gb @ Ws, dh), frob_rel(Gb.T @ hs, dW)


def check_dense(x, tau, token_chunk=4096, grad_scale=1.0, loss_abs=0.0, use_gap=True, tol_loss=TOL_LOSS,
                bf16_floor=False):
    """Every output against the oracle. bf16_floor: cases where each token's gradient is
    dominated by one or two words, so dh_s / dW_s carry the bf16 rounding of single numbers
    (up to 2^-8); the gradients are then held to the error of the exact G rounded once to bf16
    (x 1.1) where that exceeds the 2e-3 bound."""
    g = run(x, tau, token_chunk, grad_scale, use_gap=use_gap)
    hs, Ws, ht, Wt = (f64(x[k]) for k in ("h_s", "W_s", "h_t", "W_t"))
    kl, ls, lt, loss = orc.kl_forward(hs, Ws, ht, Wt, tau)
    dh, dW = orc.kl_backward(hs, Ws, ht, Wt, tau, grad_scale=grad_scale)
    gk = f64(g["kl"])
    assert np.all(np.isfinite(gk))
    assert np.all(np.abs(gk - kl) <= TOL_KL * (1 + kl)), np.max(np.abs(gk - kl) / (1 + kl))
    gl = float(g["loss"].item())
    assert abs(gl - loss) <= tol_loss * abs(loss) + loss_abs, (gl, loss)
    assert np.all(np.abs(f64(g["lse_s"]) - ls) <= TOL_LSE * (1 + np.abs(ls)))
    assert np.all(np.abs(f64(g["lse_t"]) - lt) <= TOL_LSE * (1 + np.abs(lt)))
    if use_gap:  # the gap is at least as accurate as the lse values themselves
        assert np.all(np.abs(f64(g["gap"]) - (ls - lt)) <= TOL_LSE * (1 + np.abs(ls)))
    tol_dh = tol_dW = TOL_GRAD
    if bf16_floor:
        f_dh, f_dW = bf16_g_floor(hs, Ws, ht, Wt, tau, grad_scale, dh, dW)
        tol_dh, tol_dW = max(TOL_GRAD, 1.1 * f_dh), max(TOL_GRAD, 1.1 * f_dW)
        print(f"bf16-G floor: dh {f_dh:.2e}, dW {f_dW:.2e}")
    assert frob_rel(f64(g["dh"]), dh) <= tol_dh, frob_rel(f64(g["dh"]), dh)
    assert frob_rel(f64(g["dW"]), dW) <= tol_dW, frob_rel(f64(g["dW"]), dW)
    return g


def gen(N, d_s, d_t, V, seed, w_std=0.05, normalise=False, device="cuda"):
    w = syn.Workload("case", 0, N, d_s, d_t, V, 1.0, w_std, normalise)
    return syn.make_inputs(w, device=device, seed=seed)


# ------------------------------------------------------------------------- dense, small shapes

@pytest.mark.parametrize("token_chunk", [4096, 7])
def test_tiny_workload(token_chunk):
    w = syn.WORKLOADS["tiny"]
    check_dense(syn.make_inputs(w, device="cuda"), w.tau, token_chunk)


def test_rational_golden_case():
    import importlib.util
    import json
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("rational_case", os.path.join(here, "rational_case.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    ref = json.load(open(os.path.join(here, "rational_case.json")))
    x = {k: torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).cuda()
         for k, v in zip(("h_s", "W_s", "h_t", "W_t"), mod.inputs())}
    for k, v in zip(("h_s", "W_s", "h_t", "W_t"), mod.inputs()):
        assert np.array_equal(f64(x[k]), v)  # the rationals are exact in bf16
    g = run(x, ref["tau"], grad_scale=ref["grad_scale"])
    kl = np.array(ref["kl"])
    assert np.all(np.abs(f64(g["kl"]) - kl) <= TOL_KL * (1 + kl))
    assert abs(g["loss"].item() - ref["loss"]) <= TOL_LOSS * ref["loss"]
    assert frob_rel(f64(g["dh"]), np.array(ref["dh_s"])) <= TOL_GRAD
    assert frob_rel(f64(g["dW"]), np.array(ref["dW_s"])) <= TOL_GRAD


@pytest.mark.parametrize("N,d_s,d_t,V,tau,chunk,gs,w_std", [
    (300, 136, 200, 1000, 0.7, 128, 1.0, 0.1),       # ragged everything, 3 chunks
    (1061, 256, 512, 8269, 2.0, 512, 0.37, 0.1),     # several tiles each way, ragged tails
    (129, 64, 64, 257, 1.0, 4096, 1.0, 0.1),         # one row and one column past a tile
    (129, 64, 64, 257, 1.0, 64, -0.5, 0.1),          # negative upstream gradient, 3 chunks
    (1, 8, 8, 3, 1.0, 4096, 1.0, 0.1),               # minimum sizes
    (300, 8192, 16392, 2000, 1.0, 4096, 1.0, 0.01),  # wide hidden states (a 70B-class teacher), ragged K
    (20000, 64, 64, 300, 1.0, 4096, 1.0, 0.1),       # many short units: 2 vocabulary tiles, 5 chunks
])
def test_ragged_shapes(N, d_s, d_t, V, tau, chunk, gs, w_std):
    # w_std keeps the logits' spread near the workloads' (std ~1.3 at the wide shapes): the
    # tensor cores' fp32 accumulation error grows with K and |z| (measured: logits of std 13
    # over K = 16392 put lse ~1e-3 low, past the 2e-5 (1 + |lse|) bound derived for K <= 4096)
    x = gen(N, d_s, d_t, V, seed=N + V, w_std=w_std)
    check_dense(x, tau, chunk, gs, loss_abs=1e-7)


@pytest.mark.parametrize("tau", [0.05, 40.0])
def test_extreme_temperatures(tau):
    """Near one-hot (tau = 0.05: exp((m_s - m_t)/tau) overflows fp32, the direct KL form; each
    token's gradient is then one or two words, held to the bf16-G floor) and nearly uniform
    (tau = 40: tiny KL) distributions, forward and backward."""
    x = gen(300, 128, 256, 3000, seed=31, w_std=0.1)
    check_dense(x, tau, 4096, 1.0, loss_abs=1e-9, bf16_floor=tau < 1)


def test_largest_hidden_size():
    """d_s = 65536, the largest hidden size the ABI accepts. The tensor cores accumulate each
    logit in fp32 over K/16 steps, each rounding the running sum; the result can drift by up to
    (K/16) 2^-23 of the logits' scale in one direction (measured here: the mean loss 1.3e-4
    low). The mean-loss bound is that drift, 4.9e-4 at K = 65536, instead of 1e-4; every
    other bound is the usual one."""
    x = gen(3, 65536, 64, 17, seed=20, w_std=0.005)
    check_dense(x, 1.5, 4096, 1.0, loss_abs=1e-7, tol_loss=(65536 / 16) * 2.0 ** -23)


def test_vocab_of_one_gives_zero():
    """V = 1: both distributions are a point mass, KL = 0 and G = 0 up to the fp32 accuracy of
    the row statistics (the gap lse_s - lse_t = z_s - z_t comes from fp32 sums, ~1e-7 off)."""
    N = 33
    x = gen(N, 16, 24, 1, seed=5)
    g = run(x, 1.5)
    assert torch.all(g["kl"].abs() <= 1e-6)
    z_s = (x["h_s"].double() @ x["W_s"].double().T)[:, 0]
    assert torch.allclose(g["lse_s"].double(), z_s / 1.5, rtol=1e-6, atol=1e-6)
    gmax = 1e-6 / (1.5 * N)  # |p_s - p_t| = |2^D - 1| with |D| ~ 1e-7
    assert g["dh"].abs().max().item() <= gmax * x["W_s"].float().abs().max().item() + 1e-30
    assert g["dW"].abs().max().item() <= gmax * N * x["h_s"].float().abs().max().item() + 1e-30


def test_identical_student_and_teacher_give_exact_zero():
    x = gen(200, 128, 128, 3000, seed=9, w_std=0.1)
    x["h_t"], x["W_t"] = x["h_s"].clone(), x["W_s"].clone()
    g = run(x, 1.0, token_chunk=64)
    assert torch.all(g["kl"] == 0), g["kl"].abs().max()
    assert torch.all(g["dh"] == 0) and torch.all(g["dW"] == 0)
    assert torch.equal(g["lse_s"], g["lse_t"])


def outlier_case():
    """Teacher = student except one vocabulary row: d = 0 on every other column and O(1e-2) on
    that one, so p_s and p_t agree to ~4e-5 on almost every word."""
    x = gen(500, 128, 128, 4000, seed=21, w_std=0.1)
    x["h_t"] = x["h_s"].clone()
    Wt = x["W_s"].clone()
    Wt[7] = (Wt[7].float() + 0.03 * torch.randn(128, device="cuda", generator=torch.Generator("cuda").manual_seed(5))).to(torch.bfloat16)
    x["W_t"] = Wt
    return x


def test_single_outlier_vocab_row():
    """Small KL with one large |d| (both branches of the cancellation-free sum, the mean-loss
    bound at a small loss). Forward outputs and the precise gap at the usual tolerances.

    The gradient of each token here is dominated by ONE word (G[n, 7]), so dh_s[n] is one bf16
    number times a row of W_s and carries that number's rounding error, up to 2^-8 relative:
    no sum averages it. The 2e-3 bound is therefore out of reach for any bf16 G on this case;
    the check is that the kernel is as accurate as the exact G rounded once to bf16 (its own
    fp32 arithmetic, p_t (2^D - 1) with the precise gap, adds almost nothing)."""
    x = outlier_case()
    g = run(x, 1.0, 256)
    hs, Ws, ht, Wt = (f64(x[k]) for k in ("h_s", "W_s", "h_t", "W_t"))
    kl, ls, lt, loss = orc.kl_forward(hs, Ws, ht, Wt, 1.0)
    gk = f64(g["kl"])
    assert np.all(np.abs(gk - kl) <= TOL_KL * (1 + kl))
    assert abs(g["loss"].item() - loss) <= TOL_LOSS * loss, (g["loss"].item(), loss)
    assert np.all(np.abs(f64(g["lse_s"]) - ls) <= TOL_LSE * (1 + np.abs(ls)))
    err = np.max(np.abs(f64(g["gap"]) - (ls - lt)))
    assert err <= 5e-7, err
    assert 0 < loss < 1e-2
    dh, dW = orc.kl_backward(hs, Ws, ht, Wt, 1.0)
    G = orc.kl_grad_logits(hs, Ws, ht, Wt, 1.0, 1.0, hs.shape[0])
    Gb = torch.from_numpy(G).to(torch.bfloat16).double().numpy()
    floor_dh, floor_dW = frob_rel(Gb @ Ws, dh), frob_rel(Gb.T @ hs, dW)
    e_dh, e_dW = frob_rel(f64(g["dh"]), dh), frob_rel(f64(g["dW"]), dW)
    print(f"outlier: gap err {err:.1e}; dh {e_dh:.2e} (bf16-G floor {floor_dh:.2e}), "
          f"dW {e_dW:.2e} (floor {floor_dW:.2e})")
    assert e_dh <= max(TOL_GRAD, 1.1 * floor_dh), (e_dh, floor_dh)
    assert e_dW <= max(TOL_GRAD, 1.1 * floor_dW), (e_dW, floor_dW)
    assert floor_dh <= 2.0 ** -8


def test_backward_without_gap_matches_on_ordinary_rows():
    """lse_gap is optional: with NULL the backward uses lse_s - lse_t, which is accurate enough
    wherever p_s and p_t are not near-identical."""
    check_dense(gen(300, 128, 256, 3000, seed=8, w_std=0.08), 1.0, 4096, use_gap=False)


def test_near_converged_cancellation():
    """Student logits = teacher logits + 1e-2-scale noise: KL ~ 7e-5 from two ~log V terms."""
    w = syn.WORKLOADS["llama3b_nearconv"].with_sizes(N=700, V=6000)
    x = syn.make_inputs(w, device="cuda")
    g = check_dense(x, 1.0, 256)
    assert 2e-5 < g["loss"].item() < 2e-4
    hs, Ws, ht, Wt = (f64(x[k]) for k in ("h_s", "W_s", "h_t", "W_t"))
    _, ls, lt, _ = orc.kl_forward(hs, Ws, ht, Wt, 1.0)
    err = np.max(np.abs(f64(g["gap"]) - (ls - lt)))
    err_diff = np.max(np.abs((f64(g["lse_s"]) - f64(g["lse_t"])) - (ls - lt)))
    print(f"near-converged: gap max err {err:.2e} (lse_s - lse_t: {err_diff:.2e})")
    # here both are limited by the fp32 tensor-core accumulation of z_s and z_t (~1e-6 of a
    # logit, not independent across words), not by the statistics
    assert err <= 2e-5


def test_token_chunk_invariance_and_determinism():
    x = gen(600, 128, 256, 5000, seed=3, w_std=0.08)
    a = run(x, 1.0, token_chunk=4096)
    b = run(x, 1.0, token_chunk=100)
    c = run(x, 1.0, token_chunk=4096)
    for k in ("kl", "lse_s", "lse_t", "loss", "dh", "dW"):
        assert torch.equal(a[k], c[k]), k  # bit-identical reruns
    for k in ("kl", "lse_s", "lse_t", "loss"):
        assert torch.equal(a[k], b[k]), k  # the forward does not depend on the chunk
    # the gradients differ only by fp32 summation order (the token and vocabulary blocks over
    # which dh_s and dW_s are accumulated depend on the chunk)
    assert frob_rel(f64(b["dh"]), f64(a["dh"])) < 1e-6
    assert frob_rel(f64(b["dW"]), f64(a["dW"])) < 1e-6


@pytest.mark.parametrize("chunk", [0, 1, 600, 10 ** 9])
def test_token_chunk_extremes(chunk):
    """token_chunk 0 means 4096 (bit-identical); 1 is rounded up to one 256-row block; N itself
    is one block; 10^9 is capped (at 32768 rows, then at N rounded up to 256). The forward never
    depends on the chunk; the gradients agree to fp32 summation order."""
    x = gen(600, 128, 256, 5000, seed=3, w_std=0.08)
    a = run(x, 1.0, token_chunk=4096)
    b = run(x, 1.0, token_chunk=chunk)
    for k in ("kl", "lse_s", "lse_t", "loss"):
        assert torch.equal(a[k], b[k]), k
    if chunk == 0:
        assert torch.equal(a["dh"], b["dh"]) and torch.equal(a["dW"], b["dW"])
    assert frob_rel(f64(b["dh"]), f64(a["dh"])) < 1e-6
    assert frob_rel(f64(b["dW"]), f64(a["dW"])) < 1e-6


def test_runs_on_a_side_stream():
    x = gen(256, 64, 128, 700, seed=11)
    ref = run(x, 1.0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = run(x, 1.0, stream=s)
    s.synchronize()
    for k in ref:
        assert torch.equal(ref[k], got[k]), k


def test_same_results_beside_a_concurrent_kernel():
    """The fused kernels pace clusters against each other; with another stream's kernels holding
    SMs, some clusters start late, the pacing gives up (bounded wait) and the results are still
    the same bits as in a call that ran alone."""
    x = gen(2048, 256, 512, 20000, seed=17, w_std=0.08)
    ref = run(x, 1.0, token_chunk=1024)
    busy, ours = torch.cuda.Stream(), torch.cuda.Stream()
    a = torch.randn(8192, 8192, device="cuda").to(torch.bfloat16)
    torch.cuda.synchronize()
    with torch.cuda.stream(busy):
        for _ in range(60):
            a = (a @ a) * 1e-3
    with torch.cuda.stream(ours):
        got = run(x, 1.0, token_chunk=1024, stream=ours)
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(ref[k], got[k]), k


def test_library_allocates_no_device_memory():
    """The caller owns every byte: after a first call on the device (one-time set-up), a
    forward + backward leaves the device's free memory unchanged, so the peak extra memory is
    the workspace the caller passed -- O(N) statistics or one G ring of at most 128 MiB, not
    the O(N V) of dense logits."""
    N, d_s, d_t, V, chunk = 1000, 128, 256, 5000, 512
    x = gen(N, d_s, d_t, V, seed=12)
    ws = torch.empty(_lib.hylo_kl_workspace_bytes(N, d_s, d_t, V, chunk), dtype=torch.uint8, device="cuda")
    f = dict(dtype=torch.float32, device="cuda")
    kl, ls, lt, gap = (torch.empty(N, **f) for _ in range(4))
    loss = torch.empty(1, **f)
    dh, dW = torch.empty(N, d_s, **f), torch.empty(V, d_s, **f)

    def call():
        _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 1.0, chunk, kl, ls, lt, loss, ws, lse_gap=gap)
        _lib.hylo_kl_backward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 1.0, chunk, ls, lt, 1.0, dh, dW, ws, lse_gap=gap)
        _lib.hylo_kl_sync_status()

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    # O(N) statistics or the G ring of at most 128 MiB, whichever is larger (+ 1280 B of
    # counters); below one model's fp32 logits
    assert ws.numel() <= max(6 * 32 * N * 4, 128 << 20) + 1280
    assert ws.numel() < 4 * N * V


@pytest.mark.parametrize("split_g", [False, True])
def test_autograd_wrapper(split_g):
    from hybrid_upcycling_gb300.kl import fused_hidden_state_kl
    w = syn.WORKLOADS["tiny"]
    x = syn.make_inputs(w, device="cuda")
    h_s = x["h_s"].clone().requires_grad_(True)
    W_s = x["W_s"].clone().requires_grad_(True)
    loss, kl = fused_hidden_state_kl(h_s, W_s, x["h_t"], x["W_t"], 1.0, split_g=split_g)
    (2.0 * loss).backward()
    ref = orc.kl_backward(f64(x["h_s"]), f64(x["W_s"]), f64(x["h_t"]), f64(x["W_t"]), 1.0, grad_scale=2.0)
    # the wrapper returns bf16 gradients (the input dtype): allow bf16 rounding on top
    assert frob_rel(f64(h_s.grad), ref[0]) <= TOL_GRAD + 4e-3
    assert frob_rel(f64(W_s.grad), ref[1]) <= TOL_GRAD + 4e-3
    assert abs(loss.item() - float(np.mean(f64(kl)))) < 1e-6


def test_functional_fwd_bwd_fp32_gradients_into_caller_buffers():
    """kl_fwd_bwd: fp32 gradients of grad_scale * loss written into the caller's buffers, equal
    to the plain C-ABI calls (one workspace shared by the forward and the backward)."""
    from hybrid_upcycling_gb300.kl import kl_fwd_bwd
    x = gen(300, 136, 200, 1000, seed=77, w_std=0.1)
    N, d_s, V = 300, 136, 1000
    dh = torch.full((N, d_s), float("nan"), device="cuda")
    dW = torch.full((V, d_s), float("nan"), device="cuda")
    loss, kl, dh2, dW2 = kl_fwd_bwd(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 0.7, 128, grad_scale=-1.5, dh_s=dh, dW_s=dW)
    assert dh2 is dh and dW2 is dW and dh.dtype == torch.float32
    ref = run(x, 0.7, 128, grad_scale=-1.5)
    assert torch.equal(kl, ref["kl"]) and torch.equal(loss, ref["loss"])
    assert torch.equal(dh, ref["dh"]) and torch.equal(dW, ref["dW"])


# ------------------------------------------------------------------- full workload sizes

def _sample_rows(N, chunk, k, seed):
    rng = np.random.default_rng(seed)
    fixed = {0, N - 1, min(N - 1, 127), min(N - 1, 128)}
    for c in range(chunk, N, chunk):
        fixed |= {c - 1, c}
    rest = rng.choice(N, size=max(0, k - len(fixed)), replace=False)
    return np.array(sorted(fixed | set(int(r) for r in rest)))


@pytest.mark.parametrize("name", ["llama1b_8b_8k", "stage2_64k", "qwen17b_8b", "llama3b_nearconv"])
def test_full_size_workload(name):
    w = syn.WORKLOADS[name]
    x = syn.make_inputs(w, device="cuda")
    g = run(x, w.tau, w.token_chunk)
    N = w.N
    kl_g = g["kl"].double()
    assert torch.all(torch.isfinite(kl_g)) and torch.all(torch.isfinite(g["dh"])) and torch.all(torch.isfinite(g["dW"]))
    # the loss is the mean of the per-token values
    assert abs(g["loss"].item() - kl_g.mean().item()) <= 1e-6 * abs(kl_g.mean().item())
    # sampled tokens against the oracle, over the whole vocabulary
    rows = _sample_rows(N, w.token_chunk, 160, seed=w.seed)
    Ws, Wt = f64(x["W_s"]), f64(x["W_t"])
    hs_r, ht_r = f64(x["h_s"][rows]), f64(x["h_t"][rows])
    kl, ls, lt, dh = orc.kl_rows(hs_r, Ws, ht_r, Wt, w.tau, np.arange(len(rows)), n_total=N)
    gk = f64(g["kl"][rows])
    assert np.all(np.abs(gk - kl) <= TOL_KL * (1 + kl)), np.max(np.abs(gk - kl))
    if w.near_converged:
        # the cancellation-free form keeps each token's relative error far below the mean-loss bound
        assert np.all(np.abs(gk - kl) <= TOL_LOSS * kl), np.max(np.abs(gk - kl) / kl)
    assert abs(gk.mean() - kl.mean()) <= TOL_LOSS * kl.mean()
    assert np.all(np.abs(f64(g["lse_s"][rows]) - ls) <= TOL_LSE * (1 + np.abs(ls)))
    assert np.all(np.abs(f64(g["lse_t"][rows]) - lt) <= TOL_LSE * (1 + np.abs(lt)))
    e_dh = frob_rel(f64(g["dh"][rows]), dh)
    print(f"{name}: sampled kl max err {np.max(np.abs(gk - kl)):.2e}, mean rel {abs(gk.mean() - kl.mean()) / kl.mean():.2e}, "
          f"dh rows rel {e_dh:.2e}")
    assert e_dh <= TOL_GRAD
    # invariants of dW_s at full size: zero column sums, and <dW_s, W_s> = <dh_s, h_s>
    dW = g["dW"].double()
    col = dW.sum(0).abs()
    assert torch.all(col <= 1e-3 * dW.abs().sum(0) + 1e-30)
    a = (dW * x["W_s"].double()).sum().item()
    b = (g["dh"].double() * x["h_s"].double()).sum().item()
    bound = (dW.norm() * x["W_s"].double().norm()).item()
    # Both sides sum the same bf16-G products; they differ only by fp32 accumulation, longest
    # in dh_s (K = V, one accumulator update per 16 products): allow (V/16) * 2^-24 of the bound.
    acc_tol = max(1e-5, (w.V / 16) * 2.0 ** -24)
    print(f"{name}: trace gap {abs(a - b) / bound:.2e} (tol {acc_tol:.2e})")
    assert abs(a - b) <= acc_tol * bound
    del g, dW
    torch.cuda.empty_cache()
    # dense dW_s over the full vocabulary and hidden size on a token subset (lse from the oracle
    # would be circular here, so the subset is its own problem with its own mean)
    sub = rows[:96]
    xs = {k: x[k][sub].contiguous() if k.startswith("h") else x[k] for k in x}
    gs = run(xs, w.tau, w.token_chunk, grad_scale=0.5)
    dh_ref, dW_ref = orc.kl_backward(f64(xs["h_s"]), Ws, f64(xs["h_t"]), Wt, w.tau, grad_scale=0.5)
    e_w, e_h = frob_rel(f64(gs["dW"]), dW_ref), frob_rel(f64(gs["dh"]), dh_ref)
    print(f"{name}: token-subset dense dW rel {e_w:.2e}, dh rel {e_h:.2e}")
    assert e_w <= TOL_GRAD
    assert e_h <= TOL_GRAD


# ------------------------------------------------------------- G as two bf16 terms (split)

def split_errors(x, tau, token_chunk, grad_scale=1.0):
    g = run(x, tau, token_chunk, grad_scale, split=True)
    hs, Ws, ht, Wt = (f64(x[k]) for k in ("h_s", "W_s", "h_t", "W_t"))
    kl, ls, lt, loss = orc.kl_forward(hs, Ws, ht, Wt, tau)
    dh, dW = orc.kl_backward(hs, Ws, ht, Wt, tau, grad_scale=grad_scale)
    return g, frob_rel(f64(g["dh"]), dh), frob_rel(f64(g["dW"]), dW)


# Derived bound: G = bf16(G) + bf16(G - bf16(G)) keeps ~16 significant bits (2^-16 = 1.5e-5 per
# element); fp32 logits, probabilities and GEMM accumulation add ~1e-6. 1e-4 leaves room for
# the sums' amplification; one bf16 rounding of G would give ~1e-3 here.
TOL_GRAD_SPLIT = 1e-4


@pytest.mark.parametrize("token_chunk", [4096, 100])
def test_split_g_ragged(token_chunk):
    x = gen(1061, 256, 512, 8269, seed=1061 + 8269, w_std=0.1)
    g, e_dh, e_dW = split_errors(x, 2.0, token_chunk, 0.37)
    print(f"split G (chunk {token_chunk}): dh {e_dh:.2e}, dW {e_dW:.2e}")
    assert e_dh <= TOL_GRAD_SPLIT and e_dW <= TOL_GRAD_SPLIT, (e_dh, e_dW)
    ref = run(x, 2.0, token_chunk, 0.37)
    for k in ("kl", "lse_s", "lse_t", "loss"):
        assert torch.equal(g[k], ref[k]), k  # the forward is the same call


def test_split_g_meets_the_bound_where_one_rounding_cannot():
    """The one-word-dominated cases whose plain-backward gradients sit at the bf16-G floor
    (above 2e-3): with G as two bf16 terms they are well inside the 2e-3 bound."""
    for x, tau in ((outlier_case(), 1.0), (gen(300, 128, 256, 3000, seed=31, w_std=0.1), 0.05)):
        _, e_dh, e_dW = split_errors(x, tau, 256)
        print(f"split G, tau {tau}: dh {e_dh:.2e}, dW {e_dW:.2e}")
        assert e_dh <= TOL_GRAD_SPLIT and e_dW <= TOL_GRAD_SPLIT, (tau, e_dh, e_dW)


def test_split_g_full_size_sampled():
    """hylo_kl_backward_split at the 8K-token workload's full size: sampled dh_s rows and a
    dense dW_s on a token subset against the oracle. With G this precise, dh_s's own fp32
    accumulation over K = V on the tensor cores is what remains: (V/16) 2^-24 = 4.8e-4 of the
    scale at V = 128256 (the bound the trace identity above uses), still 4x below 2e-3."""
    w = syn.WORKLOADS["llama1b_8b_8k"]
    x = syn.make_inputs(w, device="cuda")
    g = run(x, w.tau, w.token_chunk, split=True)
    rows = _sample_rows(w.N, w.token_chunk, 64, seed=w.seed + 1)
    Ws, Wt = f64(x["W_s"]), f64(x["W_t"])
    _, _, _, dh = orc.kl_rows(f64(x["h_s"][rows]), Ws, f64(x["h_t"][rows]), Wt, w.tau, np.arange(len(rows)),
                              n_total=w.N)
    e_dh = frob_rel(f64(g["dh"][rows]), dh)
    del g
    torch.cuda.empty_cache()
    sub = rows[:64]
    xs = {k: x[k][sub].contiguous() if k.startswith("h") else x[k] for k in x}
    gs = run(xs, w.tau, w.token_chunk, grad_scale=0.5, split=True)
    dh_ref, dW_ref = orc.kl_backward(f64(xs["h_s"]), Ws, f64(xs["h_t"]), Wt, w.tau, grad_scale=0.5)
    e_w = frob_rel(f64(gs["dW"]), dW_ref)
    print(f"split G full size: dh rows rel {e_dh:.2e}, token-subset dense dW rel {e_w:.2e}")
    assert e_dh <= max(TOL_GRAD_SPLIT, (w.V / 16) * 2.0 ** -24), e_dh
    assert e_w <= TOL_GRAD_SPLIT, e_w


def test_results_identical_when_clusters_start_late():
    """Pacing is a hint. Started while large matmuls on another stream hold the SMs, the
    forward's clusters begin at different times: clusters wait for absent peers up to the
    pacing limit and then switch pacing off for the launch, and the backward's persistent CTAs
    join its work queue late. Every output is bit-identical to an undisturbed run (the
    arithmetic and its order do not depend on timing)."""
    x = gen(8192, 256, 512, 30000, seed=41)
    a = run(x, 1.0)
    big = torch.randn(8192, 8192, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(big)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s2):
        for _ in range(4):
            torch.matmul(big, big, out=out)
    with torch.cuda.stream(s1):
        b = run(x, 1.0, stream=s1)
    torch.cuda.synchronize()
    for k in ("kl", "lse_s", "lse_t", "loss", "gap", "dh", "dW"):
        assert torch.equal(a[k], b[k]), k


def test_index_range_beyond_2_31_elements():
    """N = 2^21 + 37 tokens of d_s = 1024: h_s holds more than 2^31 elements (4.3 GB, byte
    offsets past 2^32), dh_s more than 2^31 fp32. The token rows repeat a period of U = 1024
    distinct rows, so the fp64 oracle evaluates the U distinct rows once: each token's KL and
    log-sum-exps are its row's, G carries the global N, dW_s = sum_u mult(u) G_u^T h_u. Every
    token's KL, the mean loss, dW_s, and dh_s on rows spread over the whole range (around the
    2^31-element offset and at the end) against it; tokens with the same inputs get the same
    bits."""
    U, N, d_s, d_t, V, tau = 1024, (1 << 21) + 37, 1024, 1536, 300, 1.0
    xu = gen(U, d_s, d_t, V, seed=55)
    reps = -(-N // U)
    x = {"h_s": xu["h_s"].repeat(reps, 1)[:N].contiguous(), "h_t": xu["h_t"].repeat(reps, 1)[:N].contiguous(),
         "W_s": xu["W_s"], "W_t": xu["W_t"]}
    assert x["h_s"].numel() > 2 ** 31
    g = run(x, tau)
    hu, Ws, htu, Wt = (f64(xu[k]) for k in ("h_s", "W_s", "h_t", "W_t"))
    kl_u, ls_u, lt_u, _ = orc.kl_forward(hu, Ws, htu, Wt, tau)
    mult = np.bincount(np.arange(N) % U, minlength=U).astype(np.float64)
    G_u = orc.kl_grad_logits(hu, Ws, htu, Wt, tau, 1.0, N)
    dW = (G_u * mult[:, None]).T @ hu
    loss = float(np.dot(mult, kl_u) / N)
    idx = torch.arange(N, device="cuda") % U
    kl_ref = torch.from_numpy(kl_u).cuda()[idx]
    assert torch.all((g["kl"].double() - kl_ref).abs() <= TOL_KL * (1 + kl_ref)).item()
    assert abs(g["loss"].item() - loss) <= TOL_LOSS * loss
    assert frob_rel(f64(g["dW"]), dW) <= TOL_GRAD, frob_rel(f64(g["dW"]), dW)
    rows = np.array(sorted({0, 1, U, (1 << 21) - 1, 1 << 21, (1 << 21) + 1, N - 1, N - 2}
                           | set(np.random.default_rng(7).choice(N, 200, replace=False).tolist())))
    dh_rows = f64(g["dh"][torch.from_numpy(rows).cuda()])
    dh_ref = G_u[rows % U] @ Ws
    assert frob_rel(dh_rows, dh_ref) <= TOL_GRAD, frob_rel(dh_rows, dh_ref)
    first = torch.from_numpy(rows % U).cuda()
    assert torch.equal(g["dh"][torch.from_numpy(rows).cuda()], g["dh"][first])
    assert torch.equal(g["kl"][torch.from_numpy(rows).cuda()], g["kl"][first])


def test_vocabulary_of_a_million_words():
    """V = 1,000,003 (ragged): 3907 vocabulary tiles in the forward, 87296-word blocks in the
    backward (the G ring's width rule at 256-token blocks) with a partial last block; every
    output against the dense oracle."""
    x = gen(200, 64, 96, 1_000_003, seed=77, w_std=0.1)
    check_dense(x, 1.0, 4096, 1.0, loss_abs=1e-7)


@pytest.mark.parametrize("d_s,d_t", [(520, 8), (264, 72)])
def test_student_wider_than_teacher(d_s, d_t):
    """d_t < d_s (the teacher's K-blocks are the fewer, one of them ragged at d_t = 8 or 72);
    every output against the dense oracle."""
    x = gen(333, d_s, d_t, 2100, seed=d_s + d_t, w_std=0.1)
    check_dense(x, 1.0, 128, 1.0, loss_abs=1e-7)


def test_forward_and_backward_replay_in_a_cuda_graph():
    """Forward + backward captured into a CUDA graph (after one eager call that sets the library
    up) and replayed twice: the outputs are bit-identical to the eager calls. The captured
    forward clears its pacing words with a captured memset and uses a tag reserved for captured
    launches, so every replay paces like an eager call; the backward's counters are cleared by
    its own captured memset."""
    x = gen(8192, 256, 512, 30000, seed=123, w_std=0.08)  # 224 work units: several waves, paced
    ref = run(x, 1.0)
    N, d_s = x["h_s"].shape
    V, d_t = x["W_t"].shape
    f = dict(dtype=torch.float32, device="cuda")
    ws = torch.empty(_lib.hylo_kl_workspace_bytes(N, d_s, d_t, V, 4096), dtype=torch.uint8, device="cuda")
    kl, lse_s, lse_t, gap = (torch.empty(N, **f) for _ in range(4))
    loss = torch.empty(1, **f)
    dh, dW = torch.empty(N, d_s, **f), torch.empty(V, d_s, **f)
    s = torch.cuda.Stream()

    def step():
        _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 1.0, 4096, kl, lse_s, lse_t, loss, ws,
                             stream=s, lse_gap=gap)
        _lib.hylo_kl_backward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 1.0, 4096, lse_s, lse_t, 1.0, dh, dW, ws,
                              stream=s, lse_gap=gap)

    with torch.cuda.stream(s):
        step()  # eager warm-up on the capture stream
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(2):
        for t in (kl, lse_s, lse_t, gap, loss, dh, dW):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        _lib.hylo_kl_sync_status()
        got = dict(kl=kl, lse_s=lse_s, lse_t=lse_t, loss=loss, gap=gap, dh=dh, dW=dW)
        for k in got:
            assert torch.equal(ref[k], got[k]), k
    # A forward alone, captured and replayed: its pacing words (after the 6 x 32 x N fp32
    # statistics: one per cluster, at most 128, then the switch; the backward's G ring reuses
    # that memory, hence the forward-only graph) carry the captured tag 1 and read finished for
    # every cluster that ran, and pacing was not switched off.
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], 1.0, 4096, kl, lse_s, lse_t, loss, ws,
                             stream=s, lse_gap=gap)
    g2.replay()
    torch.cuda.synchronize()
    _lib.hylo_kl_sync_status()
    assert torch.equal(ref["kl"], kl)
    off = (6 * 32 * N * 4 + 255) // 256 * 256
    words = ws[off:off + 8 * 129].view(torch.int64).cpu().tolist()
    ran = [w for w in words[:128] if (w >> 48) & 0xFFFF == 1]
    assert len(ran) >= 2
    assert all(w & ((1 << 48) - 1) == (1 << 48) - 1 for w in ran)
    assert (words[128] >> 48) & 0xFFFF != 1
