"""Pins for the fp64 oracle: checks against facts other than the oracle itself.

Each test would fail for a plausible slip in oracle/kl_oracle.py: a swapped KL direction
(two-class closed form), a tau^2 factor or a missing 1/tau (two-class, tau scaling,
Gaussian closed form, finite differences), a transposed operand or wrong index (finite
differences on non-square shapes, brute force, permutations), a dropped normalisation
(uniform student, library softmax), a per-chunk instead of global mean (chunk invariance).
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from oracle import kl_oracle as orc
from hybrid_upcycling_gb300 import synthetic as syn


def _rand_problem(rng, N, d_s, d_t, V, w_std=0.3):
    return (rng.standard_normal((N, d_s)), rng.standard_normal((V, d_s)) * w_std,
            rng.standard_normal((N, d_t)), rng.standard_normal((V, d_t)) * w_std)


# ----------------------------------------------------------------------------- exact cases

def test_identical_student_and_teacher_give_zero():
    rng = np.random.default_rng(1)
    h, W, _, _ = _rand_problem(rng, 9, 12, 12, 33)
    kl, lse_s, lse_t, loss = orc.kl_forward(h, W, h, W, 1.3)
    assert np.all(kl == 0.0) and loss == 0.0
    assert np.array_equal(lse_s, lse_t)
    dh, dW = orc.kl_backward(h, W, h, W, 1.3)
    assert np.all(dh == 0.0) and np.all(dW == 0.0)


def test_kl_nonnegative():
    for seed in range(5):
        rng = np.random.default_rng(100 + seed)
        kl, *_ = orc.kl_forward(*_rand_problem(rng, 17, 8, 16, 57, w_std=1.0), 0.7)
        assert np.all(kl >= -1e-14)


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


@pytest.mark.parametrize("tau", [0.5, 1.0, 2.0])
def test_two_class_closed_form(tau):
    """V = 2: KL between Bernoulli(p) and Bernoulli(q) with p = sigmoid((zt1-zt0)/tau)."""
    rng = np.random.default_rng(7)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 6, 5, 7, 2, w_std=0.8)
    kl, _, _, loss = orc.kl_forward(h_s, W_s, h_t, W_t, tau)
    for n in range(6):
        zt = [_dot(h_t[n], W_t[v]) for v in range(2)]
        zs = [_dot(h_s[n], W_s[v]) for v in range(2)]
        p = 1.0 / (1.0 + math.exp(-(zt[1] - zt[0]) / tau))
        q = 1.0 / (1.0 + math.exp(-(zs[1] - zs[0]) / tau))
        ref = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        assert abs(kl[n] - ref) <= 1e-12 * (1 + ref)
    assert abs(loss - float(np.mean(kl))) < 1e-15


def test_uniform_student_reduces_to_entropy():
    """W_s = 0 makes p_s uniform: KL = log V - H(p_t) (scipy's entropy of scipy's softmax)."""
    rng = np.random.default_rng(3)
    N, V, tau = 11, 40, 1.5
    h_s, _, h_t, W_t = _rand_problem(rng, N, 6, 9, V, w_std=0.9)
    W_s = np.zeros((V, 6))
    kl, lse_s, lse_t, _ = orc.kl_forward(h_s, W_s, h_t, W_t, tau)
    z_t = np.array([[_dot(h_t[n], W_t[v]) for v in range(V)] for n in range(N)])
    p_t = scipy.special.softmax(z_t / tau, axis=1)
    H = scipy.stats.entropy(p_t, axis=1)
    np.testing.assert_allclose(kl, math.log(V) - H, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_s, math.log(V), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_t, scipy.special.logsumexp(z_t / tau, axis=1), atol=1e-12)
    # both heads zero: both uniform, KL = 0
    kl0, *_ = orc.kl_forward(h_s, W_s, h_t, np.zeros_like(W_t), tau)
    assert np.all(np.abs(kl0) < 1e-15)


def test_matches_library_relative_entropy():
    rng = np.random.default_rng(5)
    N, V, tau = 13, 70, 0.8
    h_s, W_s, h_t, W_t = _rand_problem(rng, N, 10, 14, V, w_std=0.5)
    kl, lse_s, lse_t, _ = orc.kl_forward(h_s, W_s, h_t, W_t, tau)
    p_t = scipy.special.softmax(h_t @ W_t.T / tau, axis=1)
    p_s = scipy.special.softmax(h_s @ W_s.T / tau, axis=1)
    ref = scipy.special.rel_entr(p_t, p_s).sum(axis=1)
    np.testing.assert_allclose(kl, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse_s, scipy.special.logsumexp(h_s @ W_s.T / tau, axis=1), rtol=1e-13)


def test_brute_force_loops():
    """Plain Python loops (math.exp / math.log, no numpy) on a 3-token, 5-word problem."""
    rng = np.random.default_rng(11)
    N, d_s, d_t, V, tau, gs = 3, 4, 6, 5, 1.7, 0.9
    h_s, W_s, h_t, W_t = _rand_problem(rng, N, d_s, d_t, V, w_std=0.7)
    kl, lse_s, lse_t, loss = orc.kl_forward(h_s, W_s, h_t, W_t, tau)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, tau, grad_scale=gs)
    G = [[0.0] * V for _ in range(N)]
    for n in range(N):
        zs = [sum(h_s[n][j] * W_s[v][j] for j in range(d_s)) / tau for v in range(V)]
        zt = [sum(h_t[n][j] * W_t[v][j] for j in range(d_t)) / tau for v in range(V)]
        Zs = sum(math.exp(x) for x in zs)
        Zt = sum(math.exp(x) for x in zt)
        ps = [math.exp(x) / Zs for x in zs]
        pt = [math.exp(x) / Zt for x in zt]
        ref = sum(pt[v] * math.log(pt[v] / ps[v]) for v in range(V))
        assert abs(kl[n] - ref) < 1e-12
        assert abs(lse_s[n] - math.log(Zs)) < 1e-12 and abs(lse_t[n] - math.log(Zt)) < 1e-12
        for v in range(V):
            G[n][v] = gs * (ps[v] - pt[v]) / (tau * N)
    for n in range(N):
        for j in range(d_s):
            assert abs(dh[n][j] - sum(G[n][v] * W_s[v][j] for v in range(V))) < 1e-14
    for v in range(V):
        for j in range(d_s):
            assert abs(dW[v][j] - sum(G[n][v] * h_s[n][j] for n in range(N))) < 1e-14


def test_finite_difference_gradients():
    """Central differences of grad_scale * L in fp64 on a non-square problem."""
    rng = np.random.default_rng(13)
    N, d_s, d_t, V, tau, gs = 4, 6, 8, 16, 1.3, 2.5
    h_s, W_s, h_t, W_t = _rand_problem(rng, N, d_s, d_t, V, w_std=0.6)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, tau, grad_scale=gs)
    eps = 1e-6

    def L(hs, Ws):
        return gs * orc.kl_forward(hs, Ws, h_t, W_t, tau)[3]

    fd_h = np.zeros_like(h_s)
    for idx in np.ndindex(*h_s.shape):
        hp, hm = h_s.copy(), h_s.copy()
        hp[idx] += eps
        hm[idx] -= eps
        fd_h[idx] = (L(hp, W_s) - L(hm, W_s)) / (2 * eps)
    fd_W = np.zeros_like(W_s)
    for idx in np.ndindex(*W_s.shape):
        Wp, Wm = W_s.copy(), W_s.copy()
        Wp[idx] += eps
        Wm[idx] -= eps
        fd_W[idx] = (L(h_s, Wp) - L(h_s, Wm)) / (2 * eps)
    np.testing.assert_allclose(dh, fd_h, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dW, fd_W, rtol=1e-6, atol=1e-9)


# ----------------------------------------------------------------------------- symmetries

def test_token_permutation():
    rng = np.random.default_rng(17)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 10, 5, 7, 23)
    perm = rng.permutation(10)
    kl, *_ = orc.kl_forward(h_s, W_s, h_t, W_t, 1.0)
    klp, *_ = orc.kl_forward(h_s[perm], W_s, h_t[perm], W_t, 1.0)
    np.testing.assert_allclose(klp, kl[perm], rtol=1e-13, atol=1e-15)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, 1.0)
    dhp, dWp = orc.kl_backward(h_s[perm], W_s, h_t[perm], W_t, 1.0)
    np.testing.assert_allclose(dhp, dh[perm], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(dWp, dW, rtol=1e-12, atol=1e-16)


def test_joint_vocab_permutation():
    rng = np.random.default_rng(19)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 8, 5, 7, 29)
    perm = rng.permutation(29)
    kl, *_ = orc.kl_forward(h_s, W_s, h_t, W_t, 0.9)
    klp, *_ = orc.kl_forward(h_s, W_s[perm], h_t, W_t[perm], 0.9)
    np.testing.assert_allclose(klp, kl, rtol=1e-12, atol=1e-15)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, 0.9)
    dhp, dWp = orc.kl_backward(h_s, W_s[perm], h_t, W_t[perm], 0.9)
    np.testing.assert_allclose(dhp, dh, rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(dWp, dW[perm], rtol=1e-11, atol=1e-16)


def test_temperature_equals_weight_scaling():
    """tau=2 with W equals tau=1 with W/2 (power-of-two scaling is exact)."""
    rng = np.random.default_rng(23)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 7, 6, 9, 31, w_std=0.9)
    a = orc.kl_forward(h_s, W_s, h_t, W_t, 2.0)
    b = orc.kl_forward(h_s, W_s / 2, h_t, W_t / 2, 1.0)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13, atol=1e-15)
    dh2, dW2 = orc.kl_backward(h_s, W_s, h_t, W_t, 2.0)
    dh1, dW1 = orc.kl_backward(h_s, W_s / 2, h_t, W_t / 2, 1.0)
    np.testing.assert_allclose(dh2, dh1, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(dW2, 0.5 * dW1, rtol=1e-12, atol=1e-16)


def test_common_shift_of_student_head():
    """Adding one vector c to every row of W_s shifts each token's logits by h_s[n].c, a
    per-token constant, so the softmax and KL do not change."""
    rng = np.random.default_rng(29)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 6, 5, 8, 19)
    c = rng.standard_normal(5)
    kl, *_ = orc.kl_forward(h_s, W_s, h_t, W_t, 1.1)
    kls, *_ = orc.kl_forward(h_s, W_s + c[None, :], h_t, W_t, 1.1)
    np.testing.assert_allclose(kls, kl, rtol=1e-9, atol=1e-12)


def test_gradient_invariants():
    """sum_v G[n, v] = 0 gives zero column sums of dW_s; <dW_s, W_s> = <dh_s, h_s> because both
    equal sum_{n,v} G[n, v] z_s[n, v]."""
    rng = np.random.default_rng(31)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 12, 7, 9, 41)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, 1.0)
    scale = np.abs(dW).max()
    assert np.all(np.abs(dW.sum(axis=0)) < 1e-12 * scale * 41)
    a = float(np.sum(dW * W_s))
    b = float(np.sum(dh * h_s))
    assert abs(a - b) < 1e-12 * (abs(a) + 1e-30) + 1e-15


@pytest.mark.parametrize("chunk", [1, 7, 12, 4096])
def test_token_chunk_invariance(chunk):
    rng = np.random.default_rng(37)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 12, 5, 6, 17)
    ref = orc.kl_forward(h_s, W_s, h_t, W_t, 1.0, token_chunk=12)
    got = orc.kl_forward(h_s, W_s, h_t, W_t, 1.0, token_chunk=chunk)
    np.testing.assert_allclose(got[0], ref[0], rtol=1e-12, atol=1e-15)
    assert abs(got[3] - ref[3]) < 1e-14
    dh0, dW0 = orc.kl_backward(h_s, W_s, h_t, W_t, 1.0, token_chunk=12)
    dh1, dW1 = orc.kl_backward(h_s, W_s, h_t, W_t, 1.0, token_chunk=chunk)
    np.testing.assert_allclose(dh1, dh0, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(dW1, dW0, rtol=1e-12, atol=1e-16)


def test_rows_match_full():
    rng = np.random.default_rng(41)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 20, 6, 8, 25)
    kl, lse_s, lse_t, _ = orc.kl_forward(h_s, W_s, h_t, W_t, 1.4)
    dh, _ = orc.kl_backward(h_s, W_s, h_t, W_t, 1.4, grad_scale=0.5)
    rows = [0, 3, 19, 7]
    k, ls, lt, dhr = orc.kl_rows(h_s, W_s, h_t, W_t, 1.4, rows, grad_scale=0.5)
    np.testing.assert_allclose(k, kl[rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(ls, lse_s[rows], rtol=1e-13)
    np.testing.assert_allclose(lt, lse_t[rows], rtol=1e-13)
    np.testing.assert_allclose(dhr, dh[rows], rtol=1e-12, atol=1e-16)


def test_vocab_rows_match_full():
    """dW_s rows from the per-token log-sum-exps alone equal the rows of the full backward (a
    slip in the column's softmax, the 1/(tau N) or the transpose fails this), over several token
    chunks and with a global N larger than the rows passed."""
    rng = np.random.default_rng(43)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 23, 6, 8, 31)
    _, lse_s, lse_t, _ = orc.kl_forward(h_s, W_s, h_t, W_t, 0.7)
    _, dW = orc.kl_backward(h_s, W_s, h_t, W_t, 0.7, grad_scale=-1.5)
    rows = [0, 30, 5, 17, 5]
    got = orc.kl_grad_vocab_rows(h_s, W_s, h_t, W_t, 0.7, rows, lse_s, lse_t, grad_scale=-1.5, token_chunk=4)
    np.testing.assert_allclose(got, dW[rows], rtol=1e-11, atol=1e-16)
    # a token subset of a larger mean: its share of the full gradient, scaled by N_sub / N
    sub = orc.kl_grad_vocab_rows(h_s[:9], W_s, h_t[:9], W_t, 0.7, rows, lse_s[:9], lse_t[:9], grad_scale=-1.5,
                                 n_total=23)
    rest = orc.kl_grad_vocab_rows(h_s[9:], W_s, h_t[9:], W_t, 0.7, rows, lse_s[9:], lse_t[9:], grad_scale=-1.5,
                                  n_total=23)
    np.testing.assert_allclose(sub + rest, dW[rows], rtol=1e-11, atol=1e-16)


# ----------------------------------------------------------------------------- statistics

def _f64(t):
    return syn.to_f64_numpy(t)


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_gaussian_large_vocab_closed_form(tau):
    """Independent Gaussian logits with variances s_t^2, s_s^2 and a large vocabulary give
    E[KL] -> (s_t^2 + s_s^2) / (2 tau^2); with RMS-normalised hidden states and
    W ~ N(0, 0.02^2), s^2 = 0.02^2 * d, i.e. 1.2288 at tau=1 and 0.3072 at tau=2."""
    w = syn.WORKLOADS["llama1b_8b_8k"].with_sizes(N=48, V=16384, tau=tau)
    x = syn.make_inputs(w)
    kl, *_ = orc.kl_forward(_f64(x["h_s"]), _f64(x["W_s"]), _f64(x["h_t"]), _f64(x["W_t"]), tau)
    expect = (0.02 ** 2 * (w.d_s + w.d_t)) / (2 * tau * tau)
    assert abs(kl.mean() - expect) < 0.05 * expect


def test_tiny_workload_mean_kl():
    """tiny: h ~ N(0,1) unnormalised, W ~ N(0, 0.05^2): s_s^2 = 0.16, s_t^2 = 0.32 -> E[KL] ~ 0.24
    (V = 512 is small, so a 10% band)."""
    w = syn.WORKLOADS["tiny"]
    x = syn.make_inputs(w)
    _, _, _, loss = orc.kl_forward(_f64(x["h_s"]), _f64(x["W_s"]), _f64(x["h_t"]), _f64(x["W_t"]), 1.0)
    assert abs(loss - 0.24) < 0.024


def test_near_converged_workload_small_kl():
    """Near-converged student: z_s = z_t + 0.01 eps W_s^T, so KL ~ Var(d)/2 with
    Var(d) = 1e-4 * d_s * 0.02^2 -> 6.1e-5 (plus a few 1e-6 from bf16 rounding)."""
    w = syn.WORKLOADS["llama3b_nearconv"].with_sizes(N=32, V=4096)
    x = syn.make_inputs(w)
    kl, *_ = orc.kl_forward(_f64(x["h_s"]), _f64(x["W_s"]), _f64(x["h_t"]), _f64(x["W_t"]), 1.0)
    assert 3.5e-5 < kl.mean() < 1.1e-4
    assert np.all(kl >= 0)


def test_synthetic_inputs_are_seeded():
    w = syn.WORKLOADS["tiny"]
    a = syn.make_inputs(w)
    b = syn.make_inputs(w)
    for k in a:
        assert torch.equal(a[k], b[k])
        assert a[k].dtype == torch.bfloat16
    assert a["h_s"].shape == (64, 64) and a["W_t"].shape == (512, 128)


def test_rational_golden_fixture():
    import json
    import os
    import importlib.util
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("rational_case", os.path.join(here, "rational_case.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    g = json.load(open(os.path.join(here, "rational_case.json")))
    h_s, W_s, h_t, W_t = mod.inputs()
    kl, lse_s, lse_t, loss = orc.kl_forward(h_s, W_s, h_t, W_t, g["tau"])
    np.testing.assert_allclose(kl, g["kl"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse_s, g["lse_s"], rtol=1e-13)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, g["tau"], grad_scale=g["grad_scale"])
    np.testing.assert_allclose(dh, g["dh_s"], rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(dW, g["dW_s"], rtol=1e-11, atol=1e-16)
    assert all(k > 0 for k in g["kl"])


# ----------------------------------------------------------------------------- logits input

def test_logits_oracle_matches_hidden_state_oracle():
    """On logits z = h W^T the logits-input oracle gives the pinned hidden-state results, and
    its G contracts to the pinned gradients (dh_s = G W_s, dW_s = G^T h_s)."""
    rng = np.random.default_rng(43)
    h_s, W_s, h_t, W_t = _rand_problem(rng, 9, 6, 10, 37, w_std=0.5)
    kl, ls, lt, loss = orc.kl_forward(h_s, W_s, h_t, W_t, 1.3)
    dh, dW = orc.kl_backward(h_s, W_s, h_t, W_t, 1.3, grad_scale=0.7)
    k2, ls2, lt2, loss2, G = orc.kl_from_logits(h_s @ W_s.T, h_t @ W_t.T, 1.3, grad_scale=0.7)
    np.testing.assert_allclose(k2, kl, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(ls2, ls, rtol=1e-13)
    np.testing.assert_allclose(lt2, lt, rtol=1e-13)
    assert abs(loss2 - loss) < 1e-14
    np.testing.assert_allclose(G @ W_s, dh, rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(G.T @ h_s, dW, rtol=1e-11, atol=1e-16)


def test_logits_oracle_closed_forms_and_finite_differences():
    tau, gs = 0.9, 1.4
    z_s = np.array([[0.3, -1.2], [2.0, 0.5], [0.0, 0.0]])
    z_t = np.array([[1.1, 0.4], [-0.5, 0.7], [0.0, 0.0]])
    kl, _, _, loss, G = orc.kl_from_logits(z_s, z_t, tau, gs)
    for n in range(3):
        p = 1.0 / (1.0 + math.exp(-(z_t[n, 1] - z_t[n, 0]) / tau))
        q = 1.0 / (1.0 + math.exp(-(z_s[n, 1] - z_s[n, 0]) / tau))
        ref = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        assert abs(kl[n] - ref) <= 1e-12 * (1 + ref)
    assert kl[2] == 0.0  # identical rows
    eps = 1e-6
    for idx in np.ndindex(*z_s.shape):
        zp, zm = z_s.copy(), z_s.copy()
        zp[idx] += eps
        zm[idx] -= eps
        fd = gs * (orc.kl_from_logits(zp, z_t, tau)[3] - orc.kl_from_logits(zm, z_t, tau)[3]) / (2 * eps)
        assert abs(G[idx] - fd) < 1e-8
    assert np.all(np.abs(G.sum(axis=1)) < 1e-15)  # each row of G sums to zero


# ----------------------------------------------------------------------------- Stage-I ILD

def test_ild_closed_forms():
    """3-4-5 and 5-12-13 difference vectors have norms 5 and 13; zero differences add nothing."""
    T = np.zeros((2, 3, 4))
    S = np.zeros((2, 3, 4))
    S[0, 0, :2] = [3.0, 4.0]
    S[1, 2, 1:3] = [5.0, -12.0]
    T[0, 1] = S[0, 1] = 7.0  # equal rows
    norms, loss, grad = orc.ild_loss(S, T, grad_scale=2.0)
    assert norms[0, 0] == 5.0 and norms[1, 2] == 13.0 and norms[0, 1] == 0.0
    assert abs(loss - (5.0 + 13.0) / 3) < 1e-15
    np.testing.assert_allclose(grad[0, 0, :2], 2.0 * np.array([3.0, 4.0]) / (3 * 5.0))
    assert np.all(grad[0, 1] == 0.0)


def test_ild_scaling_and_finite_differences():
    rng = np.random.default_rng(47)
    S = rng.standard_normal((3, 5, 6))
    T = rng.standard_normal((3, 5, 6))
    _, loss, grad = orc.ild_loss(S, T, grad_scale=1.5)
    _, loss2, _ = orc.ild_loss(T + 2.5 * (S - T), T)
    assert abs(loss2 - 2.5 * loss) < 1e-12 * loss  # norms are 1-homogeneous
    _, loss_swapped, _ = orc.ild_loss(T, S)
    assert abs(loss_swapped - loss) < 1e-13 * loss  # symmetric in student and teacher
    eps = 1e-6
    for idx in [(0, 0, 0), (1, 3, 2), (2, 4, 5), (0, 2, 3)]:
        Sp, Sm = S.copy(), S.copy()
        Sp[idx] += eps
        Sm[idx] -= eps
        fd = 1.5 * (orc.ild_loss(Sp, T)[1] - orc.ild_loss(Sm, T)[1]) / (2 * eps)
        assert abs(grad[idx] - fd) < 1e-8


# ------------------------------------------------- the algebra the kernels use, in fp64

@pytest.mark.parametrize("shift,noise", [(0.0, 1.0), (0.0, 1e-3), (3.0, 1e-2)])
def test_online_statistics_forms_match_the_definition(shift, noise):
    """The kernels never form the softmaxes: they keep, per token, running maxima m_x, sums
    S_x = sum exp((z_x - m_x)/tau), A = sum e_t d and C = sum e_t (exp(-d) - 1 + d) with
    d = (z_t - z_s)/tau, e_t = exp((z_t - m_t)/tau), merged chunk by chunk with rescaling, and
    read off lse_x = m_x/tau + log S_x, KL = A/S_t - lse_t + lse_s, the cancellation-free
    KL = C' + log1p(u) - u and the gap lse_s - lse_t = log1p(u) (u = C' - A/S_t, C' = C/S_t).
    Here, in fp64 and independently of the oracle's code path, each form against the oracle's
    definition, including a common shift of the student logits (KL unchanged, gap moves)."""
    rng = np.random.default_rng(97)
    tau, V, chunk = 1.3, 1000, 96
    z_t = rng.standard_normal((5, V)) * 1.5
    z_s = z_t + shift + noise * rng.standard_normal((5, V))
    kl, ls, lt, _, _ = orc.kl_from_logits(z_s, z_t, tau)
    for n in range(5):
        mt = ms = -np.inf
        st = ss = a = c = 0.0
        for c0 in range(0, V, chunk):  # online fold, ragged last chunk
            zt, zs = z_t[n, c0:c0 + chunk], z_s[n, c0:c0 + chunk]
            nmt, nms = max(mt, zt.max()), max(ms, zs.max())
            wt, ws = math.exp((mt - nmt) / tau), math.exp((ms - nms) / tau)
            st, a, c, ss = st * wt, a * wt, c * wt, ss * ws
            mt, ms = nmt, nms
            et, es = np.exp((zt - mt) / tau), np.exp((zs - ms) / tau)
            d = (zt - zs) / tau
            st += et.sum()
            ss += es.sum()
            a += (et * d).sum()
            c += (et * (np.exp(-d) - 1 + d)).sum()
        lse_t, lse_s = mt / tau + math.log(st), ms / tau + math.log(ss)
        mu, cn = a / st, c / st
        u = cn - mu
        assert abs(lse_t - lt[n]) < 1e-12 * (1 + abs(lt[n]))
        assert abs(lse_s - ls[n]) < 1e-12 * (1 + abs(ls[n]))
        assert abs((mu - lse_t + lse_s) - kl[n]) < 1e-11 * (1 + abs(lse_t))
        if abs(u) < 0.5:  # the regime the kernels take this form in: no cancellation (the
            # oracle's own sum of p_t (l_t - l_s) keeps ~1e-10 of a KL this small)
            assert abs((cn + (math.log1p(u) - u)) - kl[n]) < 1e-9 * kl[n] + 1e-18
        else:  # still exact algebra, but cn and u are large next to KL here
            assert abs((cn + math.log1p(u) - u) - kl[n]) < 1e-13 * (1 + cn + abs(u))
        assert abs(math.log1p(u) - (ls[n] - lt[n])) < 1e-12 * (1 + abs(ls[n]))
