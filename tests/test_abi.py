"""Host-side checks of the C ABI: the shared library builds and loads, exports every entry
point include/hylo_kl.h declares, sizes its workspace as documented, and rejects bad
arguments before touching the GPU (these calls never launch a kernel)."""
import ctypes
import os
import re

import pytest
import torch

from hybrid_upcycling_gb300 import build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(hylo_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert {"hylo_kl_forward", "hylo_kl_backward", "hylo_kl_workspace_bytes"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(_lib.EXPORTS) <= names


PACE = 1280  # the fused kernels' pacing counters: one 8-byte word per cluster and a switch, to 256 B
G_RING = 128 << 20  # the backward's G staging: three blocks of tokens x words, at most 128 MiB in all


def _r256(x):
    return (x + 255) // 256 * 256


def _g_ring(N, V, chunk):
    """Bytes of the G ring as documented: 3 blocks of R x bw bf16, R = token_chunk rounded up to
    256 (at most 32768, at most N rounded up), bw = 128 MiB / (6 R) rounded down to 256 words (at
    most V rounded up)."""
    c = 4096 if chunk <= 0 else min(chunk, 32768)
    R = min(_r256(c), _r256(N))
    bw = min((G_RING // (6 * R)) // 256 * 256, _r256(V))
    return 3 * R * bw * 2


def test_workspace_bytes(lib):
    """O(N) statistics for the forward, a G ring of at most 128 MiB for the backward: the size
    is bounded independently of V x token_chunk (and never N x V)."""
    N, d_s, d_t, V = 65536, 2048, 4096, 128256
    fwd = 6 * 32 * N * 4
    # 3 blocks of 4096 tokens x 5376 words of bf16 G = 126 MiB
    assert _g_ring(N, V, 4096) == 3 * 4096 * 5376 * 2 == 126 << 20
    assert _lib.hylo_kl_workspace_bytes(N, d_s, d_t, V, 4096) == max(fwd, 126 << 20) + PACE
    for n, v, chunk in ((65536, 128256, 4096), (65536, 151936, 1024), (4096, 128256, 4096), (1000, 262144, 4096),
                        (100000, 128256, 100000), (65536, 128256, 65536), (8192, 1 << 20, 8192), (300, 1000, 7),
                        (100, 513, 100000), (64, 100, 4096), (1, 3, 0)):
        ws = _lib.hylo_kl_workspace_bytes(n, d_s, d_t, v, chunk)
        assert ws == max(_r256(6 * 32 * n * 4), _r256(_g_ring(n, v, chunk))) + PACE, (n, v, chunk)
        assert ws <= max(6 * 32 * n * 4, G_RING) + PACE, (n, v, chunk, ws)
        wss = _lib.hylo_kl_workspace_bytes_split(n, d_s, d_t, v, chunk)
        assert wss == max(_r256(6 * 32 * n * 4), 2 * _r256(_g_ring(n, v, chunk))) + PACE
        assert wss <= max(6 * 32 * n * 4, 2 * G_RING) + PACE
    # at N <= 4096 tokens (one token block) the G staging is still at most 128 MiB, not N x V
    assert _lib.hylo_kl_workspace_bytes(4096, d_s, d_t, V, 4096) < 4096 * V * 2
    assert _lib.hylo_kl_workspace_bytes(8192, 64, 64, 1000, 0) == _lib.hylo_kl_workspace_bytes(8192, 64, 64, 1000, 4096)
    # invalid sizes give 0
    assert _lib.hylo_kl_workspace_bytes(0, 64, 64, 10, 4096) == 0
    assert _lib.hylo_kl_workspace_bytes(10, 60, 64, 10, 4096) == 0
    assert _lib.hylo_kl_workspace_bytes(10, 64, 64, 0, 4096) == 0


FAKE = 0x10000  # a 256-byte aligned non-null address; never dereferenced by these calls


def _fwd(lib, **kw):
    a = dict(h_s=FAKE, W_s=FAKE, h_t=FAKE, W_t=FAKE, N=16, d_s=64, d_t=128, V=100, tau=1.0, chunk=4096,
             kl=FAKE, lse_s=FAKE, lse_t=FAKE, gap=None, loss=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.hylo_kl_forward(a["h_s"], a["W_s"], a["h_t"], a["W_t"], a["N"], a["d_s"], a["d_t"], a["V"],
                               a["tau"], a["chunk"], a["kl"], a["lse_s"], a["lse_t"], a["gap"], a["loss"], a["ws"],
                               a["wsb"], a["stream"])


def _bwd(lib, **kw):
    a = dict(h_s=FAKE, W_s=FAKE, h_t=FAKE, W_t=FAKE, N=16, d_s=64, d_t=128, V=100, tau=1.0, chunk=4096,
             lse_s=FAKE, lse_t=FAKE, gap=None, gs=1.0, dh=FAKE, dW=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.hylo_kl_backward(a["h_s"], a["W_s"], a["h_t"], a["W_t"], a["N"], a["d_s"], a["d_t"], a["V"],
                                a["tau"], a["chunk"], a["lse_s"], a["lse_t"], a["gap"], a["gs"], a["dh"], a["dW"],
                                a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(h_s=None), -1), (dict(W_t=None), -1), (dict(kl=None), -1), (dict(ws=None), -1),
    (dict(N=0), -2), (dict(V=0), -2), (dict(d_s=60), -2), (dict(d_t=4), -2), (dict(d_s=70000), -2),
    (dict(h_s=FAKE + 8), -3), (dict(ws=FAKE + 16), -3),
    (dict(tau=0.0), -4), (dict(tau=-1.0), -4), (dict(tau=float("inf")), -4), (dict(tau=float("nan")), -4),
    (dict(wsb=16), -5),
])
def test_forward_rejects_bad_arguments(lib, kw, status):
    assert _fwd(lib, **kw) == status
    assert lib.hylo_kl_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(lse_s=None), -1), (dict(dW=None), -1), (dict(N=-5), -2), (dict(d_t=12), -2),
    (dict(W_s=FAKE + 4), -3), (dict(dh=FAKE + 4), -3), (dict(tau=float("nan")), -4),
    (dict(gs=float("inf")), -4), (dict(wsb=100), -5),
])
def test_backward_rejects_bad_arguments(lib, kw, status):
    assert _bwd(lib, **kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_gpu_fails_cleanly(lib):
    st = _fwd(lib)
    assert st in (-6, -8)
    assert lib.hylo_kl_last_error()


def _logits(lib, **kw):
    a = dict(zs=FAKE, zt=FAKE, N=16, V=100, ld=104, tau=1.0, gs=1.0, kl=FAKE, ls=FAKE, lt=FAKE, loss=FAKE, dz=FAKE,
             stream=None)
    a.update(kw)
    return lib.hylo_fused_kl_logits(a["zs"], a["zt"], a["N"], a["V"], a["ld"], a["tau"], a["gs"], a["kl"], a["ls"],
                                    a["lt"], a["loss"], a["dz"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(zs=None), -1), (dict(loss=None), -1), (dict(N=0), -2), (dict(V=0), -2), (dict(ld=99), -2),
    (dict(ld=100), -2), (dict(zt=FAKE + 2), -3), (dict(dz=FAKE + 8), -3), (dict(tau=0.0), -4),
    (dict(gs=float("nan")), -4),
])
def test_logits_rejects_bad_arguments(lib, kw, status):
    assert _logits(lib, **kw) == status
    assert lib.hylo_kl_last_error()


def _ild(lib, **kw):
    a = dict(S=FAKE, T=FAKE, P=4, N=16, d=64, gs=1.0, norms=FAKE, loss=FAKE, dS=FAKE, stream=None)
    a.update(kw)
    return lib.hylo_ild_loss(a["S"], a["T"], a["P"], a["N"], a["d"], a["gs"], a["norms"], a["loss"], a["dS"],
                             a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(S=None), -1), (dict(norms=None), -1), (dict(P=0), -2), (dict(N=-1), -2), (dict(d=4), -2),
    (dict(d=68), -2), (dict(d=65544), -2), (dict(P=1 << 30, N=1 << 30), -2), (dict(T=FAKE + 4), -3),
    (dict(dS=FAKE + 2), -3), (dict(gs=float("inf")), -4),
])
def test_ild_rejects_bad_arguments(lib, kw, status):
    assert _ild(lib, **kw) == status
    assert lib.hylo_kl_last_error()


def test_split_workspace_and_rejection(lib):
    N, d_s, d_t, V = 8192, 2048, 4096, 128256
    one = _lib.hylo_kl_workspace_bytes(N, d_s, d_t, V, 4096)
    two = _lib.hylo_kl_workspace_bytes_split(N, d_s, d_t, V, 4096)
    assert one == (126 << 20) + PACE and two == (252 << 20) + PACE
    a = dict(h_s=FAKE, W_s=FAKE, h_t=FAKE, W_t=FAKE, N=16, d_s=64, d_t=128, V=100, tau=1.0, chunk=4096,
             lse_s=FAKE, lse_t=FAKE, gap=None, gs=1.0, dh=FAKE, dW=FAKE, ws=FAKE, stream=None)
    small = _lib.hylo_kl_workspace_bytes(4096, 64, 128, 100000, 4096)
    st = lib.hylo_kl_backward_split(a["h_s"], a["W_s"], a["h_t"], a["W_t"], 4096, 64, 128, 100000, 1.0, 4096,
                                    a["lse_s"], a["lse_t"], None, 1.0, a["dh"], a["dW"], a["ws"], small, None)
    assert st == -5  # the single-G workspace is too small for the split backward
    assert _lib.hylo_kl_workspace_bytes_split(0, 64, 64, 10, 4096) == 0
