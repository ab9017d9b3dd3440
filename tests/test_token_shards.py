"""Token sharding of the loss: R shards of the N tokens, each run with grad_scale = N_r / N,
reproduce the unsharded results once the per-shard dW_s are summed, the dh_s rows are
concatenated and the shard losses are combined as sum_r N_r loss_r / N.

This is the data-parallel split of Stage-II distillation (Long-Context Aware Upcycling digest,
section Experiments: FSDP training): every token's KL and dh_s row depend on its own row alone,
the mean's 1/N is global, and dW_s = G^T h_s is a sum over tokens. Checked on the oracle
(sequentially and with a world-size-2 gloo all-reduce on CPU), through the package's
orchestration (hybrid_upcycling_gb300.shard) on two gloo ranks with the oracle as the shard
compute, and through the C ABI on one GPU (sequential shards; the orchestration on one rank).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import kl_oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem(seed=5, N=23, d_s=6, d_t=10, V=31):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, d_s)), rng.standard_normal((V, d_s)) * 0.4,
            rng.standard_normal((N, d_t)), rng.standard_normal((V, d_t)) * 0.4)


def _bounds(N, R):
    cuts = [0, 7, 8, N] if R == 3 else [round(N * r / R) for r in range(R + 1)]
    return list(zip(cuts[:-1], cuts[1:]))


def _shard(h_s, W_s, h_t, W_t, lo, hi, N, tau):
    kl, _, _, loss = orc.kl_forward(h_s[lo:hi], W_s, h_t[lo:hi], W_t, tau)
    dh, dW = orc.kl_backward(h_s[lo:hi], W_s, h_t[lo:hi], W_t, tau, grad_scale=(hi - lo) / N)
    return kl, loss, dh, dW


@pytest.mark.parametrize("R", [2, 3])
def test_oracle_sequential_shards(R):
    h_s, W_s, h_t, W_t = _problem()
    N, tau = h_s.shape[0], 1.3
    kl0, _, _, loss0 = orc.kl_forward(h_s, W_s, h_t, W_t, tau)
    dh0, dW0 = orc.kl_backward(h_s, W_s, h_t, W_t, tau)
    parts = [_shard(h_s, W_s, h_t, W_t, lo, hi, N, tau) + (hi - lo,) for lo, hi in _bounds(N, R)]
    np.testing.assert_allclose(np.concatenate([p[0] for p in parts]), kl0, rtol=1e-13, atol=1e-15)
    assert abs(sum(p[4] * p[1] for p in parts) / N - loss0) <= 1e-13 * loss0
    np.testing.assert_allclose(np.concatenate([p[2] for p in parts]), dh0, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(sum(p[3] for p in parts), dW0, rtol=1e-12, atol=1e-16)
    # a shard run with grad_scale 1 (its own mean) differs by exactly N / N_r
    lo, hi = _bounds(N, R)[0]
    _, dW_own = orc.kl_backward(h_s[lo:hi], W_s, h_t[lo:hi], W_t, tau)
    np.testing.assert_allclose(dW_own * (hi - lo) / N, parts[0][3], rtol=1e-12, atol=1e-16)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    h_s, W_s, h_t, W_t = _problem()
    N, tau = h_s.shape[0], 0.8
    lo, hi = _bounds(N, world)[rank]
    kl, loss, dh, dW = _shard(h_s, W_s, h_t, W_t, lo, hi, N, tau)
    sums = torch.tensor([loss * (hi - lo)], dtype=torch.float64)
    dW_t = torch.from_numpy(dW)
    dist.all_reduce(sums)
    dist.all_reduce(dW_t)
    gathered = [None] * world
    dist.all_gather_object(gathered, dh)
    if rank == 0:
        kl0, _, _, loss0 = orc.kl_forward(h_s, W_s, h_t, W_t, tau)
        dh0, dW0 = orc.kl_backward(h_s, W_s, h_t, W_t, tau)
        out[0] = abs(sums.item() / N - loss0) / loss0
        out[1] = float(np.max(np.abs(dW_t.numpy() - dW0)) / np.max(np.abs(dW0)))
        out[2] = float(np.max(np.abs(np.concatenate(gathered) - dh0)) / np.max(np.abs(dh0)))
    dist.barrier()
    dist.destroy_process_group()


def test_gloo_two_rank_all_reduce_of_shards():
    out = mp.get_context("spawn").Manager().list([1.0, 1.0, 1.0])
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    assert max(out) <= 1e-12, list(out)


def _oracle_compute(h_s, W_s, h_t, W_t, tau, token_chunk, grad_scale):
    """The per-shard computation of hybrid_upcycling_gb300.shard, done by the fp64 oracle (test
    infrastructure: lets the orchestration run on CPU ranks)."""
    a = [t.numpy() for t in (h_s, W_s, h_t, W_t)]
    kl, _, _, loss = orc.kl_forward(*a, tau, token_chunk)
    dh, dW = orc.kl_backward(*a, tau, token_chunk, grad_scale=grad_scale)
    return torch.tensor([loss], dtype=torch.float64), torch.from_numpy(kl), torch.from_numpy(dh), torch.from_numpy(dW)


def _sharded_worker(rank, world, port, mode, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from hybrid_upcycling_gb300.shard import kl_fwd_bwd_sharded, vocab_shard
    h_s, W_s, h_t, W_t = _problem(seed=9, N=23, d_s=6, d_t=10, V=31)
    cuts = [0, 9, 23]  # uneven shards: 9 and 14 tokens
    lo, hi = cuts[rank], cuts[rank + 1]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    res = kl_fwd_bwd_sharded(t(h_s[lo:hi]), t(W_s), t(h_t[lo:hi]), t(W_t), 0.9, token_chunk=4, grad_reduce=mode,
                             upstream=0.7, compute=_oracle_compute)
    parts = [None] * world
    dist.all_gather_object(parts, (res.loss.item(), res.kl.numpy(), res.dh_s.numpy(), res.dW_s.numpy(),
                                   res.vocab_rows, res.n_total))
    if rank == 0:
        kl0, _, _, loss0 = orc.kl_forward(h_s, W_s, h_t, W_t, 0.9)
        dh0, dW0 = orc.kl_backward(h_s, W_s, h_t, W_t, 0.9, grad_scale=0.7)
        errs = [max(abs(p[0] - loss0) for p in parts) / loss0,
                float(np.max(np.abs(np.concatenate([p[1] for p in parts]) - kl0))),
                float(np.max(np.abs(np.concatenate([p[2] for p in parts]) - dh0)) / np.max(np.abs(dh0)))]
        if mode == "all_reduce":
            errs.append(max(float(np.max(np.abs(p[3] - dW0))) for p in parts) / np.max(np.abs(dW0)))
        else:  # each rank holds its vocabulary shard's rows
            rows = [p[4] for p in parts]
            assert rows == [vocab_shard(31, r, world) for r in range(world)], rows
            errs.append(max(float(np.max(np.abs(p[3] - dW0[p[4][0]:p[4][1]])))
                            for p in parts) / np.max(np.abs(dW0)))
            assert sum(r[1] - r[0] for r in rows) == 31
        assert all(p[5] == 23 for p in parts)
        for i, e in enumerate(errs):
            out[i] = e
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["all_reduce", "reduce_scatter"])
def test_sharded_orchestration_two_gloo_ranks(mode):
    """The package's token-sharded step (hybrid_upcycling_gb300.shard), its per-shard compute done
    by the oracle: two ranks with 9 and 14 tokens reproduce the unsharded loss, per-token KL, dh_s
    rows and dW_s (summed, or scattered by vocabulary rows: 31 rows over 2 ranks, padded)."""
    out = mp.get_context("spawn").Manager().list([1.0] * 4)
    mp.spawn(_sharded_worker, args=(2, _free_port(), mode, out), nprocs=2, join=True)
    assert max(out) <= 1e-12, list(out)


def test_vocab_shards_cover_the_vocabulary():
    sys.path.insert(0, ROOT)
    from hybrid_upcycling_gb300.shard import vocab_shard
    for V, world in [(31, 2), (128256, 8), (7, 8), (151936, 3)]:
        rows = [vocab_shard(V, r, world) for r in range(world)]
        assert rows[0][0] == 0 and rows[-1][1] == V
        assert all(a[1] == b[0] for a, b in zip(rows[:-1], rows[1:]))


@pytest.mark.gpu
def test_gpu_sharded_step_on_one_rank_matches_the_plain_call():
    """kl_fwd_bwd_sharded with the library compute on a one-rank NCCL group: the collectives are
    identities, so the results equal the plain C-ABI calls (same kernels, same inputs)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hybrid_upcycling_gb300 import _lib, build, synthetic as syn
    from hybrid_upcycling_gb300.shard import kl_fwd_bwd_sharded
    build.build()
    w = syn.WORKLOADS["llama1b_8b_8k"].with_sizes(N=700, V=5000)
    x = syn.make_inputs(w, device="cuda")
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        res = kl_fwd_bwd_sharded(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 512, upstream=0.5)
        _lib.hylo_kl_sync_status()
    finally:
        dist.destroy_process_group()
    N, f = w.N, dict(dtype=torch.float32, device="cuda")
    ws = torch.empty(_lib.hylo_kl_workspace_bytes(N, w.d_s, w.d_t, w.V, 512), dtype=torch.uint8, device="cuda")
    kl, ls, lt, gap = (torch.empty(N, **f) for _ in range(4))
    loss = torch.empty(1, **f)
    dh, dW = torch.empty(N, w.d_s, **f), torch.empty(w.V, w.d_s, **f)
    _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 512, kl, ls, lt, loss, ws, lse_gap=gap)
    _lib.hylo_kl_backward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, 512, ls, lt, 0.5, dh, dW, ws, lse_gap=gap)
    _lib.hylo_kl_sync_status()
    assert res.n_total == N and res.vocab_rows == (0, w.V)
    assert abs(res.loss.item() - loss.item()) <= 1e-6 * loss.item()
    assert torch.equal(res.kl, kl) and torch.equal(res.dh_s, dh) and torch.equal(res.dW_s, dW)


@pytest.mark.gpu
def test_gpu_sequential_shards_through_the_c_abi():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hybrid_upcycling_gb300 import _lib, build, synthetic as syn
    build.build()
    w = syn.WORKLOADS["llama1b_8b_8k"].with_sizes(N=1500, V=9000)
    x = syn.make_inputs(w, device="cuda")
    N, f = w.N, dict(dtype=torch.float32, device="cuda")

    def run(lo, hi, gs):
        n = hi - lo
        hs, ht = x["h_s"][lo:hi], x["h_t"][lo:hi]
        ws = torch.empty(_lib.hylo_kl_workspace_bytes(n, w.d_s, w.d_t, w.V, 512), dtype=torch.uint8, device="cuda")
        kl, ls, lt, gap = (torch.empty(n, **f) for _ in range(4))
        loss = torch.empty(1, **f)
        dh, dW = torch.empty(n, w.d_s, **f), torch.empty(w.V, w.d_s, **f)
        _lib.hylo_kl_forward(hs, x["W_s"], ht, x["W_t"], w.tau, 512, kl, ls, lt, loss, ws, lse_gap=gap)
        _lib.hylo_kl_backward(hs, x["W_s"], ht, x["W_t"], w.tau, 512, ls, lt, gs, dh, dW, ws, lse_gap=gap)
        _lib.hylo_kl_sync_status()
        return kl, loss, dh, dW

    kl0, loss0, dh0, dW0 = run(0, N, 1.0)
    cuts = [0, 257, 1000, N]  # ragged shards: 257 = one 256-token pair tile plus one token
    parts = [run(lo, hi, (hi - lo) / N) + (hi - lo,) for lo, hi in zip(cuts[:-1], cuts[1:])]
    kl = torch.cat([p[0] for p in parts])
    # per-token results depend on the row alone up to the fp32 order of the vocabulary segments
    assert torch.allclose(kl, kl0, rtol=2e-5, atol=1e-6)
    loss = sum(p[4] * p[1].double().item() for p in parts) / N
    assert abs(loss - loss0.item()) <= 1e-5 * loss0.item()
    dh = torch.cat([p[2] for p in parts])
    dW = sum(p[3].double() for p in parts)
    rel = lambda a, b: (torch.linalg.norm(a.double() - b.double()) / torch.linalg.norm(b.double())).item()
    assert rel(dh, dh0) <= 2e-4, rel(dh, dh0)
    assert rel(dW, dW0) <= 2e-4, rel(dW, dW0)
