"""bench.py under several ranks runs independent replicas and reports the whole-job rate over
the slowest rank's time. These checks run the rank aggregation on CPU with a world-size-2
gloo group (no GPU, no NCCL)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    my_ms = 100.0 + 25.0 * rank  # rank 1 is the slowest
    m = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
    out[rank] = m
    out[world + rank] = bench.whole_job_rate(65536, world, 4, m)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_rate_with_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().list([0.0] * (2 * world))
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert list(out[:world]) == [125.0, 125.0]
    expect = 65536 * 2 * 4 / 0.125
    assert out[world] == pytest.approx(expect) and out[world + 1] == pytest.approx(expect)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1, torch.device("cpu")) == 12.5
    assert bench.whole_job_rate(100, 1, 10, 1000.0) == pytest.approx(1000.0)


def test_cpu_samples_stay_in_range():
    """The CPU-baseline and reference legs sample rows of the workload: never an index past
    its last token, whatever the requested sample size (the tiny workload has 64 tokens)."""
    sys.path.insert(0, ROOT)
    import bench
    from hybrid_upcycling_gb300 import synthetic as syn
    for n, c in [(64, 256), (64, 48), (8192, 256), (1, 5), (300, 300)]:
        r = bench.sample_rows(n, c)
        assert len(r) == min(n, c) and int(r.min()) >= 0 and int(r.max()) < n
        assert len(set(r.tolist())) == len(r)
    w = syn.WORKLOADS["tiny"]
    x = syn.make_inputs(w, device="cpu")
    rate, dt = bench.cpu_oracle_rate(w, x, 256)  # more than the workload's tokens
    assert rate > 0 and dt > 0
    prepared = bench.oracle_inputs(w, x, 256)
    assert prepared[0].shape == (w.N, w.d_s) and prepared[1].shape == (w.V, w.d_s)
    assert bench.cpu_oracle_rate(w, None, 256, inputs=prepared)[0] > 0
