"""Benchmark of the fused hidden-state KL loss (fwd + bwd) on GB300.

One step = hylo_kl_forward + hylo_kl_backward over one synthetic batch of the workload
(default: the 64K-token Stage-II shape, N=65536, d_s=2048, d_t=4096, V=128256, tau=1,
token_chunk=4096). Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) the default `--mode dp` is the data-parallel step of Stage-II training:
every rank holds its own sequence of the workload's N tokens (one global batch of N x ranks
tokens) and the full LM heads, runs the forward + backward through the C ABI with
grad_scale = N / (N x ranks), and the ranks exchange the loss sum and dW_s with one NCCL
all-reduce each (hybrid_upcycling_gb300.shard; weak scaling, the collectives inside the timed
region). `--mode replicas` runs independent replicas instead (no exchange). `--impl reference`
times the fp64 CPU oracle on the host cores on a bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hybrid_upcycling_gb300 import synthetic as syn  # noqa: E402

METRIC = "fused KL fwd+bwd tokens/s and TFLOP/s as % of GB300 dense bf16 peak"
# NVIDIA's dense bf16 tensor figure for one GB300 GPU: 36 PFLOP/s with 2:4 sparsity per 8 GPUs,
# halved for dense math, divided by 8.
NOMINAL_BF16_TFLOPS = 2250.0
METRIC_LOGITS = "fused KL on logits fwd+bwd tokens/s (HBM-bound)"
METRIC_ILD = "Stage-I ILD loss fwd+bwd tokens/s (HBM-bound)"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest value over all ranks (rank 0's timing is the slowest rank's)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, steps: int, max_ms: float) -> float:
    """Units processed by all ranks per second of the slowest rank's timed region."""
    return units_per_rank * world * steps / (max_ms / 1e3)


def pipelined_e2e(host_in, slots_in, slots_out, copy_out, call, steps, stream, dev):
    """End-to-end time (ms) of `steps` steps through host memory: every step copies its inputs
    from the pinned host tensors `host_in` into a device slot, runs `call(inputs, outputs)` on
    `stream` and copies the `copy_out` outputs back to pinned host memory. Two slots of device
    inputs and outputs: step k+1's inputs and step k-1's results move on their own copy streams
    while step k computes."""
    out_host = {k: torch.empty(slots_out[0][k].shape, dtype=slots_out[0][k].dtype, pin_memory=True)
                for k in copy_out}
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    with torch.cuda.stream(cin):  # warm the copy path once
        for k in host_in:
            slots_in[0][k].copy_(host_in[k], non_blocking=True)
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=False)
    ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    for i in range(steps):
        s = i % 2
        with torch.cuda.stream(cin):
            if i >= 2:
                cin.wait_event(ev_comp[s])  # step i-2 has finished reading slot s
            for k in host_in:
                slots_in[s][k].copy_(host_in[k], non_blocking=True)
            ev_in[s].record(cin)
        stream.wait_event(ev_in[s])
        if i >= 2:
            stream.wait_event(ev_out[s])  # step i-2's results have left slot s
        with torch.cuda.stream(stream):
            call(slots_in[s], slots_out[s])
            ev_comp[s].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_comp[s])
            for k in copy_out:
                out_host[k].copy_(slots_out[s][k], non_blocking=True)
            ev_out[s].record(cout)
    e1.record(cout)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    d2h = sum(v.numel() * v.element_size() for v in out_host.values())
    return ms, d2h


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# Per path: the committed DRAM-traffic record of its dominant kernel (profiles/) and the
# sources of that kernel's translation unit; a record stays valid while they are unchanged.
TRAFFIC_RECORDS = {
    "hidden": ("bwd_pipe_traffic.txt", ("kl_bwd_pipe.cu", "kl_stats.cuh", "sm103_ptx.cuh", "hylo_internal.h")),
    "hidden_fwd": ("fused_fwd_traffic.txt", ("kl_fused.cu", "kl_stats.cuh", "sm103_ptx.cuh", "hylo_internal.h")),
    "logits": ("kl_logits_traffic.txt", ("kl_logits.cu", "kl_stats.cuh", "sm103_ptx.cuh", "hylo_internal.h")),
    "ild": ("ild_traffic.txt", ("ild.cu", "sm103_ptx.cuh", "hylo_internal.h")),
}


def kernel_source_hash(path: str = "hidden") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hybrid_upcycling_gb300", "csrc")
    for fn in TRAFFIC_RECORDS[path][1]:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, path: str = "hidden"):
    """DRAM bytes per launch of the path's dominant kernel from the committed ncu summary, if
    it was taken from the current kernel sources and for this workload (else None)."""
    p = os.path.join(ROOT, "profiles", TRAFFIC_RECORDS[path][0])
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_hash") != kernel_source_hash(path) or kv.get("workload") != workload:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let nvidia-smi start sampling before the timed region begins
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id(local: int) -> str:
    """nvidia-smi identifier of this process's GPU (its UUID when torch exposes it)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


def make_buffers(w, x, dev, split=False):
    from hybrid_upcycling_gb300 import _lib
    f = dict(dtype=torch.float32, device=dev)
    wsb = (_lib.hylo_kl_workspace_bytes_split if split else _lib.hylo_kl_workspace_bytes)(w.N, w.d_s, w.d_t, w.V,
                                                                                          w.token_chunk)
    b = {
        "split": split,
        "ws": torch.empty(wsb, dtype=torch.uint8, device=dev),
        "kl": torch.empty(w.N, **f), "lse_s": torch.empty(w.N, **f), "lse_t": torch.empty(w.N, **f),
        "gap": torch.empty(w.N, **f),
        "loss": torch.empty(1, **f), "dh": torch.empty(w.N, w.d_s, **f), "dW": torch.empty(w.V, w.d_s, **f),
    }
    return b


def step(w, x, b, stream, ev=None):
    from hybrid_upcycling_gb300 import _lib
    if ev is not None:
        ev[0].record(stream)
    _lib.hylo_kl_forward(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, w.token_chunk, b["kl"], b["lse_s"],
                         b["lse_t"], b["loss"], b["ws"], stream=stream, lse_gap=b["gap"])
    if ev is not None:
        ev[1].record(stream)
    bwd = _lib.hylo_kl_backward_split if b["split"] else _lib.hylo_kl_backward
    bwd(x["h_s"], x["W_s"], x["h_t"], x["W_t"], w.tau, w.token_chunk, b["lse_s"], b["lse_t"], 1.0, b["dh"], b["dW"],
        b["ws"], stream=stream, lse_gap=b["gap"])
    if ev is not None:
        ev[2].record(stream)


def launches_per_step(w, split: bool = False) -> int:
    # fused forward + combine + mean, then the one pipelined backward launch
    return 4


def time_repeated(fn, min_s: float = 10.0, max_calls: int = 10000):
    """Calls fn() until at least min_s seconds have passed; returns (calls, seconds)."""
    calls, t0 = 0, time.perf_counter()
    while True:
        fn()
        calls += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or calls >= max_calls:
            return calls, dt


def sample_rows(n_rows: int, count: int) -> torch.Tensor:
    """min(count, n_rows) row indices spread evenly over [0, n_rows), all in range."""
    count = max(1, min(count, n_rows))
    return torch.arange(count) * (n_rows // count)


def oracle_inputs(w, x, sample_tokens: int):
    """The oracle's fp64 host copies of `sample_tokens` rows of h (at most all of them) and of
    the full LM heads, widened once outside any timed region."""
    rows = sample_rows(w.N, sample_tokens)
    widen = lambda t: t.double().cpu().numpy()
    return (widen(x["h_s"][rows.to(x["h_s"].device)]), widen(x["W_s"]),
            widen(x["h_t"][rows.to(x["h_t"].device)]), widen(x["W_t"]))


def cpu_oracle_rate(w, x, sample_tokens: int, repeats: int = 1, inputs=None):
    """Times the fp64 oracle (forward + backward, as it stands) on `sample_tokens` tokens of the
    workload (at most all of them) with the full vocabulary and hidden sizes; returns
    (tokens/s, seconds). `inputs` (from oracle_inputs) skips re-widening the operands."""
    from oracle import kl_oracle as orc
    hs, Ws, ht, Wt = inputs if inputs is not None else oracle_inputs(w, x, sample_tokens)
    sample_tokens = hs.shape[0]
    t0 = time.perf_counter()
    for _ in range(repeats):
        orc.kl_forward(hs, Ws, ht, Wt, w.tau, w.token_chunk)
        orc.kl_backward(hs, Ws, ht, Wt, w.tau, w.token_chunk)
    dt = time.perf_counter() - t0
    return sample_tokens * repeats / dt, dt


def run_reference(args, w, rank, world):
    """Reference arm: the fp64 CPU oracle on the host cores (rank 0 only), on the same path,
    workload and metric as our arm, each step a sample of `--ref-tokens` tokens."""
    if rank != 0:
        return
    from oracle import kl_oracle as orc
    torch.manual_seed(0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    tokens = min(args.ref_tokens, w.N)
    if args.path == "hidden":
        x = syn.make_inputs(w, device=dev)
        prepared = oracle_inputs(w, x, tokens)
        del x
        one = lambda: cpu_oracle_rate(w, None, tokens, inputs=prepared)[1]
        metric, config = METRIC, config_dict(w)
        sample = f"{tokens} tokens of {w.name} per step (full V={w.V}, d_s={w.d_s}, d_t={w.d_t}), fp64 numpy"
    elif args.path == "logits":
        z = syn.make_logits(w, device=dev)
        rows = sample_rows(w.N, tokens)
        zs_h = z["z_s"][rows.to(z["z_s"].device)].double().cpu().numpy()
        zt_h = z["z_t"][rows.to(z["z_t"].device)].double().cpu().numpy()
        del z

        def one():
            t0 = time.perf_counter()
            orc.kl_from_logits(zs_h, zt_h, w.tau)
            return time.perf_counter() - t0
        metric, config = METRIC_LOGITS, config_logits(w)
        sample = f"{tokens} rows of {w.name} logits per step (V={w.V}), fp64 numpy"
    else:
        S, T = ild_states(dev)
        Sh, Th = S[:, :tokens].double().cpu().numpy(), T[:, :tokens].double().cpu().numpy()
        del S, T

        def one():
            t0 = time.perf_counter()
            orc.ild_loss(Sh, Th)
            return time.perf_counter() - t0
        metric, config = METRIC_ILD, config_ild()
        sample = f"{tokens} tokens x {ILD_SHAPE[0]} entries x d={ILD_SHAPE[2]} per step, fp64 numpy"
    for _ in range(args.warmup):
        one()
    times = [one() for _ in range(args.steps)]
    tot = sum(times)
    value = tokens * args.steps / tot
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


ILD_SHAPE = (32, 8192, 2048)  # 16 layers x {layer output, token-mixer output}, 4 x 2K tokens, d = 2048


def ild_states(dev):
    """Seeded Stage-I states: teacher N(0, 1), student = teacher + 0.05 N(0, 1), both bf16."""
    P, N, d = ILD_SHAPE
    g = torch.Generator(device=dev)
    g.manual_seed(1010)
    T = torch.randn(P, N, d, generator=g, device=dev)
    S = (T + 0.05 * torch.randn(P, N, d, generator=g, device=dev)).to(torch.bfloat16)
    return S, T.to(torch.bfloat16)


def config_logits(w):
    return {"workload": w.name + "_logits", "N": w.N, "V": w.V, "tau": w.tau,
            "l2": f"inputs larger than L2 ({4.0 * w.N * w.V / 1e9:.2f} GB of bf16 logits per step; no flush)"}


def config_ild():
    P, N, d = ILD_SHAPE
    return {"workload": "stage1_ild_1b", "P": P, "N": N, "d": d,
            "l2": f"inputs larger than L2 ({4.0 * P * N * d / 1e9:.2f} GB per step; no flush)"}


def config_dict(w):
    in_bytes = 2 * (w.N * (w.d_s + w.d_t) + w.V * (w.d_s + w.d_t))
    return {"workload": w.name, "N": w.N, "d_s": w.d_s, "d_t": w.d_t, "V": w.V, "tau": w.tau,
            "token_chunk": w.token_chunk,
            "l2": f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB of bf16 inputs per step; no flush)"}


def run_logits(args, w, rank, world, local):
    """`--path logits`: hylo_fused_kl_logits (statistics + bf16 gradient) on precomputed logits
    of the workload's shape; one step = one call over all N rows."""
    from hybrid_upcycling_gb300 import _lib, build
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    _lib.load()
    z = syn.make_logits(w, device=dev)
    f = dict(dtype=torch.float32, device=dev)
    kl, ls, lt, loss = torch.empty(w.N, **f), torch.empty(w.N, **f), torch.empty(w.N, **f), torch.empty(1, **f)
    dz = torch.empty(w.N, w.V, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(zz):
        _lib.hylo_fused_kl_logits(zz["z_s"], zz["z_t"], w.tau, 1.0, kl, ls, lt, loss, dz, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(z)
    _lib.hylo_kl_sync_status(stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(local)) as clk:
        with torch.cuda.stream(stream):
            for e in evs:
                e[0].record(stream)
                step(z)
                e[1].record(stream)
        torch.cuda.synchronize()
    _lib.hylo_kl_sync_status(stream)
    per = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(evs[0][0].elapsed_time(evs[-1][1]), world, dev)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alg_bytes = 6.0 * w.N * w.V  # read z_s, z_t (bf16) once, write dz_s (bf16) once
    achieved = alg_bytes / (float(np.mean(per)) / 1e3) / 1e9
    e2e = None
    if not args.no_e2e:
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in z.items()}
        for k in z:
            host[k].copy_(z[k])
        slots_in = [{k: torch.empty_like(v) for k, v in z.items()} for _ in range(2)]
        slots_out = [{"kl": torch.empty_like(kl), "lse_s": torch.empty_like(ls), "lse_t": torch.empty_like(lt),
                      "loss": torch.empty_like(loss), "dz": torch.empty_like(dz)} for _ in range(2)]
        n_e2e = max(2, min(args.steps, 5))
        ms, d2h = pipelined_e2e(
            host, slots_in, slots_out, ("loss", "dz"),
            lambda xi, xo: _lib.hylo_fused_kl_logits(xi["z_s"], xi["z_t"], w.tau, 1.0, xo["kl"], xo["lse_s"],
                                                     xo["lse_t"], xo["loss"], xo["dz"], stream=stream),
            n_e2e, stream, dev)
        _lib.hylo_kl_sync_status(stream)
        ms = max_over_ranks(ms, world, dev)
        e2e = {"value": whole_job_rate(w.N, world, n_e2e, ms), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "api": "hylo_fused_kl_logits (C ABI) with pinned-host logits and gradient, "
                      "copies double-buffered on their own streams"}
        del host, slots_in, slots_out
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import kl_oracle as orc
        rows = sample_rows(w.N, args.cpu_tokens)
        zs_h = z["z_s"][rows.to(dev)].double().cpu().numpy()
        zt_h = z["z_t"][rows.to(dev)].double().cpu().numpy()
        calls, dt = time_repeated(lambda: orc.kl_from_logits(zs_h, zt_h, w.tau))
        cpu = {"value": calls * len(rows) / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle",
               "sample": f"{calls} x {len(rows)} rows of {w.name} logits (V={w.V}), fp64 numpy, {dt:.1f} s"}
    if rank == 0:
        line = {
            "metric": METRIC_LOGITS, "value": whole_job_rate(w.N, world, args.steps, total_ms), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_logits(w),
            "roofline": {"kernel": "kl_logits_kernel (+mean)", "bound": "hbm", "achieved": achieved, "peak": hbm,
                         "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": recorded_traffic(config_logits(w)["workload"], "logits"),
                         "peak_kind": f"hbm_gbs ({src})", "bytes_per_launch": alg_bytes},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)


def run_ild(args, rank, world, local):
    """`--path ild`: hylo_ild_loss on the Stage-I shape of the 1B hybrid (16 layers x {layer
    output, token-mixer output} = 32 entries, 8192 tokens = 4 x 2K sequences, d = 2048)."""
    from hybrid_upcycling_gb300 import _lib, build
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    _lib.load()
    P, N, d = ILD_SHAPE
    S, T = ild_states(dev)
    norms = torch.empty(P * N, device=dev)
    loss = torch.empty(1, device=dev)
    dS = torch.empty_like(S)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            _lib.hylo_ild_loss(S, T, 1.0, norms, loss, dS, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(local)) as clk:
        with torch.cuda.stream(stream):
            for e in evs:
                e[0].record(stream)
                _lib.hylo_ild_loss(S, T, 1.0, norms, loss, dS, stream=stream)
                e[1].record(stream)
        torch.cuda.synchronize()
    _lib.hylo_kl_sync_status(stream)
    per = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(evs[0][0].elapsed_time(evs[-1][1]), world, dev)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alg = 6.0 * P * N * d
    achieved = alg / (float(np.mean(per)) / 1e3) / 1e9
    e2e = None
    if not args.no_e2e:
        host_in = {"S": torch.empty(S.shape, dtype=S.dtype, pin_memory=True),
                   "T": torch.empty(T.shape, dtype=T.dtype, pin_memory=True)}
        host_in["S"].copy_(S)
        host_in["T"].copy_(T)
        slots_in = [{"S": torch.empty_like(S), "T": torch.empty_like(T)} for _ in range(2)]
        slots_out = [{"norms": torch.empty_like(norms), "loss": torch.empty_like(loss), "dS": torch.empty_like(dS)}
                     for _ in range(2)]
        n_e2e = 5
        ms, d2h = pipelined_e2e(host_in, slots_in, slots_out, ("loss", "dS"),
                                lambda xi, xo: _lib.hylo_ild_loss(xi["S"], xi["T"], 1.0, xo["norms"], xo["loss"],
                                                                  xo["dS"], stream=stream),
                                n_e2e, stream, dev)
        _lib.hylo_kl_sync_status(stream)
        ms = max_over_ranks(ms, world, dev)
        e2e = {"value": whole_job_rate(N, world, n_e2e, ms), "unit": "tokens/s",
               "h2d_bytes_per_step": 2 * S.numel() * S.element_size(), "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "api": "hylo_ild_loss (C ABI) with pinned-host states, gradient and loss, "
                      "copies double-buffered on their own streams"}
        del host_in, slots_in, slots_out
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import kl_oracle as orc
        Sh, Th = S[:, :256].double().cpu().numpy(), T[:, :256].double().cpu().numpy()
        calls, dt = time_repeated(lambda: orc.ild_loss(Sh, Th))
        cpu = {"value": 256 * calls / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{calls} x 256 tokens x {P} entries x d={d}, fp64 numpy, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC_ILD, "value": whole_job_rate(N, world, args.steps, total_ms), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_ild(),
            "roofline": {"kernel": "ild_reg_kernel (+sum)", "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": recorded_traffic(config_ild()["workload"], "ild"),
                         "peak_kind": f"hbm_gbs ({src})", "bytes_per_launch": alg},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clk.summary(),
        }), flush=True)


def run_dp(args, w, rank, world, local):
    """`--mode dp` under torchrun: one data-parallel step per iteration (see the module docstring)."""
    from hybrid_upcycling_gb300 import _lib, build
    from hybrid_upcycling_gb300.shard import LibraryCompute, kl_fwd_bwd_sharded
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    torch.distributed.barrier()
    _lib.load()
    heads = syn.make_inputs(w, device=dev)  # the same LM heads on every rank (same seed)
    mine = syn.make_inputs(w, device=dev, seed=w.seed + 7919 * rank) if rank else heads
    x = {"h_s": mine["h_s"], "h_t": mine["h_t"], "W_s": heads["W_s"], "W_t": heads["W_t"]}
    del mine
    stream = torch.cuda.Stream(device=dev)
    comp = LibraryCompute(timing=True)

    def step(xx):
        return kl_fwd_bwd_sharded(xx["h_s"], xx["W_s"], xx["h_t"], xx["W_t"], w.tau, w.token_chunk, compute=comp,
                                  n_total=w.N * world)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(x)
    _lib.hylo_kl_sync_status(stream)
    comp.marks.clear()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(local)) as clk:
        with torch.cuda.stream(stream):
            for e in evs:
                e[0].record(stream)
                res = step(x)
                e[1].record(stream)
        torch.cuda.synchronize()
    torch.distributed.barrier()
    _lib.hylo_kl_sync_status(stream)
    total_ms = max_over_ranks(evs[0][0].elapsed_time(evs[-1][1]), world, dev)
    tokens_per_s = whole_job_rate(w.N, world, args.steps, total_ms)
    tflops = w.flops_exec() * world * args.steps / (total_ms / 1e3) / 1e12
    marks = list(comp.marks)
    comp.timing = False
    fwd_avg = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b, _ in marks])), world, dev)
    bwd_avg = max_over_ranks(float(np.mean([b.elapsed_time(c) for _, b, c in marks])), world, dev)
    e2e = None
    if not args.no_e2e:
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in x.items() if k.startswith("h")}
        for k in host:
            host[k].copy_(x[k])
        slots_in = [{k: torch.empty_like(x[k]) for k in host} for _ in range(2)]
        slots_out = [{"loss": torch.empty(1, dtype=torch.float64, device=dev),
                      "kl": torch.empty(w.N, device=dev), "dh": torch.empty(w.N, w.d_s, device=dev),
                      "dW": torch.empty(w.V, w.d_s, device=dev)} for _ in range(2)]

        def call(xi, xo):  # the heads stay resident; each step's tokens come from host memory
            r = step({"h_s": xi["h_s"], "h_t": xi["h_t"], "W_s": x["W_s"], "W_t": x["W_t"]})
            xo["loss"].copy_(r.loss)
            xo["kl"].copy_(r.kl)
            xo["dh"].copy_(r.dh_s)
            xo["dW"].copy_(r.dW_s)

        n_e2e = max(2, min(args.steps, 10))
        torch.distributed.barrier()
        ms, d2h = pipelined_e2e(host, slots_in, slots_out, ("loss", "kl", "dh", "dW"), call, n_e2e, stream, dev)
        torch.distributed.barrier()
        ms = max_over_ranks(ms, world, dev)
        e2e = {"value": whole_job_rate(w.N, world, n_e2e, ms), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "api": "hybrid_upcycling_gb300.shard.kl_fwd_bwd_sharded (C ABI per rank, NCCL all-reduce of "
                      "loss and dW_s) with pinned-host token inputs and outputs"}
        del host, slots_in, slots_out
    if rank == 0:
        peaks, peak_src = load_peaks()
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(config_dict(w), parallelism=f"dp{world} (token shards, NCCL all-reduce of loss and dW_s)",
                           global_batch_tokens=w.N * world),
            "tflops": tflops, "tflops_unit": "TFLOP/s (4 N V (2 d_s + d_t) executed flops per rank-step, all ranks)",
            "pct_of_peak": 100.0 * tflops / (NOMINAL_BF16_TFLOPS * world),
            "peak_source": "NVIDIA dense bf16, 2250 TFLOP/s per GB300 (36 PFLOP/s 2:4-sparse per 8 GPUs / 2 / 8)",
            "loss": float(res.loss.item()), "cpu_baseline": None, "e2e": e2e,
            "gpu_launches": launches_per_step(w) * args.steps, "clocks": clk.summary(),
            "fwd_ms": fwd_avg, "bwd_ms": bwd_avg,
            "collective_ms": total_ms / args.steps - fwd_avg - bwd_avg,
        }
        peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        kernels = [
            {"kernel": "fused_kl_kernel (+combine, mean)", "ms": fwd_avg, "flops_per_launch": w.flops_fwd(),
             "tflops": w.flops_fwd() / (fwd_avg / 1e3) / 1e12},
            {"kernel": "bwd_pipe_kernel", "ms": bwd_avg, "flops_per_launch": w.flops_bwd(),
             "tflops": w.flops_bwd() / (bwd_avg / 1e3) / 1e12},
        ]
        for k in kernels:
            k["frac"] = k["tflops"] / peak_sus
        dom = max(kernels, key=lambda k: k["ms"])
        line["kernels"] = kernels
        line["roofline"] = {"kernel": dom["kernel"], "bound": "tensor", "achieved": dom["tflops"], "peak": peak_sus,
                            "unit": "TFLOP/s", "frac": dom["frac"],
                            "traffic": recorded_traffic(w.name, "hidden" if dom is kernels[1] else "hidden_fwd"),
                            "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                            "flops_per_launch": dom["flops_per_launch"]}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 10; 300 for --path logits and 500 for --path ild, whose steps "
                         "take about a millisecond, so that the clock sampler sees the timed region)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="stage2_64k", choices=list(syn.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count N (same shapes otherwise)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="hidden", choices=["hidden", "logits", "ild"],
                    help="hidden: the fused hidden-state KL (default); logits: the Fused KL on precomputed logits; "
                         "ild: the Stage-I ILD alignment loss")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph (reported as 'graph'; one GPU)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--split-g", action="store_true",
                    help="time hylo_kl_backward_split (G as two bf16 terms) instead of hylo_kl_backward")
    ap.add_argument("--cpu-tokens", type=int, default=256, help="oracle sample size for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=48, help="oracle tokens per reference-arm step")
    ap.add_argument("--dp-one-rank", action="store_true",
                    help="run the data-parallel step on a one-rank NCCL group (checks that code path on one GPU)")
    ap.add_argument("--mode", default="dp", choices=["dp", "replicas"],
                    help="under torchrun: dp = data-parallel token shards with NCCL all-reduce of loss and dW_s "
                         "(default); replicas = independent copies of the workload")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 10 if args.impl == "reference" else {"hidden": 10, "logits": 300, "ild": 500}[args.path]
    rank, world, local = dist_env()
    w = syn.WORKLOADS[args.workload]
    if args.tokens is not None:
        if args.tokens < 1:
            raise SystemExit("--tokens must be >= 1")
        # renamed: no DRAM-traffic record (taken per named workload) applies to another N
        w = w.with_sizes(N=args.tokens, name=f"{w.name}_n{args.tokens}")

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 or args.dp_one_rank:
        import torch.distributed as dist
        if world == 1:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", "29517")
            dist.init_process_group("nccl", device_id=dev, rank=0, world_size=1)
        else:
            dist.init_process_group("nccl", device_id=dev)
    if args.path in ("logits", "ild"):
        if args.path == "logits":
            run_logits(args, w, rank, world, local)
        else:
            run_ild(args, rank, world, local)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if (world > 1 and args.mode == "dp") or args.dp_one_rank:
        run_dp(args, w, rank, world, local)
        torch.distributed.destroy_process_group()
        return
    from hybrid_upcycling_gb300 import _lib, build
    if rank == 0:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    _lib.load()

    x = syn.make_inputs(w, device=dev)
    b = make_buffers(w, x, dev, split=args.split_g)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(w, x, b, stream)
    _lib.hylo_kl_sync_status(stream)

    # ----------------------------------------------------------------- device-resident timing
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(local)) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                step(w, x, b, stream, evs[i])
        torch.cuda.synchronize()
    barrier()
    _lib.hylo_kl_sync_status(stream)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(evs[0][0].elapsed_time(evs[-1][2]), world, dev)

    # ----------------------------------------------------------------- the same step as a CUDA graph
    graph = None
    if args.graph and world == 1:
        # one step (forward + backward: 4 kernels and the backward's counter memset) captured once
        # and replayed; the per-kernel figures above stay those of the eager loop
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(w, x, b, stream)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                g.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        _lib.hylo_kl_sync_status(stream)
        g_ms = ga.elapsed_time(gb)
        graph = {"ms_per_step": g_ms / args.steps, "value": whole_job_rate(w.N, 1, args.steps, g_ms),
                 "unit": "tokens/s", "steps": args.steps,
                 "what": "the step captured once in a CUDA graph and replayed (launch overhead removed)"}
        del g
    ms_per_step = total_ms / args.steps
    tokens_per_s = whole_job_rate(w.N, world, args.steps, total_ms)
    tflops = w.flops_exec() * world * args.steps / (total_ms / 1e3) / 1e12
    loss_val = float(b["loss"].item())

    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    fwd_avg, bwd_avg = float(np.mean(fwd_ms)), float(np.mean(bwd_ms))
    # split G: the gradient products run over both bf16 terms of G (twice the 4 N V d_s)
    bwd_flops = w.flops_bwd() + (4.0 * w.N * w.V * w.d_s if args.split_g else 0.0)
    kernels = [
        # the forward window also holds the combine and mean kernels (~0.1 ms at 64K)
        {"kernel": "fused_kl_kernel (+combine, mean)", "ms": fwd_avg, "flops_per_launch": w.flops_fwd(),
         "tflops": w.flops_fwd() / (fwd_avg / 1e3) / 1e12},
        {"kernel": "bwd_pipe_kernel", "ms": bwd_avg, "flops_per_launch": bwd_flops,
         "tflops": bwd_flops / (bwd_avg / 1e3) / 1e12},
    ]
    for k in kernels:
        k["frac"] = k["tflops"] / peak_sus
    dom = max(kernels, key=lambda k: k["ms"])
    traffic = recorded_traffic(w.name, "hidden" if dom is kernels[1] else "hidden_fwd")

    # ----------------------------------------------------------------- end-to-end via host buffers
    e2e = None
    if not args.no_e2e:
        # Every step copies its inputs in from pinned host memory and its results (kl, loss, dh_s,
        # dW_s) out (double-buffered, see pipelined_e2e).
        host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in x.items()}
        for k in x:
            host[k].copy_(x[k])
        xd = [{k: torch.empty_like(v) for k, v in x.items()} for _ in range(2)]
        # one shared workspace (and flags); fresh output buffers for the second slot
        bo = [b, {k: (torch.empty_like(v) if torch.is_tensor(v) and k != "ws" else v) for k, v in b.items()}]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        e2e_steps = max(2, min(args.steps, 10))  # fill and drain (first upload, last download) amortised over the steps
        barrier()
        e2e_ms, d2h = pipelined_e2e(host, xd, bo, ("kl", "loss", "dh", "dW"),
                                    lambda xi, xo: step(w, xi, xo, stream), e2e_steps, stream, dev)
        barrier()
        _lib.hylo_kl_sync_status(stream)
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        e2e = {"value": whole_job_rate(w.N, world, e2e_steps, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "api": "hylo_kl_forward + hylo_kl_backward (C ABI) with pinned-host inputs/outputs, "
                      "copies double-buffered on their own streams"}
        del xd, host, bo

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res = []
        n_s = len(sample_rows(w.N, args.cpu_tokens))
        prepared = oracle_inputs(w, x, n_s)
        calls, dt = time_repeated(lambda: res.append(cpu_oracle_rate(w, x, n_s, inputs=prepared)[1]))
        rate = n_s * calls / sum(res)
        cpu = {"value": rate, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{calls} x {n_s} tokens of {w.name} (full V and d), fp64 numpy "
                         f"forward+backward, {sum(res):.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(config_dict(w), **({"g_terms": 2} if args.split_g else {})),
            "tflops": tflops, "tflops_unit": "TFLOP/s (4 N V (2 d_s + d_t) executed flops per step)",
            "pct_of_peak": 100.0 * tflops / NOMINAL_BF16_TFLOPS,
            "peak_source": "NVIDIA dense bf16, 2250 TFLOP/s per GB300 (36 PFLOP/s 2:4-sparse per 8 GPUs / 2 / 8)",
            "pct_of_measured_peak": 100.0 * tflops / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
            "measured_peak_source": f"bf16_tflops ({peak_src}, cuBLAS 8192^3 burst)",
            "ms_x_median_sm_ghz": None,
            "fwd_ms": fwd_avg, "bwd_ms": bwd_avg, "loss": loss_val,
            "kernels": kernels,
            "roofline": {"kernel": dom["kernel"], "bound": "tensor",
                         "achieved": dom["tflops"], "peak": peak_sus, "unit": "TFLOP/s", "frac": dom["frac"],
                         "traffic": traffic, "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                         "flops_per_launch": dom["flops_per_launch"]},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step(w, args.split_g) * args.steps,
            **({"graph": graph} if graph is not None else {}),
            "clocks": clk.summary(),
            "memory": {"workspace_bytes": int(b["ws"].numel()), "dense_fp32_logits_bytes": 4 * w.N * w.V,
                       "note": "the library allocates nothing; the caller's workspace is its only scratch"},
        }
        if line["clocks"].get("sm_mhz"):
            line["ms_x_median_sm_ghz"] = ms_per_step * line["clocks"]["sm_mhz"] / 1e3
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
