"""Benchmark of the hot path: fused selected-token logprob + mismatch statistics.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

One step = tim_token_logprob over a Qwen3-8B-shaped LM head (N = 8192 tokens,
D = 4096, V = 151936, bf16 operands, fp32 accumulation) followed by
tim_mismatch_stats over its output against synthetic rollout logprobs (16
sequences x 512 tokens, first 128 of each masked as prompt, C = 2).  The head
weight (1.2 GB) is larger than L2, and L2 is also flushed (a 256 MiB write)
before every timed step.  Steps are timed with CUDA events on the launching
stream; the timed region is bracketed by a barrier and a device synchronise;
the max over ranks is reported.  With --gpus N > 1 (under torchrun) every rank
runs its own replica of the workload: the path shards by rows with no
exchange, so value = N x tokens / max-rank time ("scaling": "weak").

--impl reference times the fp64 CPU oracle (the only other implementation of
the method) on the host cores over a bounded row sample of the same workload.
Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "fused selected-token logprob tokens/s and TFLOP/s vs GB300 dense bf16 peak"
UNIT = "tokens/s"
WORKLOAD = "qwen3_8b"
K2_BW_TOKENS = 1 << 27


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of
# the kernel at the benchmark's shape, keyed by a hash of the kernel's sources at capture time;
# reported as `traffic` (with `traffic_source`) only while the sources are unchanged, else null.
MEASURED_TRAFFIC = {
    # token logprob, N = 8192, D = 4096, V = 151936: 2666996480 read + 15407872 written
    ("k1", "78fc418be590bdf5"): 2666996480 + 15407872,
    # mismatch pass, 2^27 tokens (sequence kernel + fold): 1229469952 read + 496668160 written
    ("k2", "c4e714ca643ef1b7"): 1222002176 + 7467776 + 496668160,
    # TIS-weighted PPO surrogate, 2^27 tokens (sequence + fold): 2497949440 read + 1027808000 written
    ("ppo", "a17407344a379435"): 2494668800 + 3280640 + 1027808000,
    # mismatch monitor, 2^27 tokens, its three kernels: 1227772160 read + 109240320 written
    ("monitor", "eb7d64113d4ae0f5"): 9882624 + 1208898304 + 8991232 + 109240320,
}
TRAFFIC_SOURCE = "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch at this shape, " \
                 "stored with a hash of the kernel sources it was taken on"
K2_TRAFFIC_TOKENS = 1 << 27       # the captures were taken at the bandwidth runs' size
PPO_TRAFFIC_TOKENS = 1 << 27
MONITOR_TRAFFIC_TOKENS = 1 << 27
# L2 flush before each timed launch of a single call: 1 GiB, 8x the L2; its
# ~0.15 ms fill also lets the host enqueue the timed call before the GPU
# reaches the start event, so host-side call overhead stays out of the time.
FLUSH_BYTES = 1 << 30


def source_hash(kind: str) -> str:
    import hashlib
    d = os.path.join(ROOT, "rollout_logprob_mismatch_gb300", "csrc")
    files = {"k1": ("k1_token_logprob.cu", "k1_internal.h", "tim_ptx.cuh", "tim_internal.h", "unit_ring.cuh"),
             "k2": ("k2_mismatch_stats.cu", "k2_internal.h", "tim_ptx.cuh", "tim_internal.h"),
             "ppo": ("tis_ppo.cu", "ppo_internal.h", "tim_ptx.cuh", "tim_internal.h"),
             "monitor": ("mismatch_monitor.cu", "monitor_internal.h", "tim_ptx.cuh", "tim_internal.h")}[kind]
    m = hashlib.sha1()
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def measured_traffic(kind: str):
    return MEASURED_TRAFFIC.get((kind, source_hash(kind)))


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------- dist helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(world: int, tokens_per_rank: int, steps: int, t_max: float) -> float:
    """Whole-job tokens/s: every rank processed `tokens_per_rank` tokens per step;
    the job took the slowest rank's time."""
    return world * tokens_per_rank * steps / t_max


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload
def make_workload(seed: int = 0, tokens: int | None = None):
    cfg = wl.CONFIGS[WORKLOAD]
    if tokens:   # a smaller batch of the same head, for profiling runs (whole sequences of 512)
        n = max(512, tokens // 512 * 512)
        cfg = dataclasses.replace(cfg, N=n, num_seqs=n // 512)
    h, W = wl.draw_head(cfg, seed=seed)
    a = wl.draw_targets(cfg, cfg.N, seed=seed)
    off = wl.draw_segments(cfg, seed=seed)
    mask = wl.draw_mask(cfg, off, seed=seed)
    return cfg, h, W, a, off, mask


def stream_of(dev):
    import torch
    return torch.cuda.current_stream(dev)


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(cfg, h, W, a, off, mask, budget_s: float, seed: int = 0):
    """The oracle on a bounded sample: token logprob on R rows (all host
    threads), mismatch statistics on the whole batch.  Returns (tokens/s,
    description, threads, seconds spent)."""
    import oracle
    threads = cpu_threads()
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    probe_rows = rng.choice(cfg.N, size=min(cfg.N, threads), replace=False)
    oracle.token_logprob(h, W, a, rows=probe_rows, nthreads=threads)
    t_round = time.perf_counter() - t0          # one row on every thread
    rounds = max(1, int(budget_s / max(t_round, 1e-3)))
    R = min(cfg.N, rounds * threads)
    rows = rng.choice(cfg.N, size=R, replace=False)
    t0 = time.perf_counter()
    lp, _ = oracle.token_logprob(h, W, a, rows=rows, nthreads=threads)
    t_k1 = time.perf_counter() - t0
    l_tr = np.full(cfg.N, -1.0, np.float32)
    l_tr[rows] = lp.astype(np.float32)
    l_ro = wl.draw_rollout(cfg, l_tr, seed=seed)
    t0 = time.perf_counter()
    oracle.mismatch_stats(l_tr, l_ro, mask, off, C=cfg.C)
    t_k2_1 = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.mismatch_stats(l_tr, l_ro, mask, off, C=cfg.C, nthreads=threads)
    t_k2 = time.perf_counter() - t0
    sec_per_token = t_k1 / R + t_k2 / cfg.N
    desc = ("token logprob on %d of %d rows (%d threads, %.1f s) + mismatch stats on all %d tokens "
            "(%d threads %.4f s; 1 thread %.4f s), extrapolated to tokens/s"
            % (R, cfg.N, threads, t_k1, cfg.N, threads, t_k2, t_k2_1))
    return 1.0 / sec_per_token, desc, threads, t_k1 + t_k2


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg, h, W, a, off, mask = make_workload()
    budget = float(os.environ.get("TIM_BENCH_ORACLE_SECONDS", "8"))
    vals = []
    desc, threads = "", 1
    for i in range(args.warmup + args.steps):
        v, desc, threads, _ = time_oracle(cfg, h, W, a, off, mask, budget / max(1, args.steps), seed=i)
        if i >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": cfg.N / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg):
    return {"workload": "%s_head+mismatch" % cfg.name, "N": cfg.N, "D": cfg.D, "V": cfg.V,
            "num_seqs": cfg.num_seqs, "seq_len": cfg.seq_len, "prompt_len": cfg.prompt_len, "C": cfg.C,
            "operands": "bf16 h[N,D], bf16 W[V,D], fp32 accumulate",
            "l2": "weights 1.2 GB > L2, and L2 flushed (256 MiB write) before each timed step"}


# ----------------------------------------------------------------------------- gb300 arm
def run_gb300(args):
    import torch
    import rollout_logprob_mismatch_gb300 as tim
    from rollout_logprob_mismatch_gb300 import build as tim_build

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = dist_init(world, "nccl")
    if rank == 0 or dist is None:
        tim_build.build()
    barrier(dist, dev)
    tim.load()
    peaks = load_peaks()

    if args.only == "monitor":
        r = monitor_bandwidth(tim, dev, stream_of(dev), peaks, tokens=args.tokens or K2_BW_TOKENS,
                              reps=args.steps, warmup=args.warmup)
        tim.check()
        if rank == 0:
            print(json.dumps(r))
        return 0
    if args.only == "ppo":
        r = ppo_bandwidth(tim, dev, stream_of(dev), peaks, tokens=args.tokens or K2_BW_TOKENS,
                          reps=args.steps, warmup=args.warmup)
        tim.check()
        if rank == 0:
            print(json.dumps(r))
        return 0
    if args.only == "k2bw":
        # the mismatch pass alone on a large batch (profiling runs)
        r = mismatch_bandwidth(tim, dev, stream_of(dev), peaks, tokens=args.tokens or K2_BW_TOKENS,
                               reps=args.steps, warmup=args.warmup)
        tim.check()
        if rank == 0:
            print(json.dumps(r))
        return 0
    if args.only == "k1" and args.head != WORKLOAD:
        r = k1_head_only(tim, dev, stream_of(dev), args.head, reps=args.steps, warmup=args.warmup)
        tim.check()
        if rank == 0:
            print(json.dumps(r))
        return 0
    cfg, h, W, a, off, mask = make_workload(seed=rank, tokens=args.tokens)
    N, D, V = cfg.N, cfg.D, cfg.V
    stream = torch.cuda.current_stream(dev)
    hd = torch.from_numpy(h.view(np.int16)).to(dev).view(torch.bfloat16)
    Wd = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    ad = torch.from_numpy(a).to(dev)
    offd = torch.from_numpy(off).to(dev)
    maskd = torch.from_numpy(mask).to(dev)
    lp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    # rollout logprobs = trainer logprobs + N(0, 0.01^2), drawn once from a first pass
    tim.token_logprob(hd, Wd, ad, lp, lse)
    l_ro = wl.draw_rollout(cfg, lp.cpu().numpy(), seed=rank)
    rod = torch.from_numpy(l_ro).to(dev)
    S = len(off) - 1
    k2out = {"seq_stats": torch.empty((S, 12), dtype=torch.float32, device=dev),
             "seq_flags": torch.empty(S, dtype=torch.int32, device=dev),
             "batch": torch.empty(20, dtype=torch.float64, device=dev), "token_weight": None}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        tim.token_logprob(hd, Wd, ad, lp, lse)
        tim.mismatch_stats(lp, rod, maskd, offd, C=cfg.C, out=k2out)

    if args.only == "backward":
        r = backward_measure(tim, dev, stream, peaks, hd, Wd, ad, reps=args.steps, warmup=args.warmup)
        tim.check()
        if rank == 0:
            print(json.dumps(r))
        return 0
    if args.only == "fp32head":
        r = fp32_head_measure(tim, dev, stream, peaks, hd, ad, V, reps=args.steps, warmup=args.warmup)
        tim.check()
        if rank == 0:
            print(json.dumps(r))
        return 0

    if args.only:
        # one kernel family alone (profiling runs): warm-up, then timed launches
        fn = (lambda: tim.token_logprob(hd, Wd, ad, lp, lse)) if args.only == "k1" else \
             (lambda: tim.mismatch_stats(lp, rod, maskd, offd, C=cfg.C, out=k2out))
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tim.check()
        if rank == 0:
            print(json.dumps({"only": args.only, "N": N, "avg_launch_ms": e0.elapsed_time(e1) / args.steps}))
        return 0
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    tim.check()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index).__enter__()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        tim.token_logprob(hd, Wd, ad, lp, lse)
        ev[i][1].record(stream)
        tim.mismatch_stats(lp, rod, maskd, offd, C=cfg.C, out=k2out)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    tim.check()
    t_k1 = [ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(K)]
    t_k2 = [ev[i][1].elapsed_time(ev[i][2]) * 1e-3 for i in range(K)]
    t_step = sum(t_k1) + sum(t_k2)
    t_max = max_over_ranks(t_step, dist, dev)
    value = aggregate_value(world, N, K, t_max)
    k1_avg = float(np.mean(t_k1))
    k2_avg = float(np.mean(t_k2))
    flops = 2.0 * N * V * D
    achieved = flops / k1_avg / 1e12

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    h_host = torch.from_numpy(h.view(np.int16)).pin_memory()
    a_host = torch.from_numpy(a).pin_memory()
    ro_host = torch.from_numpy(l_ro).pin_memory()
    m_host = torch.from_numpy(mask).pin_memory()
    o_host = torch.from_numpy(off).pin_memory()
    b_host = torch.empty(20, dtype=torch.float64).pin_memory()
    s_host = torch.empty((S, 12), dtype=torch.float32).pin_memory()
    f_host = torch.empty(S, dtype=torch.int32).pin_memory()
    # two device copies of the inputs: while step i computes on one, the copy
    # stream brings step i + 1's inputs into the other (every step's inputs
    # still cross host -> device inside the timed span)
    bufs = [{"h": torch.empty((N, D), dtype=torch.int16, device=dev),
             "a": torch.empty(N, dtype=torch.int32, device=dev),
             "ro": torch.empty(N, dtype=torch.float32, device=dev),
             "m": torch.empty(N, dtype=torch.uint8, device=dev),
             "o": torch.empty(S + 1, dtype=torch.int32, device=dev)} for _ in range(2)]
    copy_stream = torch.cuda.Stream(dev)

    def upload(buf):
        buf["h"].copy_(h_host, non_blocking=True)
        buf["a"].copy_(a_host, non_blocking=True)
        buf["ro"].copy_(ro_host, non_blocking=True)
        buf["m"].copy_(m_host, non_blocking=True)
        buf["o"].copy_(o_host, non_blocking=True)

    def run_e2e(steps):
        """`steps` steps through the public API; returns the span in seconds."""
        copied = [torch.cuda.Event() for _ in range(steps)]
        done = [torch.cuda.Event() for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy_stream.wait_event(t0)
        with torch.cuda.stream(copy_stream):
            upload(bufs[0])
        copied[0].record(copy_stream)
        for i in range(steps):
            buf = bufs[i % 2]
            stream.wait_event(copied[i])
            tim.token_logprob(buf["h"].view(torch.bfloat16), Wd, buf["a"], lp, lse)
            tim.mismatch_stats(lp, buf["ro"], buf["m"], buf["o"], C=cfg.C, out=k2out)
            done[i].record(stream)
            b_host.copy_(k2out["batch"], non_blocking=True)
            s_host.copy_(k2out["seq_stats"], non_blocking=True)
            f_host.copy_(k2out["seq_flags"], non_blocking=True)
            if i + 1 < steps:   # the other buffer is free once step i - 1 has finished with it
                if i >= 1:
                    copy_stream.wait_event(done[i - 1])
                with torch.cuda.stream(copy_stream):
                    upload(bufs[(i + 1) % 2])
                copied[i + 1].record(copy_stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) * 1e-3

    run_e2e(args.warmup)
    barrier(dist, dev)
    t_e2e = run_e2e(K)
    clocks.__exit__(None, None, None)   # sampled over both timed regions
    t_e2e = max_over_ranks(t_e2e, dist, dev)
    h2d = h_host.numel() * 2 + a_host.numel() * 4 + ro_host.numel() * 4 + m_host.numel() + o_host.numel() * 4
    d2h = b_host.numel() * 8 + s_host.numel() * 4 + f_host.numel() * 4

    k2_bw = mismatch_bandwidth(tim, dev, stream, peaks) if not args.skip_k2_bandwidth else None
    ppo_bw = ppo_bandwidth(tim, dev, stream, peaks) if not args.skip_ppo else None
    mon_bw = monitor_bandwidth(tim, dev, stream, peaks) if not args.skip_monitor else None
    sweep = batch_size_sweep(tim, dev, stream, Wd, D, V, peaks) if not args.skip_sweep else None
    heads = head_shapes_measure(tim, dev, stream, peaks) if not args.skip_heads else None
    fp32h = fp32_head_measure(tim, dev, stream, peaks, hd, ad, V) if not args.skip_fp32_head else None
    bwd = backward_measure(tim, dev, stream, peaks, hd, Wd, ad) if not args.skip_backward else None
    tim.check()

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.skip_cpu_baseline:
        v, desc, threads, _ = time_oracle(cfg, h, W, a, off, mask,
                                          float(os.environ.get("TIM_BENCH_ORACLE_SECONDS", "16")))
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
    peak = peaks["bf16_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_max / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg),
        "tflops": world * flops * K / t_max / 1e12,
        "roofline": {"kernel": "tim_token_logprob (fused LM head + online LSE + gather)",
                     "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": "%s bf16 burst" % peaks["source"],
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "traffic": measured_traffic("k1") if (N, D, V) == (8192, 4096, 151936) else None,
                     "traffic_source": TRAFFIC_SOURCE if measured_traffic("k1") is not None else None,
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "algorithmic_bytes_per_launch": 2 * N * D + 2 * V * D + 12 * N,
                     "algorithmic_flops_per_launch": flops,
                     "avg_launch_ms": k1_avg * 1e3},
        "mismatch_pass": {"avg_launch_us": k2_avg * 1e6,
                          "algorithmic_bytes": 9 * N + 4 * (S + 1) + 52 * S + 160},
        "cpu_baseline": cpu,
        "e2e": {"value": aggregate_value(world, N, K, t_e2e), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": 4 * K,
        "clocks": clocks.summary(),
    }
    if k2_bw is not None:
        line["mismatch_bandwidth"] = k2_bw
    if ppo_bw is not None:
        line["tis_ppo"] = ppo_bw
    if mon_bw is not None:
        line["mismatch_monitor"] = mon_bw
    if fp32h is not None:
        line["fp32_head"] = fp32h
    if bwd is not None:
        line["backward"] = bwd
    if sweep is not None:
        line["sweep"] = sweep
    if heads is not None:
        line["head_shapes"] = heads
    print(json.dumps(line), flush=True)
    return 0


def k1_head_only(tim, dev, stream, name, reps, warmup):
    """The token logprob alone on another head shape of the workloads (profiling
    runs): h ~ N(0, 1), W ~ N(0, w_std^2) in bf16 and uniform targets drawn on
    the device, as in head_shapes_measure."""
    import torch
    cfg = wl.CONFIGS[name]
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    N, D, V = cfg.N, cfg.D, cfg.V
    h = (torch.randn((N, D), generator=g, device=dev) * cfg.h_std).to(torch.bfloat16)
    W = (torch.randn((V, D), generator=g, device=dev) * cfg.w_std).to(torch.bfloat16)
    a = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int32)
    lp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    for _ in range(warmup):
        tim.token_logprob(h, W, a, lp, lse)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        tim.token_logprob(h, W, a, lp, lse)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t = e0.elapsed_time(e1) * 1e-3 / reps
    return {"only": "k1", "head": name, "N": N, "D": D, "V": V, "avg_launch_ms": t * 1e3,
            "tflops": 2.0 * N * V * D / t / 1e12}


def draw_head_on_device(cfg, g, dev):
    """h, W and targets with the laws of the workload config, drawn on the
    device: h ~ N(0, h_std^2) with an iid fraction h_outlier_frac of entries
    scaled by h_outlier_scale, W ~ N(0, w_std^2), both rounded to bf16;
    targets uniform, or for "top5mix" 70% a uniform pick among the row's five
    largest logits (from a plain torch matmul: input shaping only) and 30%
    uniform."""
    import torch
    N, D, V = cfg.N, cfg.D, cfg.V
    h = torch.randn((N, D), generator=g, device=dev) * cfg.h_std
    if cfg.h_outlier_frac > 0.0:
        hit = torch.rand((N, D), generator=g, device=dev) < cfg.h_outlier_frac
        h = torch.where(hit, h * cfg.h_outlier_scale, h)
        del hit
    h = h.to(torch.bfloat16)
    W = (torch.randn((V, D), generator=g, device=dev) * cfg.w_std).to(torch.bfloat16)
    a = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int32)
    if cfg.target_mode == "top5mix":
        top5 = torch.empty((N, 5), dtype=torch.int64, device=dev)
        for s in range(0, N, 2048):
            top5[s:s + 2048] = torch.topk((h[s:s + 2048] @ W.T).float(), 5, dim=-1).indices
        pick = torch.rand(N, generator=g, device=dev) < 0.7
        col = torch.randint(0, 5, (N, 1), generator=g, device=dev)
        a = torch.where(pick, top5.gather(1, col)[:, 0].to(torch.int32), a)
        del top5
    return h, W, a


def draw_rollout_on_device(cfg, lp, g):
    """Rollout logprobs with the config's laws: trainer + N(0, rollout_std^2),
    plus an iid fraction outlier_frac of tokens shifted by +-outlier_shift."""
    import torch
    ro = lp + cfg.rollout_std * torch.randn(lp.shape[0], generator=g, device=lp.device)
    if cfg.outlier_frac > 0.0:
        hit = torch.rand(lp.shape[0], generator=g, device=lp.device) < cfg.outlier_frac
        sign = torch.where(torch.rand(lp.shape[0], generator=g, device=lp.device) < 0.5, -1.0, 1.0)
        ro = torch.where(hit, ro + sign * cfg.outlier_shift, ro)
    return ro


def head_shapes_measure(tim, dev, stream, peaks, names=("llama3_8b", "dsv3"), reps=5, warmup=2):
    """The step (token logprob + mismatch statistics) on the other head shapes
    of the workloads: the Llama-3-8B-shaped head (N = 32768 in lognormal
    sequences, 30% masked, rollout outliers of +-1.0 on 0.5% of tokens) and
    the DeepSeek-V3-shaped one (N = 16384, D = 7168, 32 x 512, 1% of h entries
    scaled x20, 70% of targets among each row's top-5 logits), all inputs with
    the configs' laws, drawn on the device; L2 flushed before each step.  The
    token logprob is also timed on plain inputs (h, W Gaussian, uniform
    targets) of the same shapes, to show what the values change."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = []

    def time_step(h, W, a, ro, maskd, offd, lp, lse, k2out, with_k2=True):
        for _ in range(warmup):
            tim.token_logprob(h, W, a, lp, lse)
            if with_k2:
                tim.mismatch_stats(lp, ro, maskd, offd, C=cfg.C, out=k2out)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        for i in range(reps):
            flush.fill_(i)
            ev[i][0].record(stream)
            tim.token_logprob(h, W, a, lp, lse)
            ev[i][1].record(stream)
            if with_k2:
                tim.mismatch_stats(lp, ro, maskd, offd, C=cfg.C, out=k2out)
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        return (float(np.mean([e[0].elapsed_time(e[1]) * 1e-3 for e in ev])),
                float(np.mean([e[1].elapsed_time(e[2]) * 1e-3 for e in ev])))

    for name in names:
        cfg = wl.CONFIGS[name]
        N, D, V = cfg.N, cfg.D, cfg.V
        off = wl.draw_segments(cfg, seed=0)
        S = len(off) - 1
        offd = torch.from_numpy(off).to(dev)
        maskd = torch.from_numpy(wl.draw_mask(cfg, off, seed=0)).to(dev)
        lp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        k2out = {"seq_stats": torch.empty((S, 12), dtype=torch.float32, device=dev),
                 "seq_flags": torch.empty(S, dtype=torch.int32, device=dev),
                 "batch": torch.empty(20, dtype=torch.float64, device=dev), "token_weight": None}
        h, W, a = draw_head_on_device(cfg, g, dev)
        tim.token_logprob(h, W, a, lp, lse)
        ro = draw_rollout_on_device(cfg, lp, g)
        t1, t2 = time_step(h, W, a, ro, maskd, offd, lp, lse, k2out)
        del h, W, a
        # the same shapes on plain inputs: what the input values change
        hp = (torch.randn((N, D), generator=g, device=dev) * cfg.h_std).to(torch.bfloat16)
        Wp = (torch.randn((V, D), generator=g, device=dev) * cfg.w_std).to(torch.bfloat16)
        ap = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int32)
        t1p, _ = time_step(hp, Wp, ap, ro, maskd, offd, lp, lse, k2out, with_k2=False)
        del hp, Wp, ap
        flops = 2.0 * N * V * D
        out.append({"workload": "%s_head+mismatch" % name, "N": N, "D": D, "V": V, "num_seqs": S,
                    "inputs": "the config's laws (outliers, top-5 targets where the config has them)",
                    "step_ms": (t1 + t2) * 1e3, "tokens_per_s": N / (t1 + t2),
                    "token_logprob_ms": t1 * 1e3, "tflops": flops / t1 / 1e12,
                    "frac": flops / t1 / 1e12 / peaks["bf16_tflops"], "bound": "tensor",
                    "frac_of_sustained": flops / t1 / 1e12 / peaks["bf16_tflops_sustained"],
                    "mismatch_pass_us": t2 * 1e6,
                    "token_logprob_ms_plain_inputs": t1p * 1e3})
        del lp, lse, ro
    return out


def batch_size_sweep(tim, dev, stream, Wd, D, V, peaks, sizes=(1, 7, 512, 4096, 32768), reps=5):
    """tim_token_logprob alone on the same head at the batch-invariance sweep's
    batch sizes (random rows; L2 flushed before each launch).  Small batches
    are bound by reading W from HBM, so GB/s of W + h is reported beside TFLOP/s."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = []
    for n in sizes:
        h = torch.randn((n, D), generator=g, device=dev).to(torch.bfloat16)
        a = torch.randint(0, V, (n,), generator=g, device=dev, dtype=torch.int32)
        lp = torch.empty(n, dtype=torch.float32, device=dev)
        lse = torch.empty(n, dtype=torch.float32, device=dev)
        for _ in range(2):
            tim.token_logprob(h, Wd, a, lp, lse)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
        for i in range(reps):
            flush.fill_(i)
            ev[i][0].record(stream)
            tim.token_logprob(h, Wd, a, lp, lse)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t = float(np.mean([e0.elapsed_time(e1) * 1e-3 for e0, e1 in ev]))
        bytes_ = 2.0 * V * D + 2.0 * n * D + 12.0 * n
        out.append({"N": n, "avg_launch_us": t * 1e6, "tokens_per_s": n / t,
                    "tflops": 2.0 * n * V * D / t / 1e12, "hbm_gbs": bytes_ / t / 1e9,
                    "hbm_frac": bytes_ / t / 1e9 / peaks["hbm_gbs"]})
        del h, a, lp, lse
    return out


def mismatch_bandwidth(tim, dev, stream, peaks, tokens=K2_BW_TOKENS, reps=10, warmup=3):
    """tim_mismatch_stats alone on `tokens` tokens (2^27 by default) in
    Llama-like segments (lognormal lengths, median 1024, clipped to
    [128, 4096]), 30% masked, with per-token weights written; L2 flushed before
    each launch.  Reports HBM GB/s."""
    import torch
    Nt = tokens
    cfg = wl.HeadConfig("bw", N=Nt, D=8, V=8, seq_layout="lognormal", mask_drop=0.3)
    off = wl.draw_segments(cfg, seed=7)
    S = len(off) - 1
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    l_tr = torch.log(torch.rand(Nt, device=dev, generator=g).clamp_min_(1e-30))
    l_ro = l_tr + 0.02 * torch.randn(Nt, device=dev, generator=g)
    mask = (torch.rand(Nt, device=dev, generator=g) >= 0.3).to(torch.uint8)
    offd = torch.from_numpy(off).to(dev)
    out = {"seq_stats": torch.empty((S, 12), dtype=torch.float32, device=dev),
           "seq_flags": torch.empty(S, dtype=torch.int32, device=dev),
           "batch": torch.empty(20, dtype=torch.float64, device=dev),
           "token_weight": torch.empty(Nt, dtype=torch.float32, device=dev)}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        tim.mismatch_stats(l_tr, l_ro, mask, offd, out=out)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        flush.fill_(i)
        ev[i][0].record(stream)
        tim.mismatch_stats(l_tr, l_ro, mask, offd, out=out)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(reps)]))
    algo = 9 * Nt + 4 * Nt + 4 * (S + 1) + 52 * S + 160
    gbs = algo / t / 1e9
    tr = measured_traffic("k2")
    return {"tokens": Nt, "num_seqs": S, "avg_launch_us": t * 1e6, "algorithmic_bytes": algo,
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
            "frac_of_8000": gbs / 8000.0, "bound": "hbm",
            "traffic": None if tr is None or Nt != K2_TRAFFIC_TOKENS else tr,
            "traffic_source": None if tr is None or Nt != K2_TRAFFIC_TOKENS else TRAFFIC_SOURCE}


def backward_measure(tim, dev, stream, peaks, hd, Wd, ad, reps=5, warmup=2):
    """The token logprob's backward on the bench's head shape: g ~ N(0, 1) per
    token, lse from the forward; one call = per row chunk (up to 16384 rows)
    the fused dz kernel (logits recomputed, never stored in fp32) and one
    launch of the pair-UMMA GEMMs dh = dz W and dW (+)= dz^T h; L2 flushed
    before each call.
    Work 3 x 2NVD FLOP (recompute, dh, dW) against the bf16 peak: five calls
    back to back (they run at the power cap: burst and sustained fractions),
    and three single calls each after 0.2 s without work (burst)."""
    import torch
    N, D = hd.shape
    V = Wd.shape[0]
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    grad = torch.randn(N, generator=g, device=dev)
    _, lse = tim.token_logprob(hd, Wd, ad)
    dh = torch.empty((N, D), dtype=torch.float32, device=dev)
    dW = torch.empty((V, D), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        tim.token_logprob_backward(hd, Wd, ad, grad, lse, dh=dh, dW=dW)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        flush.fill_(i)
        ev[i][0].record(stream)
        tim.token_logprob_backward(hd, Wd, ad, grad, lse, dh=dh, dW=dW)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(reps)]))
    # The same call after the GPU has idled (a trainer's backward between other
    # work): each of three calls follows an L2 flush and 0.2 s without work.
    singles = []
    for i in range(3):
        flush.fill_(i)
        torch.cuda.synchronize(dev)
        time.sleep(0.2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        tim.token_logprob_backward(hd, Wd, ad, grad, lse, dh=dh, dW=dW)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        singles.append(e0.elapsed_time(e1) * 1e-3)
    t1 = float(np.mean(singles))
    flops = 3 * 2.0 * N * V * D
    del dh, dW
    return {"N": N, "D": D, "V": V, "avg_call_ms": t * 1e3, "tokens_per_s": N / t,
            "tflops": flops / t / 1e12, "bound": "tensor", "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": flops / t / 1e12 / peaks["bf16_tflops"],
            "frac_of_sustained": flops / t / 1e12 / peaks["bf16_tflops_sustained"],
            "timing": "%d calls back to back (the power cap holds the clock down)" % reps,
            "single_call_ms": t1 * 1e3, "single_call_tflops": flops / t1 / 1e12,
            "single_call_frac": flops / t1 / 1e12 / peaks["bf16_tflops"],
            "single_call_timing": "3 calls, each after 0.2 s idle and an L2 flush; against the burst peak",
            "parts": "per row chunk: fused dz kernel + one launch of both GEMMs dh, dW (tcgen05 pair UMMA, ours)"}


def fp32_head_measure(tim, dev, stream, peaks, hd, ad, V, reps=5, warmup=3):
    """The FP32 LM head on the bench's head shape: fp32 W ~ N(0, 0.02^2) drawn
    on the device, split into three bf16 parts (timed: HBM-bound, 4 B read +
    6 B written per weight), then the fused token logprob over the parts
    (timed; L2 flushed before each call).  TFLOP/s are given both as the fp32
    head's 2NVD and as the 3 x 2NVD bf16 tensor work against the bf16 peak."""
    import torch
    N, D = hd.shape
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    Wf = torch.randn((V, D), generator=g, device=dev) * 0.02
    Ws = tim.split_weight_fp32(Wf)
    lp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        tim.token_logprob_fp32_head(hd, Ws, ad, lp, lse)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        flush.fill_(i)
        ev[i][0].record(stream)
        tim.split_weight_fp32(Wf, out=Ws)
        ev[i][1].record(stream)
        flush.fill_(i + 1)
        ev[i][2].record(stream)
        tim.token_logprob_fp32_head(hd, Ws, ad, lp, lse)
        ev[i][3].record(stream)
    torch.cuda.synchronize(dev)
    t_split = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(reps)]))
    t_head = float(np.mean([ev[i][2].elapsed_time(ev[i][3]) * 1e-3 for i in range(reps)]))
    flops = 2.0 * N * V * D
    split_bytes = 4 * V * D + Ws.numel() * 2
    del Wf, Ws
    return {"N": N, "D": D, "V": V, "avg_launch_ms": t_head * 1e3, "tokens_per_s": N / t_head,
            "fp32_head_tflops": flops / t_head / 1e12, "tensor_tflops": 3 * flops / t_head / 1e12,
            "bound": "tensor", "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": 3 * flops / t_head / 1e12 / peaks["bf16_tflops"],
            "split": {"avg_us": t_split * 1e6, "bytes": split_bytes, "gbs": split_bytes / t_split / 1e9,
                      "frac_of_hbm": split_bytes / t_split / 1e9 / peaks["hbm_gbs"]}}


def monitor_bandwidth(tim, dev, stream, peaks, tokens=K2_BW_TOKENS, reps=10, warmup=3):
    """tim_mismatch_monitor alone on `tokens` tokens (2^27 by default), inputs
    drawn on the device like the mismatch pass's (30% masked, delta ~
    N(0, 0.02^2)), rejection flags written; L2 flushed before each call.
    Algorithmic bytes: one read of the inputs and the flags written (10 B per
    token); the design reads them once more for its sample (at most 2^20
    tokens) and moves the few percent of keys it collects."""
    import torch
    Nt = tokens
    g = torch.Generator(device=dev)
    g.manual_seed(8)
    l_tr = torch.log(torch.rand(Nt, device=dev, generator=g).clamp_min_(1e-30))
    l_ro = l_tr + 0.02 * torch.randn(Nt, device=dev, generator=g)
    mask = (torch.rand(Nt, device=dev, generator=g) >= 0.3).to(torch.uint8)
    out = {"batch": torch.empty(7, dtype=torch.float64, device=dev),
           "token_reject": torch.empty(Nt, dtype=torch.uint8, device=dev)}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    call = lambda: tim.mismatch_monitor(l_tr, l_ro, mask, 0.05, out=out)  # noqa: E731
    for _ in range(warmup):
        call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        flush.fill_(i)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(reps)]))
    algo = 10 * Nt + 56
    gbs = algo / t / 1e9
    tr = measured_traffic("monitor")
    return {"tokens": Nt, "avg_launch_us": t * 1e6, "algorithmic_bytes": algo, "achieved": gbs,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "bound": "hbm",
            "passes_over_inputs": 1, "sample_tokens": min(Nt, 1 << 20),
            "tokens_per_s": Nt / t,
            "traffic": None if tr is None or Nt != MONITOR_TRAFFIC_TOKENS else tr,
            "traffic_source": None if tr is None or Nt != MONITOR_TRAFFIC_TOKENS else TRAFFIC_SOURCE}


def ppo_bandwidth(tim, dev, stream, peaks, tokens=K2_BW_TOKENS, reps=10, warmup=3):
    """tim_tis_ppo alone on `tokens` tokens (2^27 by default): the segments of
    workloads.draw_ppo_inputs (lognormal lengths, median 1024, clipped to
    [128, 4096]) with the same laws for the other inputs drawn on the device
    (30% masked, l_old = -Gamma(0.6, 3), rollout and current policy as
    N(0, 0.02^2) / N(0, 0.1^2) drifts, per-sequence N(0, 1) advantages);
    token loss and gradient written; L2 flushed before each launch."""
    import torch
    Nt = tokens
    cfg = wl.HeadConfig("ppo", N=Nt, D=8, V=8, seq_layout="lognormal", mask_drop=0.3, seed=9)
    off = wl.draw_segments(cfg)
    S = len(off) - 1
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    torch.manual_seed(9)   # the gamma sampler draws from the default generator
    gamma = torch.distributions.Gamma(torch.tensor(0.6, device=dev), torch.tensor(1.0 / 3.0, device=dev))
    l_old = -gamma.sample((Nt,))
    l_ro = l_old + 0.02 * torch.randn(Nt, device=dev, generator=g)
    l_th = l_old + 0.1 * torch.randn(Nt, device=dev, generator=g)
    mask = (torch.rand(Nt, device=dev, generator=g) >= 0.3).to(torch.uint8)
    offd = torch.from_numpy(off).to(dev)
    lens = offd[1:] - offd[:-1]
    adv = torch.repeat_interleave(torch.randn(S, device=dev, generator=g), lens.long())
    out = {"token_loss": torch.empty(Nt, dtype=torch.float32, device=dev),
           "token_grad": torch.empty(Nt, dtype=torch.float32, device=dev),
           "seq_loss": torch.empty(S, dtype=torch.float32, device=dev),
           "batch": torch.empty(9, dtype=torch.float64, device=dev)}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    call = lambda: tim.tis_ppo(l_th, l_old, l_ro, adv, mask, offd, eps_low=0.2, eps_high=0.28, C=2.0,  # noqa: E731
                               out=out)
    for _ in range(warmup):
        call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        flush.fill_(i)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(reps)]))
    algo = 25 * Nt + 4 * (S + 1) + 4 * S + 72
    gbs = algo / t / 1e9
    tr = measured_traffic("ppo")
    return {"tokens": Nt, "num_seqs": S, "avg_launch_us": t * 1e6, "algorithmic_bytes": algo,
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
            "bound": "hbm", "tokens_per_s": Nt / t,
            "traffic": None if tr is None or Nt != PPO_TRAFFIC_TOKENS else tr,
            "traffic_source": None if tr is None or Nt != PPO_TRAFFIC_TOKENS else TRAFFIC_SOURCE}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-k2-bandwidth", action="store_true")
    ap.add_argument("--skip-sweep", action="store_true")
    ap.add_argument("--skip-heads", action="store_true", help="skip the Llama- and DeepSeek-shaped heads")
    ap.add_argument("--skip-ppo", action="store_true")
    ap.add_argument("--skip-monitor", action="store_true")
    ap.add_argument("--skip-fp32-head", action="store_true")
    ap.add_argument("--skip-backward", action="store_true")
    ap.add_argument("--only", choices=["k1", "k2", "k2bw", "ppo", "monitor", "fp32head", "backward"], default=None,
                    help="time one call alone (for profiling); prints a short line, not the contract line")
    ap.add_argument("--tokens", type=int, default=None,
                    help="smaller batch of the same head (profiling runs only)")
    ap.add_argument("--head", choices=["qwen3_8b", "llama3_8b", "dsv3"], default=WORKLOAD,
                    help="with --only k1: the head shape (profiling runs only)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps, always
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
