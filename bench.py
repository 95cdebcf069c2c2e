"""Benchmark of the fused scaled linear layer on GB300.

Default workload (the decode linear the metric is quoted on): FP8_Dynamic,
K=4096, N=12288, per-token activation and per-channel weight scales, + bias,
SiLU, bf16 out, at every token bucket M in {1, 2, 4, 8, 16, 24, 32}.

One step = one fused call per token bucket on each of NSETS independent
weight sets (7 x NSETS calls).  The sets rotate so that a weight set is
touched again only after more than twice the L2 capacity of other weights
has streamed through; each call therefore reads its weights from HBM.  The
calls of one step are captured once into a CUDA graph per step and replayed.

value = algorithmic HBM bytes of all calls (each tensor once) / device time,
in GB/s, summed over ranks (replicas: the layer does not shard across GPUs
here).  Per-bucket microseconds per call are reported beside it.

``--impl reference`` times the CPU oracle (plain C, float64) on a bounded
sample of the same workload instead.
``--config NAME`` measures another workload (bf16_small, fp8_calls,
w8a8_int8, block_fp8, prefill_bf16, prefill_unfused, and fp8_quant_calls /
int8_quant_calls: bf16 activations quantised per token in the same plan run;
fp8_swiglu_calls: the gated unit of an MLP, W [2 x 12288, 4096];
``--m`` picks token counts) and prints its own line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused scaled-GEMM HBM GB/s (FP8_Dynamic decode linear, K=4096 N=12288, M=1..32)"
NSETS = 6


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="fp8_dynamic")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--m", default=None, help="token counts for --config runs, e.g. 1,16")
    ap.add_argument("--tuning", default=None,
                    help="tuning override for --config runs, JSON, e.g. "
                         '\'{"tile_n":256,"stages":4,"split_k":1,"swap_ab":0,"stream_k":1}\'')
    return ap.parse_args()


# ------------------------------------------------------------ helpers -----

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_aggregate(local_ms: float, local_units: float, dist=None):
    """(max of the timed region over ranks, sum of the work all ranks did).
    Replicas: every rank runs the whole workload on its own GPU; the job's
    throughput is the total work over the slowest rank's time."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(local_ms), float(local_units)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=dev)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        mx = [float(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows)}


# -------------------------------------------------------- native arm ------

def device_problem(p, torch):
    def codes(a, kind):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if kind == "bf16":
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.cuda()
    d = {"A": codes(p.A, p.dtype), "W": codes(p.W, p.dtype)}
    d["s_a"] = None if p.s_a is None else torch.from_numpy(np.ascontiguousarray(p.s_a)).cuda()
    d["s_w"] = None if p.s_w is None else torch.from_numpy(np.ascontiguousarray(p.s_w)).cuda()
    d["bias"] = None if p.bias is None else codes(p.bias, "bf16")
    d["residual"] = None if p.residual is None else codes(p.residual, "bf16")
    d["Y"] = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
    return d


def weight_set(base, seed, torch):
    """Another independent weight set of the same shapes (new seed)."""
    from epilogue_tcgen05_tmem_gb300 import inputs
    q = inputs.make_problem(1, base.N, base.K, base.dtype, base.scale, act=base.act,
                            bias=base.bias is not None, seed=seed)
    W = torch.from_numpy(np.ascontiguousarray(q.W)).cuda() if base.dtype != "bf16" else \
        torch.from_numpy(q.W.view(np.int16)).view(torch.bfloat16).cuda()
    s_w = None if q.s_w is None else torch.from_numpy(np.ascontiguousarray(q.s_w)).cuda()
    b = None if q.bias is None else torch.from_numpy(q.bias.view(np.int16)).view(torch.bfloat16).cuda()
    return W, s_w, b


def run_native(args):
    import torch
    import epilogue_tcgen05_tmem_gb300 as eg
    from epilogue_tcgen05_tmem_gb300 import inputs, traffic

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    eg.lib()
    peaks = measured_peaks()

    # ---- workload: token buckets x weight sets -----------------------------
    base = inputs.workload("fp8_dynamic", 32, seed=0)
    tokens = list(inputs.DECODE_TOKENS)
    Wd = [weight_set(base, 0, torch)] + [weight_set(base, 100 + i, torch) for i in range(NSETS - 1)]
    plans, acts = {}, {}
    for M in tokens:
        p = inputs.take_tokens(base, M)
        plans[M] = eg.Plan(M, p.N, p.K, p.dtype, p.scale, p.act, bias=True, pdl=True)
        d = device_problem(p, torch)
        acts[M] = d
    bytes_per_call = {M: traffic.algorithmic_bytes(M, base.N, base.K, "e4m3", "token_channel",
                                                   bias=True) for M in tokens}
    calls_per_step = len(tokens) * NSETS
    bytes_per_step = sum(bytes_per_call.values()) * NSETS
    weight_bytes = base.N * base.K
    stream = torch.cuda.Stream()

    def enqueue_step(s):
        for j in range(NSETS):
            W, s_w, b = Wd[j]
            for M in tokens:
                d = acts[M]
                plans[M].run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=s.cuda_stream)

    # graph of one step (all buckets x all weight sets, each set visited once)
    with torch.cuda.stream(stream):
        enqueue_step(stream)  # first calls encode descriptors outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue_step(stream)
    torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()

    # ---- timed region -------------------------------------------------------
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    ms, total_bytes = rank_aggregate(e0.elapsed_time(e1), bytes_per_step * args.steps, pg)
    ms_per_step = ms / args.steps
    value = total_bytes / (ms * 1e-3) / 1e9
    avg_launch_us = ms * 1e3 / (args.steps * calls_per_step)
    achieved = (bytes_per_step / calls_per_step) / (avg_launch_us * 1e-6) / 1e9

    # ---- per-bucket microseconds per call (graph of NSETS*R calls) ---------
    per_m = {}
    for M in tokens:
        gm = torch.cuda.CUDAGraph()
        R = 8
        with torch.cuda.graph(gm, stream=stream):
            for _ in range(R):
                for j in range(NSETS):
                    W, s_w, b = Wd[j]
                    d = acts[M]
                    plans[M].run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=stream.cuda_stream)
        for _ in range(3):
            gm.replay()
        torch.cuda.synchronize()
        reps = 20
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                gm.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * R * NSETS)
        per_m[str(M)] = {"us_per_call": round(us, 3),
                         "GB_s": round(bytes_per_call[M] / (us * 1e-6) / 1e9, 1),
                         "hbm_frac": round(bytes_per_call[M] / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                         "tuning": plans[M].tuning}

    # ---- end to end through host buffers -----------------------------------
    e2e = run_e2e(args, torch, eg, plans, acts, Wd, tokens, bytes_per_step, stream)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded SplitMix64 normals; 1% outlier channels x10; e4m3 per-token/per-channel)",
        "config": {"workload": "fp8_dynamic_decode", "M": tokens, "K": base.K, "N": base.N,
                   "epilogue": "scale+bias+SiLU, bf16 out", "weight_sets": NSETS,
                   "calls_per_step": calls_per_step, "bytes_per_step": bytes_per_step,
                   "l2": f"inputs larger than L2: {NSETS} rotating weight sets "
                         f"({NSETS * weight_bytes / 1e6:.0f} MB of weights per step)",
                   "timing": "CUDA events around CUDA-graph replays of whole steps",
                   "parallelism": f"replicas x{world}"},
        "per_m": per_m,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": measured_traffic("fp8_dynamic_decode"), "peak_source": peaks["source"],
                     "kernel": "fused_linear_kernel<e4m3, token_channel, swap_ab>"},
        "e2e": e2e, "gpu_launches": args.steps * calls_per_step, "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(base)
    for pl in plans.values():
        pl.close()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


def kernel_source_sha256():
    """Hash of the fused kernel's device sources: a stored ncu traffic figure
    holds only for the kernel it was captured on."""
    import hashlib
    h = hashlib.sha256()
    for f in ("eg_kernel.cuh", "eg_ptx.cuh"):
        with open(os.path.join(ROOT, "epilogue_tcgen05_tmem_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(key):
    """DRAM bytes (read + write) per launch from the committed ncu summary of
    this kernel, or None when there is none or the kernel has changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_sha256") != kernel_source_sha256():
        return None
    return rec["dram_bytes_per_launch"]


def run_e2e(args, torch, eg, plans, acts, Wd, tokens, bytes_per_step, stream):
    """Same metric through the C ABI with host buffers: every call copies its
    activations (A, s_a) from pinned host memory and reads Y back."""
    host = {}
    for M in tokens:
        d = acts[M]
        host[M] = {"A": d["A"].cpu().pin_memory(), "s_a": d["s_a"].cpu().pin_memory(),
                   "Y": torch.empty(d["Y"].shape, dtype=torch.bfloat16).pin_memory()}
    steps = args.e2e_steps or max(3, min(args.steps, 50))
    h2d = sum(host[M]["A"].numel() + 4 * host[M]["s_a"].numel() for M in tokens) * NSETS
    d2h = sum(host[M]["Y"].numel() * 2 for M in tokens) * NSETS

    def one_step():
        for j in range(NSETS):
            W, s_w, b = Wd[j]
            for M in tokens:
                d, h = acts[M], host[M]
                d["A"].copy_(h["A"], non_blocking=True)
                d["s_a"].copy_(h["s_a"], non_blocking=True)
                plans[M].run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=stream.cuda_stream)
                h["Y"].copy_(d["Y"], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            one_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            one_step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": round(bytes_per_step * steps / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4)}


# ----------------------------------------------------------- CPU oracle ----

def oracle_sample(base, n_cols):
    """The decode workload restricted to the first n_cols output channels, at
    every token bucket (the oracle as it stands, all host cores)."""
    import oracle
    from epilogue_tcgen05_tmem_gb300 import inputs, traffic
    sub = inputs.Problem(base.M, n_cols, base.K, base.dtype, base.scale, base.act,
                         base.bias[:n_cols], None, base.A, np.ascontiguousarray(base.W[:n_cols]),
                         base.s_a, np.ascontiguousarray(base.s_w[:n_cols]))
    probs = [inputs.take_tokens(sub, M) for M in inputs.DECODE_TOKENS]
    nbytes = sum(traffic.problem_bytes(q) for q in probs)
    t0 = time.perf_counter()
    for q in probs:
        oracle.linear(q)
    return nbytes, time.perf_counter() - t0


def cpu_baseline(base, target_s=10.0):
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    nbytes, dt = oracle_sample(base, 256)
    n = int(min(base.N, max(256, 256 * target_s / max(dt, 1e-3))))
    n = max(256, (n // 256) * 256)
    # the whole sample, repeated until about target_s seconds of CPU work
    total_b, total_t, reps = 0, 0.0, 0
    while total_t < target_s or reps == 0:
        b, t = oracle_sample(base, n)
        total_b, total_t, reps = total_b + b, total_t + t, reps + 1
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"all 7 token buckets (M=1..32) over the first {n} of {base.N} output "
                      f"channels, one weight set, {reps} passes; {total_t:.2f} s",
            "seconds": round(total_t, 3)}


def run_reference(args):
    """Reference arm: the CPU oracle timed on the machine's host cores, each step a
    bounded sample of the same workload."""
    import oracle
    from epilogue_tcgen05_tmem_gb300 import inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return
    oracle.build()
    base = inputs.workload("fp8_dynamic", 32, seed=0)
    cores = oracle.default_threads()
    _, dt = oracle_sample(base, 128)
    per_col = dt / 128
    budget = 120.0  # seconds for all timed steps
    n = int(budget / max(args.steps, 1) / max(per_col, 1e-9))
    n = max(8, min(base.N, (n // 8) * 8))
    for _ in range(args.warmup if args.warmup < 3 else 3):
        oracle_sample(base, n)
    total_b, total_t = 0, 0.0
    for _ in range(args.steps):
        b, t = oracle_sample(base, n)
        total_b += b
        total_t += t
    v = total_b / total_t / 1e9
    sample = (f"each step: all 7 token buckets (M=1..32) over the first {n} of {base.N} "
              f"output channels")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_t * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "fp8_dynamic_decode", "K": base.K, "N": base.N,
                   "M": list(inputs.DECODE_TOKENS)},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------ other workloads ----

def run_config(args):
    """One line for another workload (for the measurement tables)."""
    import torch
    import epilogue_tcgen05_tmem_gb300 as eg
    from epilogue_tcgen05_tmem_gb300 import inputs, traffic
    torch.cuda.set_device(dist_env()[2])
    eg.lib()
    peaks = measured_peaks()
    name = args.config
    unfused = name == "prefill_unfused"
    # quantisation prologue: bf16 activations in, per-token quantisation
    # and the GEMM in one plan run
    quant = name in ("fp8_quant_calls", "int8_quant_calls")
    # gated unit (SwiGLU) of an MLP with hidden 4096 and intermediate 12288:
    # W [2 x 12288, 4096] FP8, per-token / per-channel scales
    gated = name == "fp8_swiglu_calls"
    wl = {"prefill_unfused": "prefill_bf16", "fp8_quant_calls": "fp8_calls",
          "int8_quant_calls": "w8a8_int8", "fp8_swiglu_calls": "fp8_calls"}.get(name, name)
    Ms = [None]
    if wl in ("w8a8_int8", "fp8_calls"):
        Ms = list(inputs.DECODE_TOKENS)
    elif wl == "block_fp8":
        Ms = [1, 8, 32, 2048]
    if args.m:
        Ms = [int(x) for x in args.m.split(",")]
    if wl == "fp8_calls":
        wl = "fp8_dynamic"
    rows = []
    for M in Ms:
        if gated:
            p = inputs.make_gated_problem(M, 12288, 4096, "e4m3", "token_channel", act="silu",
                                          outlier_frac=0.01)
        else:
            p = inputs.workload(wl, M)
        d = device_problem(p, torch)
        plan = eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=p.bias is not None,
                       residual=p.residual is not None, residual_pre_act=p.residual_pre_act,
                       pdl=not unfused, quant_a=quant, gated=gated,
                       tuning=json.loads(args.tuning) if args.tuning else None)
        nb = traffic.problem_bytes(p)
        if gated:
            # two weight halves and their scales; the output is N wide
            nb += p.N * p.K + p.N * 4
        if quant:
            # the layer reads bf16 activations instead of codes and scales
            X = torch.from_numpy(inputs.activations_bf16(p.M, p.K, outlier_frac=0.01)).view(
                torch.bfloat16).cuda()
            nb += p.M * p.K * 2 - p.M * p.K - p.M * 4
            d["A"], d["s_a"] = X, None
        fl = traffic.flops(p.M, p.N, p.K)
        # rotate weight copies so repeated calls do not hit L2
        nw = max(1, math.ceil(2 * 129e6 / max(p.W.nbytes, 1)) + 1)
        Ws = [d["W"]] + [d["W"].clone() for _ in range(min(nw, 8) - 1)]
        T1 = T2 = None
        if unfused:
            T1 = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
            T2 = torch.empty_like(T1)

        def call(W):
            if unfused:
                plan.run_unfused(d["A"], W, d["Y"], T1, T2, d["s_a"], d["s_w"], d["bias"],
                                 d["residual"])
            else:
                plan.run(d["A"], W, d["Y"], d["s_a"], d["s_w"], d["bias"], d["residual"])
        for i in range(max(args.warmup, 3)):
            call(Ws[i % len(Ws)])
        torch.cuda.synchronize()
        reps = max(args.steps, 10)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            call(Ws[i % len(Ws)])
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        # SM clocks and throttle reasons under this load: about 0.6 s more of
        # the same calls, sampled by nvidia-smi
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        time.sleep(0.15)
        for i in range(max(1, int(0.6e6 / max(us, 1e-3)))):
            call(Ws[i % len(Ws)])
        torch.cuda.synchronize()
        clocks = sampler.stop()
        tf = fl / (us * 1e-6) / 1e12
        gbs = nb / (us * 1e-6) / 1e9
        peak_tf = peaks["bf16_tflops"] * (2 if p.dtype == "e4m3" else 1)
        rows.append({"M": p.M, "N": p.N, "K": p.K, "us_per_call": round(us, 3),
                     "TFLOP_s": round(tf, 2), "GB_s": round(gbs, 1),
                     "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                     "tensor_frac": round(tf / peak_tf, 4), "tuning": plan.tuning,
                     "clocks": clocks})
        plan.close()
        del d, Ws
        torch.cuda.empty_cache()
    print(json.dumps({"config": name, "rows": rows, "peaks": peaks}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.config != "fp8_dynamic":
        run_config(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
