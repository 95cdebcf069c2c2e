"""Benchmark of the fused scaled linear layer on GB300.

Default workload (the decode linear the metric is quoted on): FP8_Dynamic,
K=4096, N=12288, per-token activation and per-channel weight scales, + bias,
SiLU, bf16 out, at every token bucket M in {1, 2, 4, 8, 16, 24, 32}.

One step = one fused call per token bucket on each of NSETS independent
weight sets (7 x NSETS calls), bucket by bucket with the weight set changing
on every call, so a set is read again only after the other NSETS - 1 sets
(more than twice the L2 capacity) have streamed through: every call reads
its weights from HBM.  The calls of one step are captured once into a CUDA
graph and replayed; each call is a programmatic dependent of the previous
one.  The timed region (exactly --steps replays) is cut into at least 10
repeats whose median is reported beside the whole-region value.

value = algorithmic HBM bytes of all calls (each tensor once) / device time,
in GB/s, summed over ranks (replicas: the layer does not shard across GPUs
here).  Per token bucket the line also carries the pipelined interval
between back-to-back calls and the isolated latency of one call (a graph
holding one call, after an L2 flush).  The same run measures the other
configurations (W8A8_INT8 and Block_FP8 decode, FP8_Dynamic and Block_FP8
at 2048 tokens, the bf16 4096^3 prefill fused and unfused) under "configs",
each with its SM clocks.

``--impl reference`` times the CPU oracle (plain C, float64) on a bounded
sample of the same workload instead.
``--config NAME`` measures another workload (bf16_small, fp8_calls,
w8a8_int8, block_fp8, prefill_bf16, prefill_unfused, and fp8_quant_calls /
int8_quant_calls: bf16 activations quantised per token in the same plan run;
fp8_swiglu_calls: the gated unit of an MLP, W [2 x 12288, 4096];
``--m`` picks token counts) and prints its own line.
``--trace-timeline`` prints the per-call device timeline of one replayed
step (first CTA start, first TMA, last CTA end of every call).
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
NSETS = 7


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="fp8_dynamic")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--repeats", type=int, default=10,
                    help="repeats the timed region is cut into (at least 10)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the default workload (no other configurations)")
    ap.add_argument("--trace-timeline", action="store_true")
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


def l2_bytes(torch):
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 1024 * 1024


def time_graph(torch, enqueue, stream, repeats=10, warmup=3):
    """Capture enqueue(stream) into one CUDA graph and time `repeats`
    replays of it with CUDA events on `stream`: per-replay milliseconds."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue(stream)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(repeats + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(repeats):
            g.replay()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    del g
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(repeats)]


def time_isolated(torch, enqueue, stream, flush, repeats=30):
    """Latency of one call on its own: a graph holding that one call,
    replayed after a write of more than twice the L2 capacity (so neither
    its weights nor its predecessor's work are in L2, and no call of the
    same layer runs before it); events around the replay only.  Median
    microseconds."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue(stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(repeats)]
    with torch.cuda.stream(stream):
        for e0, e1 in pairs:
            flush.zero_()
            e0.record(stream)
            g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    del g
    return statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in pairs)


def clocks_during(torch, loop_fn, seconds=0.6):
    """nvidia-smi SM clocks and throttle reasons while loop_fn() runs
    repeatedly for about `seconds`."""
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.15)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        loop_fn()
        torch.cuda.synchronize()
    return sampler.stop()


def weight_copies(W, n, torch):
    """n device copies of a weight tensor (the first is W itself)."""
    return [W] + [W.clone() for _ in range(n - 1)]


def rotate_count(weight_bytes, l2):
    """Weight copies for a rotation in which a copy is read again only after
    more than twice the L2 capacity of other weights went through."""
    return max(2, math.ceil(2 * l2 / max(weight_bytes, 1)) + 1)


def decode_rows(torch, eg, inputs, traffic, base, tokens, peaks, stream, flush, l2):
    """Per token bucket of one decode workload (`base` holds its largest
    token count): the pipelined interval (a graph of back-to-back calls, the
    weight copy changing on every call, each call a programmatic dependent
    of the previous one), the isolated latency of one call, GB/s and the
    fraction of the HBM roofline for both, and the SM clocks under the
    first bucket's load."""
    d0 = device_problem(base, torch)
    nw = rotate_count(d0["W"].numel() * d0["W"].element_size(), l2)
    Ws = weight_copies(d0["W"], nw, torch)
    rows, clocks = {}, None
    for M in tokens:
        p = inputs.take_tokens(base, M)
        d = device_problem(p, torch)
        plan = eg.Plan(M, p.N, p.K, p.dtype, p.scale, p.act, bias=p.bias is not None,
                       residual=p.residual is not None, pdl=True)
        nb = traffic.problem_bytes(p)

        def call(W, s, d=d, plan=plan):
            plan.run(d["A"], W, d["Y"], d["s_a"], d0["s_w"], d0["bias"], d["residual"],
                     stream=s.cuda_stream)
        with torch.cuda.stream(stream):
            call(Ws[0], stream)
        torch.cuda.synchronize()
        R = 4 * nw
        ms = time_graph(torch, lambda s: [call(Ws[i % nw], s) for i in range(R)], stream)
        us = statistics.median(ms) * 1e3 / R
        iso = time_isolated(torch, lambda s: call(Ws[1], s), stream, flush)
        if clocks is None:
            def loop():
                with torch.cuda.stream(stream):
                    for i in range(R):
                        call(Ws[i % nw], stream)
            clocks = clocks_during(torch, loop)
        gbs = nb / (us * 1e-6) / 1e9
        rows[str(M)] = {"us_per_call": round(us, 3), "GB_s": round(gbs, 1),
                        "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                        "isolated_us": round(iso, 3),
                        "isolated_hbm_frac": round(nb / (iso * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                        "tuning": plan.tuning}
        plan.close()
        del d
    del Ws, d0
    return rows, clocks


def large_m_row(torch, eg, traffic, p, peaks, stream, l2, unfused=False):
    """One tensor-bound call (2048 tokens, or the 4096^3 prefill): median of
    10 timed graphs of 10 back-to-back calls over rotated input copies (A, W
    and the residual: a copy is read again only after more than the L2
    capacity of other data); TFLOP/s against the dtype's dense peak (E4M3:
    twice the measured bf16 figure, the nominal ratio).  With unfused, the
    same problem through the three-kernel path too."""
    d = device_problem(p, torch)
    plan = eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=p.bias is not None,
                   residual=p.residual is not None, residual_pre_act=p.residual_pre_act, pdl=True)
    nb = traffic.problem_bytes(p)
    fl = traffic.flops(p.M, p.N, p.K)
    nsets = 2 if nb > 2 * l2 else 3
    sets = [(d["A"], d["W"], d["residual"])]
    for _ in range(nsets - 1):
        sets.append((d["A"].clone(), d["W"].clone(),
                     None if d["residual"] is None else d["residual"].clone()))

    def call(i, s):
        A, W, R = sets[i % nsets]
        plan.run(A, W, d["Y"], d["s_a"], d["s_w"], d["bias"], R, stream=s.cuda_stream)
    with torch.cuda.stream(stream):
        call(0, stream)
    torch.cuda.synchronize()
    R = 10
    ms = time_graph(torch, lambda s: [call(i, s) for i in range(R)], stream)
    us = statistics.median(ms) * 1e3 / R
    peak_tf = peaks["bf16_tflops"] * (2 if p.dtype == "e4m3" else 1)
    tf = fl / (us * 1e-6) / 1e12
    row = {"M": p.M, "N": p.N, "K": p.K, "us_per_call": round(us, 3), "TFLOP_s": round(tf, 1),
           "tensor_frac": round(tf / peak_tf, 4), "peak_TFLOP_s": round(peak_tf, 1),
           "peak_source": peaks["source"] + (" bf16 x 2" if p.dtype == "e4m3" else " bf16 burst"),
           "GB_s": round(nb / (us * 1e-6) / 1e9, 1), "tuning": plan.tuning,
           "repeats_us_per_call": [round(x * 1e3 / R, 2) for x in ms]}

    def loop():
        with torch.cuda.stream(stream):
            for i in range(R):
                call(i, stream)
    row["clocks"] = clocks_during(torch, loop)
    if unfused:
        T1 = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
        T2 = torch.empty_like(T1)
        uplan = eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=p.bias is not None,
                        residual=p.residual is not None, residual_pre_act=p.residual_pre_act)

        def ucall(i, s):
            A, W, Rr = sets[i % nsets]
            uplan.run_unfused(A, W, d["Y"], T1, T2, d["s_a"], d["s_w"], d["bias"], Rr,
                              stream=s.cuda_stream)
        with torch.cuda.stream(stream):
            ucall(0, stream)
        torch.cuda.synchronize()
        ums = time_graph(torch, lambda s: [ucall(i, s) for i in range(R)], stream)
        uus = statistics.median(ums) * 1e3 / R
        row["unfused"] = {"us_per_call": round(uus, 3), "kernels_per_call": 3,
                          "extra_bytes": traffic.unfused_extra_bytes(p.M, p.N),
                          "fused_saves_us": round(uus - us, 3),
                          "fused_speedup": round(uus / us, 4)}
        uplan.close()
    plan.close()
    del sets, d
    return row


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
    l2 = l2_bytes(torch)

    # ---- workload: token buckets x weight sets -----------------------------
    base = inputs.workload("fp8_dynamic", 32, seed=0)
    tokens = list(inputs.DECODE_TOKENS)
    Wd = [weight_set(base, 0, torch)] + [weight_set(base, 100 + i, torch) for i in range(NSETS - 1)]
    plans, acts = {}, {}
    for M in tokens:
        p = inputs.take_tokens(base, M)
        plans[M] = eg.Plan(M, p.N, p.K, p.dtype, p.scale, p.act, bias=True, pdl=True)
        acts[M] = device_problem(p, torch)
    bytes_per_call = {M: traffic.algorithmic_bytes(M, base.N, base.K, "e4m3", "token_channel",
                                                   bias=True) for M in tokens}
    # the weight set changes on every call: bucket by bucket, each bucket
    # over all NSETS sets, so a set is read again only after the other
    # NSETS - 1 sets (more than twice the L2 capacity) went through
    order = [(M, j) for M in tokens for j in range(NSETS)]
    calls_per_step = len(order)
    bytes_per_step = sum(bytes_per_call[M] for M, _ in order)
    weight_bytes = base.N * base.K
    assert (NSETS - 1) * weight_bytes > 2 * l2 or l2 > 200e6
    stream = torch.cuda.Stream()

    def enqueue_step(s):
        for M, j in order:
            W, s_w, b = Wd[j]
            d = acts[M]
            plans[M].run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=s.cuda_stream)

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

    # ---- timed region: exactly `steps` replays, cut into >= 10 repeats ------
    n_rep = min(args.steps, max(10, args.repeats))
    bounds = [args.steps * i // n_rep for i in range(n_rep + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for r in range(n_rep):
            for _ in range(bounds[r + 1] - bounds[r]):
                g.replay()
            ev[r + 1].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    local_ms = ev[0].elapsed_time(ev[-1])
    rep_ms = [ev[r].elapsed_time(ev[r + 1]) / (bounds[r + 1] - bounds[r]) for r in range(n_rep)]
    ms, total_bytes = rank_aggregate(local_ms, bytes_per_step * args.steps, pg)
    ms_per_step = ms / args.steps
    value = total_bytes / (ms * 1e-3) / 1e9
    avg_launch_us = ms * 1e3 / (args.steps * calls_per_step)
    achieved = (bytes_per_step / calls_per_step) / (avg_launch_us * 1e-6) / 1e9
    del g

    # ---- per bucket: pipelined interval and isolated latency ----------------
    flush = torch.empty(int(2.2 * l2), dtype=torch.uint8, device="cuda")
    per_m = {}
    for M in tokens:
        d = acts[M]

        def call(j, s, M=M, d=d):
            W, s_w, b = Wd[j]
            plans[M].run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=s.cuda_stream)
        R = 4
        msr = time_graph(torch, lambda s: [call(j, s) for _ in range(R) for j in range(NSETS)],
                         stream)
        us = statistics.median(msr) * 1e3 / (R * NSETS)
        iso = time_isolated(torch, lambda s: call(1, s), stream, flush)
        per_m[str(M)] = {"us_per_call": round(us, 3),
                         "GB_s": round(bytes_per_call[M] / (us * 1e-6) / 1e9, 1),
                         "hbm_frac": round(bytes_per_call[M] / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                         "isolated_us": round(iso, 3),
                         "isolated_hbm_frac": round(
                             bytes_per_call[M] / (iso * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                         "tuning": plans[M].tuning}

    # ---- end to end through host buffers -----------------------------------
    e2e = run_e2e(args, torch, eg, plans, acts, Wd, order, bytes_per_step, stream)
    for pl in plans.values():
        pl.close()
    del Wd, acts
    torch.cuda.empty_cache()

    # ---- the other configurations, under the same clock ---------------------
    configs = {}
    if not args.no_configs:
        configs = other_configs(torch, eg, inputs, traffic, peaks, stream, flush, l2)
    del flush
    torch.cuda.empty_cache()

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded SplitMix64 normals; 1% outlier channels x10; e4m3 per-token/per-channel)",
        "config": {"workload": "fp8_dynamic_decode", "M": tokens, "K": base.K, "N": base.N,
                   "epilogue": "scale+bias+SiLU, bf16 out", "weight_sets": NSETS,
                   "call_order": "bucket by bucket, the weight set changing on every call",
                   "calls_per_step": calls_per_step, "bytes_per_step": bytes_per_step,
                   "l2": f"inputs larger than L2: {NSETS} rotating weight sets "
                         f"({NSETS * weight_bytes / 1e6:.0f} MB of weights per step); a set is "
                         f"read again after {(NSETS - 1) * weight_bytes / 1e6:.0f} MB of other "
                         f"weights (L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA events around CUDA-graph replays of whole steps; each call "
                             "a programmatic dependent of the previous one",
                   "parallelism": f"replicas x{world}"},
        "repeats": {"n": n_rep, "ms_per_step_median": round(statistics.median(rep_ms), 5),
                    "ms_per_step_min": round(min(rep_ms), 5),
                    "ms_per_step_max": round(max(rep_ms), 5),
                    "value_median": round(bytes_per_step / (statistics.median(rep_ms) * 1e-3) / 1e9, 2)},
        "per_m": per_m,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": measured_traffic("fp8_dynamic_decode"), "peak_source": peaks["source"],
                     "kernel": "fused_linear_kernel<e4m3, token_channel, swap_ab>",
                     "launch_duration": "timed region / launches (back-to-back calls overlap "
                                        "through programmatic dependent launch)"},
        "configs": configs,
        "e2e": e2e, "gpu_launches": args.steps * calls_per_step, "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(base)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


def other_configs(torch, eg, inputs, traffic, peaks, stream, flush, l2):
    """The other workloads of the measurement table, timed in the same run:
    W8A8_INT8 and Block_FP8 decode per token bucket (pipelined and
    isolated), FP8_Dynamic and Block_FP8 at 2048 tokens, and the bf16
    4096^3 prefill block fused and through the unfused three-kernel path."""
    cfg = {}
    base = inputs.workload("w8a8_int8", 32)
    rows, clocks = decode_rows(torch, eg, inputs, traffic, base, list(inputs.DECODE_TOKENS),
                               peaks, stream, flush, l2)
    cfg["w8a8_int8_decode"] = {"K": base.K, "N": base.N, "epilogue": "scale + bf16 residual",
                               "per_m": rows, "clocks": clocks}
    del base
    torch.cuda.empty_cache()
    # Block_FP8: the 2048-token problem; its first 1, 8 and 32 tokens are
    # the decode problems (per-token data is row-local)
    big = inputs.workload("block_fp8", 2048)
    rows, clocks = decode_rows(torch, eg, inputs, traffic, inputs.take_tokens(big, 32), [1, 8, 32],
                               peaks, stream, flush, l2)
    cfg["block_fp8_decode"] = {"K": big.K, "N": big.N, "per_m": rows, "clocks": clocks}
    torch.cuda.empty_cache()
    cfg["block_fp8_m2048"] = large_m_row(torch, eg, traffic, big, peaks, stream, l2)
    del big
    torch.cuda.empty_cache()
    cfg["fp8_dynamic_m2048"] = large_m_row(torch, eg, traffic, inputs.workload("fp8_dynamic", 2048),
                                           peaks, stream, l2)
    torch.cuda.empty_cache()
    cfg["prefill_bf16_4096"] = large_m_row(torch, eg, traffic, inputs.workload("prefill_bf16"),
                                           peaks, stream, l2, unfused=True)
    torch.cuda.empty_cache()
    return cfg


def run_trace_timeline(args):
    """Per-call timeline of one replay of the default step (every call with
    its own plan and trace buffer): for each call, the first CTA start, the
    first TMA issued after its wait on the previous kernel, and the last CTA
    end, relative to the step's first CTA start.  Prints one JSON line."""
    import torch
    import epilogue_tcgen05_tmem_gb300 as eg
    from epilogue_tcgen05_tmem_gb300 import inputs

    torch.cuda.set_device(dist_env()[2])
    eg.lib()
    base = inputs.workload("fp8_dynamic", 32, seed=0)
    tokens = list(inputs.DECODE_TOKENS)
    Wd = [weight_set(base, 0, torch)] + [weight_set(base, 100 + i, torch) for i in range(NSETS - 1)]
    acts = {M: device_problem(inputs.take_tokens(base, M), torch) for M in tokens}
    order = [(M, j) for M in tokens for j in range(NSETS)]
    calls = []
    for M, j in order:
        pl = eg.Plan(M, base.N, base.K, "e4m3", "token_channel", "silu", bias=True, pdl=True)
        ctas = pl.launch_info["grid"]
        buf = torch.zeros(ctas, eg.EG_TRACE_POINTS, dtype=torch.int64, device="cuda")
        pl.set_trace(buf)
        calls.append((M, j, pl, buf))
    stream = torch.cuda.Stream()

    def enqueue(s):
        for M, j, pl, _ in calls:
            W, s_w, b = Wd[j]
            d = acts[M]
            pl.run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=s.cuda_stream)
    with torch.cuda.stream(stream):
        enqueue(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue(stream)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    for _, _, _, buf in calls:
        buf.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    step_ms = e0.elapsed_time(e1)
    tr = [buf.cpu().numpy() for _, _, _, buf in calls]
    t0 = min(int(t[:, 0][t[:, 0] > 0].min()) for t in tr)
    from epilogue_tcgen05_tmem_gb300 import trace as trace_mod
    rows = []
    prev_end = None
    detail = {}
    for i in (0, 1, len(calls) // 2, len(calls) - 1):
        M, j = calls[i][0], calls[i][1]
        detail[f"call{i}_M{M}_set{j}"] = trace_mod.summarize(tr[i], t0)
    for (M, j, pl, _), t in zip(calls, tr):
        st = t[:, 0][t[:, 0] > 0]
        ft = t[:, 2][t[:, 2] > 0]
        en = t[:, 7][t[:, 7] > 0]
        r = {"M": M, "set": j, "ctas": int(st.size),
             "start_us": round((int(st.min()) - t0) / 1e3, 3),
             "first_tma_us": round((int(ft.min()) - t0) / 1e3, 3) if ft.size else None,
             "end_us": round((int(en.max()) - t0) / 1e3, 3)}
        r["span_us"] = round(r["end_us"] - r["start_us"], 3)
        r["overlap_prev_us"] = None if prev_end is None else round(prev_end - r["start_us"], 3)
        prev_end = r["end_us"]
        rows.append(r)
    # isolated calls: one call per graph replay after an L2 flush, traced
    flush = torch.empty(int(2.2 * l2_bytes(torch)), dtype=torch.uint8, device="cuda")
    iso = {}
    for i in (0, len(calls) - 1):
        M, j, pl, buf = calls[i]
        W, s_w, b = Wd[j]
        d = acts[M]
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi, stream=stream):
            pl.run(d["A"], W, d["Y"], d["s_a"], s_w, b, None, stream=stream.cuda_stream)
        for _ in range(3):
            gi.replay()
        torch.cuda.synchronize()
        buf.zero_()
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            gi.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t = buf.cpu().numpy()
        st, en = t[:, 0][t[:, 0] > 0], t[:, 7][t[:, 7] > 0]
        # the split-K last arrivers' reduction and store (store_begin ->
        # epilogue done) and everyone else's arrival -> epilogue done
        last = t[:, 14] > 0
        red = (t[last, 6] - t[last, 14]) / 1e3
        red_only = (t[last & (t[:, 13] > 0), 13] - t[last & (t[:, 13] > 0), 14]) / 1e3
        rest = (t[~last & (t[:, 12] > 0), 6] - t[~last & (t[:, 12] > 0), 12]) / 1e3
        iso[f"M{M}_set{j}"] = {"event_us": round(e0.elapsed_time(e1) * 1e3, 3),
                               "trace_span_us": round((int(en.max()) - int(st.min())) / 1e3, 3),
                               "last_arriver_reduce_store_us": [round(float(np.percentile(red, q)), 3)
                                                                for q in (0, 50, 90, 100)] if red.size else None,
                               "last_arriver_reduce_first_chunk_us": [round(float(np.percentile(red_only, q)), 3)
                                                                      for q in (0, 50, 90, 100)] if red_only.size else None,
                               "others_arrived_to_done_us": [round(float(np.percentile(rest, q)), 3)
                                                             for q in (0, 50, 90, 100)] if rest.size else None,
                               "points": trace_mod.summarize(t)}
        del gi
    for _, _, pl, _ in calls:
        pl.close()
    spans = [r["span_us"] for r in rows]
    print(json.dumps({"trace": "fp8_dynamic_decode step", "calls": len(rows),
                      "step_ms_events": round(step_ms, 4),
                      "step_us_trace": round(rows[-1]["end_us"] - rows[0]["start_us"], 3),
                      "sum_of_spans_us": round(sum(spans), 3),
                      "mean_interval_us": round((rows[-1]["end_us"] - rows[0]["start_us"]) / len(rows), 3),
                      "points": detail, "isolated": iso, "rows": rows}), flush=True)


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


def run_e2e(args, torch, eg, plans, acts, Wd, order, bytes_per_step, stream):
    """Same metric through the C ABI with host buffers.  Every step copies the
    activations (A, s_a) of all its calls from pinned host memory to the
    device in one transfer and reads all of its outputs Y back in one
    transfer.  The copies run on two copy streams: a step's inputs go up
    while the previous step computes and its outputs come down while the
    next one computes (two device buffer sets alternate).  Two steps are
    captured into one CUDA graph with the copies and the cross-stream waits;
    the timed region covers every copy and every GEMM of every step."""
    def r256(n):
        return (n + 255) // 256 * 256

    offs, na, ny = [], 0, 0
    for M, _ in order:
        a_bytes = acts[M]["A"].numel() * acts[M]["A"].element_size()
        s_off = na + r256(a_bytes)
        offs.append((na, s_off, ny))
        na = s_off + r256(4 * M)
        ny += r256(acts[M]["Y"].numel() * 2)
    h_in = torch.empty(na, dtype=torch.uint8).pin_memory()
    for (a_off, s_off, _), (M, _) in zip(offs, order):
        a = acts[M]["A"].contiguous().view(torch.uint8).reshape(-1).cpu()
        h_in[a_off:a_off + a.numel()].copy_(a)
        s = acts[M]["s_a"].contiguous().view(torch.uint8).reshape(-1).cpu()
        h_in[s_off:s_off + s.numel()].copy_(s)
    d_in = [torch.empty(na, dtype=torch.uint8, device="cuda") for _ in range(2)]
    d_out = [torch.empty(ny, dtype=torch.uint8, device="cuda") for _ in range(2)]
    h_out = [torch.empty(ny, dtype=torch.uint8).pin_memory() for _ in range(2)]
    h2d = sum(acts[M]["A"].numel() * acts[M]["A"].element_size() + 4 * M for M, _ in order)
    d2h = sum(acts[M]["Y"].numel() * 2 for M, _ in order)
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def views(b, c, M):
        a_off, s_off, y_off = offs[c]
        d = acts[M]
        A = d_in[b][a_off:a_off + d["A"].numel() * d["A"].element_size()].view(d["A"].dtype).view(d["A"].shape)
        s_a = d_in[b][s_off:s_off + 4 * M].view(torch.float32)
        Y = d_out[b][y_off:y_off + d["Y"].numel() * 2].view(torch.bfloat16).view(d["Y"].shape)
        return A, s_a, Y

    def two_steps(s):
        # inputs of both steps go up first (the second step's while the first computes)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        up.wait_stream(s)
        with torch.cuda.stream(up):
            for b in range(2):
                d_in[b].copy_(h_in, non_blocking=True)
                ev_in[b].record(up)
        for b in range(2):
            s.wait_event(ev_in[b])
            for c, (M, j) in enumerate(order):
                W, s_w, bias = Wd[j]
                A, s_a, Y = views(b, c, M)
                plans[M].run(A, W, Y, s_a, s_w, bias, None, stream=s.cuda_stream)
            # this step's outputs come down while the next one computes
            down.wait_stream(s)
            with torch.cuda.stream(down):
                h_out[b].copy_(d_out[b], non_blocking=True)
        s.wait_stream(down)
        s.wait_stream(up)

    pairs = max(2, ((args.e2e_steps or max(3, min(args.steps, 50))) + 1) // 2)
    msr = time_graph(torch, two_steps, stream, repeats=pairs, warmup=2)
    ms = sum(msr)
    steps = 2 * pairs
    # the outputs read back equal the device results of a plain run
    for c, (M, j) in enumerate(order[:1]):
        _, _, Y = views(1, c, M)
        y_off = offs[c][2]
        host = h_out[1][y_off:y_off + Y.numel() * 2].view(torch.bfloat16).view(Y.shape)
        assert torch.equal(host.view(torch.int16), Y.cpu().view(torch.int16))
    return {"value": round(bytes_per_step * steps / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "copies": "one host-to-device transfer of the step's activations and one "
                      "device-to-host transfer of its outputs, pinned host memory, on their own "
                      "streams overlapping the neighbouring step's GEMMs; two steps per CUDA graph"}


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
    elif args.trace_timeline:
        run_trace_timeline(args)
    elif args.config != "fp8_dynamic":
        run_config(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
