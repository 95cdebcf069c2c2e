"""Offline per-shape sweep of the fused kernel's tuning space.

For one problem shape and each token bucket it times every valid
(tile_n, stages, split_k, swap_ab, ...) point under CUDA-graph replay, over
enough rotating weight copies that the weights stream from HBM, and keeps
the fastest (ties within 1% go to the plain split over the balanced one, then the
smaller split_k, then no swap, then fewer stages).  The rows it prints (or writes with --out) are the format of
``csrc/eg_tuning_table.inc``; the library consults that table before its
default rule.

Rows are keyed by the epilogue class too (plain, gated unit, behind the
quantisation prologue: workloads fp8_swiglu, fp8_quant, int8_quant).

This is the offline autotuning step of "Helion linear backend in vLLM"
(sections "One kernel instead of three" and "How the autotuner searches":
split_k over powers of two up to 256 and swap_ab as tunables of one kernel;
benchmarking under CUDA graphs; one tuned configuration per token bucket
1, 2, 4, 8, 16, 24, 32).  The space here is small, so it is searched
exhaustively.

    python -m epilogue_tcgen05_tmem_gb300.sweep --workload fp8_dynamic --out rows.inc
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

TILE_N = (16, 32, 64, 128, 256)
SPLITS = (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 64)
L2_BYTES = 129 * 2 ** 20


def candidates(p, swaps=(0, 1)):
    # block scales: tiles up to 128 wide, and 256 wide with rows over M
    max_bn = 64 if p.dtype == "int8" else 256
    elems = 64 if p.dtype == "bf16" else 128
    k_tiles = -(-p.K // elems)
    if p.M > 32:
        yield from _midrange_candidates(p, swaps, max_bn, k_tiles)
        return
    for swap in swaps:
        cols = p.M if swap else p.N
        for bn in TILE_N:
            if bn > max_bn:
                continue
            if bn > 16 and bn // 2 >= cols:          # a smaller tile already covers cols
                continue
            if p.scale == "block" and bn > 128 and swap:
                continue
            for stages in (2, 3, 4, 6, 8):
                for s in SPLITS:
                    if s > k_tiles or (s > 1 and k_tiles // s < 2):
                        continue
                    yield dict(tile_n=bn, stages=stages, split_k=s, swap_ab=swap, stream_k=0,
                               cluster_reduce=0, cta_pair=0)
                    # the same split reduced inside a cluster (2, 4 or 8 CTAs)
                    if s in (2, 4, 8):
                        yield dict(tile_n=bn, stages=stages, split_k=s, swap_ab=swap, stream_k=0,
                                   cluster_reduce=1, cta_pair=0)
                # balanced split-K with 1 or 2 CTAs per SM
                for sk in (1, 2):
                    yield dict(tile_n=bn, stages=stages, split_k=1, swap_ab=swap, stream_k=sk,
                               cluster_reduce=0, cta_pair=0)


def _midrange_candidates(p, swaps, max_bn, k_tiles):
    """A smaller space above 32 tokens: wide tiles, a few ring depths, light
    split-K and balanced split-K with one CTA per SM."""
    for swap in swaps:
        cols = p.M if swap else p.N
        if swap and p.M > 256:
            continue
        for bn in (64, 128, 192, 224, 256):
            if bn > max_bn or (bn > 64 and bn // 2 >= cols):
                continue
            # tile_n 192 and 224 (whole waves for some N) exist without
            # swap-AB for bf16 and per-token/channel FP8
            if bn in (192, 224) and (swap or p.scale == "block" or p.dtype == "int8"):
                continue
            if p.scale == "block" and bn > 128 and swap:
                continue
            for stages in (3, 4, 6):
                for s in (1, 2, 4):
                    if s > k_tiles or (s > 1 and k_tiles // s < 2):
                        continue
                    yield dict(tile_n=bn, stages=stages, split_k=s, swap_ab=swap, stream_k=0,
                               cluster_reduce=0, cta_pair=0)
                yield dict(tile_n=bn, stages=stages, split_k=1, swap_ab=swap, stream_k=1,
                           cluster_reduce=0, cta_pair=0)
        # CTA pairs (256-row tiles, half the weight tile per CTA): plain
        # per-token/channel or bf16 layers, rows over M
        if swap or p.scale == "block" or p.dtype == "int8":
            continue
        for bn in (128, 256):
            if bn > max_bn or (bn > 128 and bn // 2 >= cols):
                continue
            for stages in (4, 5, 6, 8):
                yield dict(tile_n=bn, stages=stages, split_k=1, swap_ab=0, stream_k=0,
                           cluster_reduce=0, cta_pair=1)


# Epilogue classes of the table rows (eg_tuning.h): plain, gated unit,
# behind the per-token quantisation prologue.
EPI_PLAIN, EPI_GATED, EPI_QUANT = 0, 1, 2

# Sweepable workloads beyond inputs.workload(): the gated unit of the
# FP8_Dynamic decode shape (W [2 x 12288, 4096]) and the FP8 / INT8 decode
# layers behind the quantisation prologue (bf16 activations in).
VARIANTS = {"fp8_swiglu": ("fp8_dynamic", EPI_GATED), "fp8_quant": ("fp8_dynamic", EPI_QUANT),
            "int8_quant": ("w8a8_int8", EPI_QUANT)}

GATED_TILES = {0: (64, 128), 1: (16, 32, 64)}  # gated kernels: tile_n per swap_ab


def sweep_problem(workload, M):
    """(problem, epilogue class) of a workload name at M tokens."""
    from epilogue_tcgen05_tmem_gb300 import inputs
    base, epi = VARIANTS.get(workload, (workload, EPI_PLAIN))
    if epi == EPI_GATED:
        p = inputs.make_gated_problem(M, 12288, 4096, "e4m3", "token_channel", act="silu",
                                      outlier_frac=0.01)
    else:
        p = inputs.workload(base, M)
    return p, epi


def gated_ok(c):
    return c["tile_n"] in GATED_TILES[c["swap_ab"]] and not c["cluster_reduce"] and not c["cta_pair"]


def time_config(eg, torch, p, d, Ws, tuning, reps=3, calls=None, epi=EPI_PLAIN):
    try:
        plan = eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=p.bias is not None,
                       residual=p.residual is not None, residual_pre_act=p.residual_pre_act,
                       pdl=True, tuning=tuning, gated=epi == EPI_GATED, quant_a=epi == EPI_QUANT)
    except eg.EgError:
        return None
    stream = torch.cuda.Stream()
    calls = calls or max(len(Ws), 8)

    def enqueue():
        for i in range(calls):
            plan.run(d["A"], Ws[i % len(Ws)], d["Y"], d["s_a"], d["s_w"], d["bias"],
                     d["residual"], stream=stream.cuda_stream)
    try:
        with torch.cuda.stream(stream):
            enqueue()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue()
        g.replay()
        torch.cuda.synchronize()
        if plan.device_status() != eg.EG_OK:
            return None
        times = []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(reps):
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / calls)
        return float(np.median(times))
    finally:
        plan.close()


def pick(results):
    best = min(t for _, t in results)
    near = [(c, t) for c, t in results if t <= best * 1.01]
    near.sort(key=lambda ct: (ct[0]["stream_k"], ct[0]["cluster_reduce"], ct[0]["split_k"],
                              ct[0]["swap_ab"], ct[0]["stages"], ct[1]))
    return near[0]


def sweep(workload, tokens, swaps=(0, 1), verbose=True):
    import torch

    import epilogue_tcgen05_tmem_gb300 as eg
    from epilogue_tcgen05_tmem_gb300 import inputs
    eg.lib()
    rows = []
    for M in tokens:
        p, epi = sweep_problem(workload, M)
        A = torch.from_numpy(np.ascontiguousarray(p.A))
        W = torch.from_numpy(np.ascontiguousarray(p.W))
        if p.dtype == "bf16":
            A, W = A.view(torch.int16).view(torch.bfloat16), W.view(torch.int16).view(torch.bfloat16)
        if epi == EPI_QUANT:
            # the layer reads bf16 activations and quantises them itself
            A = torch.from_numpy(inputs.activations_bf16(p.M, p.K, outlier_frac=0.01)).view(
                torch.bfloat16)
        d = {"A": A.cuda(), "s_a": None, "s_w": None, "bias": None, "residual": None}
        if p.s_a is not None:
            d["s_a"] = torch.from_numpy(p.s_a).cuda()
            d["s_w"] = torch.from_numpy(p.s_w).cuda()
        if p.bias is not None:
            d["bias"] = torch.from_numpy(p.bias.view(np.int16)).view(torch.bfloat16).cuda()
        if p.residual is not None:
            d["residual"] = torch.from_numpy(p.residual.view(np.int16)).view(torch.bfloat16).cuda()
        d["Y"] = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
        W0 = W.cuda()
        nw = min(8, max(1, math.ceil(2 * L2_BYTES / max(W0.numel() * W0.element_size(), 1)) + 1))
        Ws = [W0] + [W0.clone() for _ in range(nw - 1)]
        results = []
        for c in candidates(p, swaps):
            if epi == EPI_GATED and not gated_ok(c):
                continue
            t = time_config(eg, torch, p, d, Ws, c, epi=epi)
            if t is not None:
                results.append((c, t))
        c, t = pick(results)
        bucket = M if M <= 2048 else 0
        row = (eg.DTYPES[p.dtype], eg.SCALES[p.scale], p.N, p.K, bucket, epi, c["tile_n"],
               c["stages"], c["split_k"], c["swap_ab"], c["stream_k"], c["cluster_reduce"],
               c["cta_pair"])
        rows.append(row)
        if verbose:
            top = sorted(results, key=lambda ct: ct[1])[:6]
            best_sk = min((ct for ct in results if ct[0]["stream_k"]), key=lambda ct: ct[1],
                          default=None)
            print(json.dumps({"workload": workload, "M": M, "best": c, "us": round(t, 3),
                              "tried": len(results),
                              "top": [[ct[0], round(ct[1], 3)] for ct in top],
                              "best_stream_k": None if best_sk is None else
                              [best_sk[0], round(best_sk[1], 3)]}), flush=True)
        del Ws, W0, d
        torch.cuda.empty_cache()
    return rows


def format_rows(rows, comment=""):
    out = []
    if comment:
        out.append(f"// {comment}")
    for r in rows:
        out.append("    {%d, %d, %d, %d, %d, %d, %d, %d, %d, %d, %d, %d, %d}," % r)
    return "\n".join(out) + "\n"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="fp8_dynamic")
    ap.add_argument("--tokens", default="1,2,4,8,16,24,32")
    ap.add_argument("--swaps", default="0,1")
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    tokens = [int(x) for x in a.tokens.split(",")]
    rows = sweep(a.workload, tokens, tuple(int(x) for x in a.swaps.split(",")))
    text = format_rows(rows, f"{a.workload}: swept on this GPU")
    if a.out:
        with open(a.out, "a") as f:
            f.write(text)
    print(text)


if __name__ == "__main__":
    main()
