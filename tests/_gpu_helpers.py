"""Helpers shared by the GPU parity tests: move a seeded problem to the
device, run it through the C ABI and compare with the oracle."""
import math
import re

import numpy as np
import torch

import epilogue_tcgen05_tmem_gb300 as eg
import oracle

_EG_H = None


def header_functions():
    """Function names declared in include/eg.h."""
    import os
    global _EG_H
    if _EG_H is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "eg.h")
        src = open(path).read()
        _EG_H = sorted(set(re.findall(r"EG_API\s+[\w\s\*]+?\b(eg_\w+)\s*\(", src)))
    return _EG_H


def dev_codes(arr, dtype):
    t = torch.from_numpy(np.ascontiguousarray(arr))
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def to_device(p, debug=False, y_pad=0):
    """Device tensors of problem p; Y is allocated with `y_pad` canary
    elements before and after it (filled with 0xFFFF bf16 NaN / 0xFFFFFFFF)."""
    d = {"A": dev_codes(p.A, p.dtype), "W": dev_codes(p.W, p.dtype)}
    d["s_a"] = None if p.s_a is None else torch.from_numpy(np.ascontiguousarray(p.s_a, np.float32)).cuda()
    d["s_w"] = None if p.s_w is None else torch.from_numpy(np.ascontiguousarray(p.s_w, np.float32)).cuda()
    d["bias"] = None if p.bias is None else dev_codes(p.bias, "bf16")
    d["residual"] = None if p.residual is None else dev_codes(p.residual, "bf16")
    out = getattr(p, "out", "bf16")
    if debug:
        dt = torch.int32 if p.dtype == "int8" else torch.float32
        buf = torch.full((p.M * p.N + 2 * y_pad,), -1, dtype=torch.int32, device="cuda").view(dt)
    elif out == "e4m3":
        buf = torch.full((p.M * p.N + 2 * y_pad,), 0xFF, dtype=torch.uint8, device="cuda")
    else:
        buf = torch.full((p.M * p.N + 2 * y_pad,), -1, dtype=torch.int16, device="cuda").view(
            torch.float16 if out == "f16" else torch.bfloat16)
    d["s_y"] = torch.tensor([p.s_y], dtype=torch.float32, device="cuda") if out == "e4m3" else None
    d["_ybuf"] = buf
    d["Y"] = buf[y_pad:y_pad + p.M * p.N].view(p.M, p.N)
    d["_pad"] = y_pad
    return d


def canaries_intact(d):
    pad = d["_pad"]
    if pad == 0:
        return True
    b = d["_ybuf"]
    if b.dtype == torch.uint8:
        return bool((b[:pad] == 0xFF).all().item() and (b[-pad:] == 0xFF).all().item())
    raw = b.view(torch.int32 if b.element_size() == 4 else torch.int16)
    return bool((raw[:pad] == -1).all().item() and (raw[-pad:] == -1).all().item())


def make_plan(p, tuning=None, debug=False, graph=False):
    return eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=p.bias is not None,
                   residual=p.residual is not None, residual_pre_act=p.residual_pre_act,
                   debug_accum=debug, graph=graph, tuning=tuning,
                   out="bf16" if debug else getattr(p, "out", "bf16"),
                   gated=bool(p.meta.get("gated")))


def run(p, tuning=None, debug=False, graph=False, y_pad=64, plan=None, d=None):
    own = plan is None
    plan = plan or make_plan(p, tuning, debug, graph)
    d = d or to_device(p, debug, y_pad)
    plan.run(d["A"], d["W"], d["Y"], d["s_a"], d["s_w"], d["bias"], d["residual"], s_y=d.get("s_y"))
    torch.cuda.synchronize()
    st = plan.device_status()
    assert st == eg.EG_OK, eg.last_error_detail()
    assert canaries_intact(d), "write outside Y"
    out = d["Y"].cpu()
    if own:
        plan.close()
    return out, d


def bits(y):
    """torch bf16 / fp16 tensor -> numpy uint16 bits (uint8 codes stay codes)."""
    if y.dtype == torch.uint8:
        return y.contiguous().numpy()
    return y.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.bfloat16).double().numpy()


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def assert_close_rms(y_bits, ref_bits, rel=1e-2, max_ulp_frac=1e-3):
    """Bound: max |Y - Y_oracle| <= 1e-2 * rms(Y_oracle), applied per element
    as max(1e-2 * rms, one bf16 ulp of Y_oracle).  Above |Y| ~ 1.28 rms the
    bf16 spacing itself exceeds 1e-2 * rms, so one rounding step that the
    fp32 accumulation order can flip is the resolution of the output there;
    such elements must sit exactly one ulp away, and be rare."""
    y, r = bf16_f64(y_bits), bf16_f64(ref_bits)
    assert np.all(np.isfinite(y)), "non-finite output"
    if r.size == 0:
        return 0.0, 0.0
    rms = math.sqrt(float(np.mean(r * r)))
    diff = np.abs(y - r)
    tol = rel * rms
    over = diff > tol + 1e-30
    if over.any():
        assert np.all(diff[over] <= bf16_ulp(r[over])), \
            f"max err {float(diff.max()):.4g} > max({rel} * rms {rms:.4g}, 1 ulp)"
        assert over.mean() <= max_ulp_frac, f"{int(over.sum())} one-ulp elements ({over.mean():.2e})"
    return float(diff.max()), rms


def ulp_dist(a_bits, b_bits):
    """Distance in bf16 ulps between two arrays of bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def f16_ulp(x):
    """Spacing of fp16 values at |x| (11 significant bits, subnormal floor)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def assert_close_out(y, ref, out, rel=1e-2, max_off_frac=1e-2):
    """The bound for the narrowed outputs.  fp16: as for bf16, per element
    max(1e-2 * rms, one fp16 ulp of the oracle value).  E4M3 codes: the
    format's own step is coarser than 1e-2 * rms, so the kernel's code is the
    oracle's or its neighbour (the float32 epilogue value can sit on the
    other side of a rounding boundary than the float64 one), neighbours
    being rare."""
    if out == "bf16":
        return assert_close_rms(y, ref, rel)
    if out == "f16":
        yv = y.view(np.float16).astype(np.float64)
        rv = ref.view(np.float16).astype(np.float64)
        assert np.all(np.isfinite(yv)), "non-finite output"
        rms = float(np.sqrt(np.mean(rv * rv))) if rv.size else 0.0
        diff = np.abs(yv - rv)
        over = diff > rel * rms + 1e-30
        if over.any():
            assert np.all(diff[over] <= f16_ulp(rv[over])), f"max err {diff.max():.4g}"
            assert over.mean() <= 1e-3
        return
    def ordered(c):
        c = c.astype(np.int64)
        return np.where(c & 0x80, -(c & 0x7F), c)
    d = np.abs(ordered(y) - ordered(ref))
    assert d.max() <= 1, f"E4M3 codes {int(d.max())} steps apart"
    assert (d > 0).mean() <= max_off_frac, f"{int((d > 0).sum())} codes one step off"
