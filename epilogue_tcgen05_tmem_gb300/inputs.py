"""Seeded synthetic inputs for the fused scaled linear layer.

This module is the one piece shared by the CUDA path's tests/bench and by
the CPU oracle's tests.  It holds none of the layer's arithmetic: it only
draws random numbers and stores them in the input formats the layer takes
(bf16, FP8-e4m3 or INT8 codes plus fp32 scales).

Generator (documented so any reader can re-derive every byte):

* SplitMix64, counter based.  For tensor stream ``s`` under seed ``seed`` the
  key is ``mix(seed * 0x100000001B3 + s)`` and draw ``i`` is
  ``mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` where ``mix`` is the SplitMix64
  finaliser.  Uniforms are ``((u >> 11) + 0.5) * 2**-53`` in (0, 1).
* Normals by Box-Muller in float64: draws ``2j`` and ``2j+1`` give
  ``r = sqrt(-2 ln u0)``, ``t = 2 pi u1`` and elements ``2j -> r cos t``,
  ``2j+1 -> r sin t``.
* Stream ids: A=1, W=2, bias=3, residual=4, outlier channels=5.

Storage formats (the layer's inputs, prepared once on the host):

* bf16: float64 -> float32 -> bf16 (round to nearest even), via torch casts.
* FP8-e4m3 with scale ``s = amax / 448`` over the scale group (a token row,
  an output channel, a 1x128 or 128x128 block); codes are
  ``e4m3(clamp(x / s, -448, 448))`` with torch's round-to-nearest-even cast.
  ``amax == 0`` gives ``s = 1``.
* INT8 with ``s = amax / 127`` and ``q = clip(rint(x / s), -127, 127)``.

The pages (Helion linear backend in vLLM, section on the one tunable
kernel) define the three scale formats: FP8_Dynamic (per-token activation,
per-channel weight), W8A8_INT8 (same scaling in INT8) and Block_FP8 (1x128
activation blocks, 128x128 weight blocks).  How a value is quantised is not
stated there; the rule above is this library's input recipe.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

STREAM_A, STREAM_W, STREAM_BIAS, STREAM_RES, STREAM_OUTLIER = 1, 2, 3, 4, 5

_CHUNK = 1 << 22


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return _mix_int(seed * 0x100000001B3 + stream)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit draws ``start .. start+count-1`` of one stream."""
    key = np.uint64(stream_key(seed, stream))
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + ctr * _GOLDEN)


def _normal_chunk(seed, stream, start_pair, npairs):
    u = uniform_u64(seed, stream, 2 * start_pair, 2 * npairs)
    f = ((u >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(f[0::2]))
    t = (2.0 * math.pi) * f[1::2]
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """float64 N(0, std^2) samples, row-major over ``shape``."""
    n = int(np.prod(shape))
    npairs = (n + 1) // 2
    chunks = [(p, min(_CHUNK, npairs - p)) for p in range(0, npairs, _CHUNK)]
    if len(chunks) <= 1:
        parts = [_normal_chunk(seed, stream, p, c) for p, c in chunks]
    else:
        with ThreadPoolExecutor(max_workers=min(16, len(chunks))) as ex:
            parts = list(ex.map(lambda pc: _normal_chunk(seed, stream, *pc), chunks))
    flat = np.concatenate(parts)[:n] if parts else np.zeros(0)
    if std != 1.0:
        flat *= std
    return flat.reshape(shape)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Seeded Fisher-Yates shuffle of 0..n-1 (draw i picks among n-i)."""
    u = uniform_u64(seed, stream, 0, max(n - 1, 0))
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(u[n - 1 - i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


# ---------------------------------------------------------------- storage ---

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _e4m3_codes(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(x32, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _safe_scale(amax: np.ndarray, qmax: float) -> np.ndarray:
    s = (amax.astype(np.float32) / np.float32(qmax)).astype(np.float32)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def quant_rows(x: np.ndarray, dtype: str):
    """Per-row (per-token or per-output-channel) quantisation of a 2-D array."""
    x32 = x.astype(np.float32)
    amax = np.abs(x32).max(axis=1) if x32.shape[1] else np.zeros(x32.shape[0], np.float32)
    if dtype == "e4m3":
        s = _safe_scale(amax, 448.0)
        q = _e4m3_codes(x32 / s[:, None])
    elif dtype == "int8":
        s = _safe_scale(amax, 127.0)
        q = np.clip(np.rint(x32 / s[:, None]), -127, 127).astype(np.int8)
    else:
        raise ValueError(dtype)
    return q, s


def quant_blocks(x: np.ndarray, br: int, bc: int):
    """e4m3 quantisation with one fp32 scale per (br x bc) block; returns
    codes and scales shaped [ceil(R/br), ceil(C/bc)]."""
    R, C = x.shape
    nr, nc = -(-R // br), -(-C // bc)
    x32 = x.astype(np.float32)
    pad = np.zeros((nr * br, nc * bc), np.float32)
    pad[:R, :C] = np.abs(x32)
    amax = pad.reshape(nr, br, nc, bc).max(axis=(1, 3))
    s = _safe_scale(amax, 448.0)
    full = np.repeat(np.repeat(s, br, axis=0), bc, axis=1)[:R, :C]
    q = _e4m3_codes(x32 / full)
    return q, s


# -------------------------------------------------------------- problems ---

@dataclass
class Problem:
    """One synthetic fused-linear problem in the layer's input formats.

    A is [M, K] and W is [N, K] (both K-major).  ``s_a``/``s_w`` are fp32:
    [M] and [N] for token/channel scaling, [M, K/128] and [N/128, K/128] for
    block scaling, None for bf16.  bias is bf16 bits [N] or None, residual is
    bf16 bits [M, N] or None.
    """
    M: int
    N: int
    K: int
    dtype: str            # "bf16" | "e4m3" | "int8"
    scale: str            # "none" | "token_channel" | "block"
    act: str              # "none" | "relu" | "gelu_erf" | "gelu_tanh" | "silu"
    bias: np.ndarray | None
    residual: np.ndarray | None
    A: np.ndarray
    W: np.ndarray
    s_a: np.ndarray | None = None
    s_w: np.ndarray | None = None
    residual_pre_act: bool = False
    name: str = ""
    meta: dict = field(default_factory=dict)
    out: str = "bf16"     # output format: "bf16" | "f16" | "e4m3" (codes of Y / s_y)
    s_y: float = 1.0      # per-tensor output scale (E4M3 output only)


def make_problem(M, N, K, dtype="bf16", scale=None, act="none", bias=False,
                 residual=False, residual_pre_act=False, seed=0, a_std=1.0,
                 w_std=None, bias_std=0.1, outlier_frac=0.0, outlier_mult=10.0,
                 name="") -> Problem:
    """Draw one problem.  Defaults follow the pages' decode/prefill
    workloads: A ~ N(0,1), W ~ N(0,1)/sqrt(K), bias ~ N(0, 0.1), R ~ N(0,1)."""
    if scale is None:
        scale = "none" if dtype == "bf16" else "token_channel"
    if w_std is None:
        w_std = 1.0 / math.sqrt(K) if K > 0 else 1.0
    a = normal(seed, STREAM_A, (M, K), a_std)
    if outlier_frac > 0 and K > 0:
        nout = int(round(outlier_frac * K))
        cols = np.sort(permutation(seed, STREAM_OUTLIER, K)[:nout])
        a[:, cols] *= outlier_mult
    w = normal(seed, STREAM_W, (N, K), w_std)
    s_a = s_w = None
    if dtype == "bf16":
        A, W = to_bf16_bits(a), to_bf16_bits(w)
    elif scale == "token_channel":
        A, s_a = quant_rows(a, dtype)
        W, s_w = quant_rows(w, dtype)
    elif scale == "block":
        if dtype != "e4m3":
            raise ValueError("block scaling is defined for e4m3 only")
        A, s_a = quant_blocks(a, 1, 128)
        W, s_w = quant_blocks(w, 128, 128)
    else:
        raise ValueError((dtype, scale))
    b = to_bf16_bits(normal(seed, STREAM_BIAS, (N,), bias_std)) if bias else None
    r = to_bf16_bits(normal(seed, STREAM_RES, (M, N))) if residual else None
    return Problem(M, N, K, dtype, scale, act, b, r, A, W, s_a, s_w,
                   residual_pre_act, name)


def take_tokens(p: Problem, m: int) -> Problem:
    """The first ``m`` tokens of a problem (per-token data is row-local, so
    this equals drawing the problem with M = m rows)."""
    s_a = None if p.s_a is None else np.ascontiguousarray(p.s_a[:m])
    r = None if p.residual is None else np.ascontiguousarray(p.residual[:m])
    return Problem(m, p.N, p.K, p.dtype, p.scale, p.act, p.bias, r,
                   np.ascontiguousarray(p.A[:m]), p.W, s_a, p.s_w,
                   p.residual_pre_act, p.name, dict(p.meta), p.out, p.s_y)


# Workloads of the pages, restated as seeded synthetic problems.
DECODE_TOKENS = (1, 2, 4, 8, 16, 24, 32)


def workload(name: str, M: int | None = None, seed: int = 0) -> Problem:
    if name == "bf16_small":            # M=64 N=256 K=512, +bias, exact GELU
        return make_problem(64, 256, 512, "bf16", act="gelu_erf", bias=True,
                            seed=seed, name=name)
    if name == "fp8_dynamic":           # K=4096 N=12288, +bias, SiLU
        p = make_problem(max(32, M or 32), 12288, 4096, "e4m3", "token_channel", act="silu",
                         bias=True, outlier_frac=0.01, seed=seed, name=name)
        return take_tokens(p, M or 32)
    if name == "w8a8_int8":             # K=12288 N=4096, + residual
        p = make_problem(max(32, M or 32), 4096, 12288, "int8", "token_channel",
                         residual=True, seed=seed, name=name)
        return take_tokens(p, M or 32)
    if name == "block_fp8":             # K=5120 N=25600
        return make_problem(M or 32, 25600, 5120, "e4m3", "block", seed=seed,
                            name=name)
    if name == "prefill_bf16":          # 4096^3, bias + residual, then GELU
        return make_problem(4096, 4096, 4096, "bf16", act="gelu_tanh", bias=True,
                            residual=True, residual_pre_act=True, seed=seed,
                            name=name)
    raise KeyError(name)


def activations_bf16(M: int, K: int, seed: int = 0, outlier_frac: float = 0.0,
                     outlier_mult: float = 10.0) -> np.ndarray:
    """bf16 bit patterns [M, K] of the activations make_problem draws (the
    same seed streams and outlier columns), before any quantisation: the
    input of the per-token quantisation prologue."""
    a = normal(seed, STREAM_A, (M, K), 1.0)
    if outlier_frac > 0 and K > 0:
        nout = int(round(outlier_frac * K))
        cols = np.sort(permutation(seed, STREAM_OUTLIER, K)[:nout])
        a[:, cols] *= outlier_mult
    return to_bf16_bits(a)


def make_gated_problem(M, N, K, dtype="bf16", scale=None, act="silu", bias=False,
                       residual=False, seed=0, outlier_frac=0.0) -> Problem:
    """A gated (SwiGLU when act is SiLU) layer: W [2N, K] holds the gate half
    then the up half (each quantised per row like any weight), s_w and bias
    cover the 2N rows; the output and the residual are [M, N]."""
    p = make_problem(M, 2 * N, K, dtype, scale, act=act, bias=bias, residual=False, seed=seed,
                     outlier_frac=outlier_frac)
    p.N = N
    if residual:
        p.residual = to_bf16_bits(normal(seed, STREAM_RES, (M, N)))
    p.meta["gated"] = True
    return p
