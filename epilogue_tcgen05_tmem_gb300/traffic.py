"""Algorithmic traffic and work of one fused linear-layer call.

Algorithmic bytes count every tensor the layer reads or writes exactly once
(the fused kernel's ideal HBM traffic): A, W, their scales, bias, the
residual and Y.  Split-K workspace traffic is overhead, not counted.

The unfused three-kernel path ("Helion + TorchInductor co-operation:
operator fusion", section "Anatomy of the opacity barrier", table of VRAM
accesses) additionally writes and reads back two [M, N] bf16 intermediates
(GEMM output, then bias/activation input): 4 extra transfers of
M * N * 2 bytes.  At 4096 x 4096 one such intermediate is the page's
"exactly 32 MB" (33,554,432 bytes).
"""
from __future__ import annotations

ELT = {"bf16": 2, "e4m3": 1, "int8": 1}


def algorithmic_bytes(M, N, K, dtype, scale, bias=False, residual=False) -> int:
    e = ELT[dtype]
    b = M * K * e + N * K * e
    if scale == "token_channel":
        b += 4 * M + 4 * N
    elif scale == "block":
        kb = K // 128
        b += 4 * M * kb + 4 * ((N + 127) // 128) * kb
    if bias:
        b += 2 * N
    if residual:
        b += 2 * M * N
    b += 2 * M * N  # Y
    return b


def flops(M, N, K) -> int:
    return 2 * M * N * K


def unfused_intermediate_bytes(M, N, elt_bytes=2) -> int:
    """Size of one materialised [M, N] intermediate."""
    return M * N * elt_bytes


def unfused_extra_bytes(M, N, elt_bytes=2) -> int:
    """Extra HBM traffic of the 3-kernel path over the fused one: two
    intermediates, each written once and read once."""
    return 4 * unfused_intermediate_bytes(M, N, elt_bytes)


def problem_bytes(p) -> int:
    return algorithmic_bytes(p.M, p.N, p.K, p.dtype, p.scale, p.bias is not None,
                             p.residual is not None)
