"""Host-side byte accounting, pinned to the numbers the pages print."""
import os

from epilogue_tcgen05_tmem_gb300 import traffic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.txt")


def _facts():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            out[k] = [float(x) if "." in x else int(x) for x in v]
    return out


def test_intermediate_is_exactly_32_mb():
    M, N, elt, nbytes = _facts()["intermediate"]
    assert traffic.unfused_intermediate_bytes(M, N, elt) == nbytes == 32 * 2 ** 20


def test_pointwise_kernel_element_count():
    M, N, n = _facts()["pointwise_elements"]
    assert M * N == n


def test_fused_vs_unfused_access_counts():
    # 3 kernels: 6 VRAM accesses per element; fused: 2.  For the bias+GELU
    # block, the unfused path adds two intermediates written and read once.
    unf, fused = _facts()["vram_accesses_per_element"]
    M = N = 4096
    assert traffic.unfused_extra_bytes(M, N) == (unf - fused) * traffic.unfused_intermediate_bytes(M, N)


def test_decode_bytes_formulas():
    # FP8 decode: W 12288x4096 e4m3 + s_w + bias + per token (A + s_a + Y)
    for M in (1, 32):
        b = traffic.algorithmic_bytes(M, 12288, 4096, "e4m3", "token_channel", bias=True)
        assert b == 50_405_376 + 28_676 * M
        b = traffic.algorithmic_bytes(M, 4096, 12288, "int8", "token_channel", residual=True)
        assert b == 50_348_032 + 28_676 * M
        b = traffic.algorithmic_bytes(M, 25600, 5120, "e4m3", "block")
        assert b == 131_104_000 + 56_480 * M
    assert traffic.flops(4096, 4096, 4096) == 137_438_953_472
