"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bounds:
  * INT8: int32 accumulators bit-exact (debug output), bf16 outputs within
    1 bf16 ulp without split-K (checked with split-K too);
  * everything else: max |Y - Y_oracle| <= 1e-2 * rms(Y_oracle);
  * float32 debug accumulators: max |acc - acc_oracle| <= 1e-4 * rms.
"""
import numpy as np
import pytest
import torch

import epilogue_tcgen05_tmem_gb300 as eg
import oracle
from epilogue_tcgen05_tmem_gb300 import inputs
from tests._gpu_helpers import (assert_close_out, assert_close_rms, bits, canaries_intact,
                                make_plan, run, to_device, ulp_dist)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from epilogue_tcgen05_tmem_gb300 import _build
    _build.build()
    eg.lib()


def check_full(p, tuning=None, rel=1e-2):
    y, _ = run(p, tuning)
    ref = oracle.linear(p)
    if p.dtype == "int8" and (tuning is None or tuning.get("split_k", 1) >= 1):
        d = ulp_dist(bits(y), ref)
        assert d.max() <= 1, f"int8 ulp distance {d.max()}"
    else:
        assert_close_rms(bits(y), ref, rel)
    return y


# ------------------------------------------------------------ bf16 -------

def test_bf16_small_workload_default_tuning():
    # M=64 N=256 K=512, +bias, exact GELU
    check_full(inputs.workload("bf16_small"))


@pytest.mark.parametrize("tuning", [
    dict(tile_n=64, stages=2, split_k=1, swap_ab=0),
    dict(tile_n=128, stages=4, split_k=1, swap_ab=0),
    dict(tile_n=256, stages=3, split_k=1, swap_ab=0),
    dict(tile_n=16, stages=4, split_k=1, swap_ab=0),
    dict(tile_n=64, stages=4, split_k=1, swap_ab=1),
    dict(tile_n=128, stages=4, split_k=2, swap_ab=0),
    dict(tile_n=64, stages=3, split_k=4, swap_ab=1),
])
def test_bf16_small_workload_tunings(tuning):
    check_full(inputs.workload("bf16_small"), tuning)


ODD = [(1, 8, 64), (3, 24, 72), (17, 136, 200), (31, 200, 136), (33, 64, 512),
       (130, 264, 520), (129, 129 + 7, 64 * 3 + 8)]


@pytest.mark.parametrize("M,N,K", ODD)
@pytest.mark.parametrize("swap", [0, 1])
def test_bf16_ragged_shapes(M, N, K, swap):
    p = inputs.make_problem(M, N, K, "bf16", act="gelu_tanh", bias=True, residual=True, seed=11)
    bn = 64 if not swap else (16 if M <= 16 else 32 if M <= 32 else 64)
    check_full(p, dict(tile_n=bn, stages=3, split_k=1, swap_ab=swap))


@pytest.mark.parametrize("act", ["none", "relu", "gelu_erf", "gelu_tanh", "silu"])
@pytest.mark.parametrize("pre", [False, True])
def test_bf16_every_epilogue(act, pre):
    p = inputs.make_problem(70, 192, 320, "bf16", act=act, bias=True, residual=True,
                            residual_pre_act=pre, seed=5)
    check_full(p)
    check_full(p, dict(tile_n=32, stages=4, split_k=3, swap_ab=1))


@pytest.mark.parametrize("S", [2, 3, 5, 8])
@pytest.mark.parametrize("swap", [0, 1])
def test_split_k_bf16_and_determinism(S, swap):
    p = inputs.make_problem(40, 320, 1024, "bf16", act="silu", bias=True, seed=7)
    t = dict(tile_n=64, stages=4, split_k=S, swap_ab=swap)
    plan = make_plan(p, t)
    assert plan.workspace_bytes > 0
    d = to_device(p)
    y1, _ = run(p, plan=plan, d=d)
    y2, _ = run(p, plan=plan, d=d)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "split-K not deterministic"
    assert_close_rms(bits(y1), oracle.linear(p))
    plan.close()


def test_k_zero_and_empty_problems():
    p = inputs.make_problem(5, 24, 0, "bf16", act="gelu_erf", bias=True, seed=1)
    y, _ = run(p)
    assert np.array_equal(bits(y), oracle.linear(p))
    for M, N in [(0, 16), (4, 0)]:
        q = inputs.make_problem(M, N, 64, "bf16", seed=1)
        plan = make_plan(q)
        d = to_device(q)
        plan.run(d["A"], d["W"], d["Y"])
        assert plan.last_launch_count() == 0
        plan.close()


# ------------------------------------------------------------ FP8 -------

@pytest.mark.parametrize("M", inputs.DECODE_TOKENS)
def test_fp8_token_channel_small(M):
    p = inputs.make_problem(M, 384, 1024, "e4m3", "token_channel", act="silu", bias=True,
                            outlier_frac=0.01, seed=2)
    check_full(p)
    check_full(p, dict(tile_n=32 if M > 16 else 16, stages=4, split_k=4, swap_ab=1))
    check_full(p, dict(tile_n=64, stages=4, split_k=2, swap_ab=0))


def test_fp8_token_channel_large_m():
    p = inputs.make_problem(300, 520, 768, "e4m3", "token_channel", act="gelu_tanh",
                            bias=True, residual=True, seed=4)
    check_full(p)
    check_full(p, dict(tile_n=256, stages=4, split_k=1, swap_ab=0))


def _sampled(p, y, npts=3000, seed=0, int8_ulp=False):
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, p.M, npts), np.full(8, p.M - 1), np.zeros(8, int)])
    ns = np.concatenate([rng.integers(0, p.N, npts), np.arange(p.N - 8, p.N), np.arange(8)])
    ref, _ = oracle.linear_points(p, ms, ns)
    got = bits(y)[ms, ns]
    if int8_ulp:
        assert ulp_dist(got, ref).max() <= 1
    else:
        assert_close_rms(got, ref)


@pytest.mark.parametrize("M", inputs.DECODE_TOKENS)
def test_fp8_dynamic_full_size_sampled(M):
    """K=4096 N=12288 decode linear, default (bench) tuning, sampled outputs."""
    p = inputs.workload("fp8_dynamic", M)
    y, _ = run(p)
    _sampled(p, y)


def test_fp8_dynamic_m2048_full_size_sampled():
    """K=4096 N=12288 at 2048 tokens (the table's large-M row), sampled."""
    p = inputs.workload("fp8_dynamic", 2048)
    y, _ = run(p)
    _sampled(p, y, npts=1500)


# ------------------------------------------------------------ INT8 ------

@pytest.mark.parametrize("M,N,K", [(1, 136, 384), (7, 256, 1024), (32, 384, 2048), (130, 200, 640)])
def test_int8_exact_accumulator_and_one_ulp(M, N, K):
    p = inputs.make_problem(M, N, K, "int8", "token_channel", residual=True, seed=9)
    yacc, _ = run(p, debug=True)
    _, _, acc64 = oracle.linear(p, want_acc=True)
    assert np.array_equal(yacc.numpy().astype(np.int64), acc64), "int32 accumulator not exact"
    for t in (None, dict(tile_n=16 if M <= 16 else 32 if M <= 32 else 64, stages=3,
                         split_k=3, swap_ab=1),
              dict(tile_n=64, stages=3, split_k=1, swap_ab=0)):
        y, _ = run(p, t)
        d = ulp_dist(bits(y), oracle.linear(p))
        assert d.max() <= 1, f"tuning {t}: {d.max()} ulp"


@pytest.mark.parametrize("M", [1, 8, 32])
def test_w8a8_int8_full_size(M):
    p = inputs.workload("w8a8_int8", M)
    yacc, _ = run(p, debug=True)
    rng = np.random.default_rng(1)
    ms = rng.integers(0, M, 2000)
    ns = rng.integers(0, p.N, 2000)
    _, acc = oracle.linear_points(p, ms, ns)
    assert np.array_equal(yacc.numpy()[ms, ns].astype(np.int64), acc.astype(np.int64))
    y, _ = run(p)
    _sampled(p, y, int8_ulp=True)


# ------------------------------------------------------- Block FP8 ------

@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (8, 384, 1024), (32, 130, 384), (200, 264, 640)])
def test_block_fp8_small(M, N, K):
    p = inputs.make_problem(M, N, K, "e4m3", "block", seed=13)
    check_full(p)
    check_full(p, dict(tile_n=32, stages=4, split_k=2, swap_ab=1))
    check_full(p, dict(tile_n=128, stages=4, split_k=1, swap_ab=0))


@pytest.mark.parametrize("M", [1, 32, 2048])
def test_block_fp8_full_size_sampled(M):
    p = inputs.workload("block_fp8", M)
    y, _ = run(p)
    _sampled(p, y, npts=1500 if M > 32 else 600)


def test_block_fp8_m2048_cta_pairs_sampled():
    """The Block_FP8 layer at 2048 tokens on 256 x 256 CTA-pair tiles,
    sampled outputs against the oracle."""
    p = inputs.workload("block_fp8", 2048)
    y, _ = run(p, dict(tile_n=256, stages=3, split_k=1, swap_ab=0, cta_pair=1))
    _sampled(p, y, npts=1500, seed=3)


WIDE_BLOCK = [
    dict(tile_n=256, stages=4, split_k=1, swap_ab=0),
    dict(tile_n=256, stages=3, split_k=1, swap_ab=0, stream_k=1),
    dict(tile_n=256, stages=2, split_k=2, swap_ab=0),          # accumulator-commit release
    # CTA pairs: 256 x 256 tiles, each CTA promoting its 128 rows
    dict(tile_n=256, stages=4, split_k=1, swap_ab=0, cta_pair=1),
    dict(tile_n=256, stages=2, split_k=1, swap_ab=0, cta_pair=1),  # accumulator-commit release
]


@pytest.mark.parametrize("tuning", WIDE_BLOCK)
@pytest.mark.parametrize("M,N,K", [(300, 640, 1024), (130, 512, 2048), (17, 256, 384)])
def test_block_fp8_wide_tiles(M, N, K, tuning):
    """256-wide promotion tiles (two weight blocks per tile, 128 running sums
    per epilogue thread, scales read per K block into registers): ragged M,
    N not a multiple of 256 (the second weight block of the last tile lies
    past N), several K splits, and CTA pairs (M = 17: the odd CTA's rows all
    lie past M; M = 130: two of them are valid)."""
    p = inputs.make_problem(M, N, K, "e4m3", "block", act="gelu_erf", bias=True,
                            residual=True, seed=17)
    check_full(p, tuning)


STAGED_CASES = [
    # dtype, scale, M, N, K, tuning, epilogue
    ("bf16", "none", 300, 520, 640, dict(tile_n=64, stages=4, split_k=1, swap_ab=0),
     dict(act="gelu_tanh", bias=True, residual=True, residual_pre_act=True)),
    ("bf16", "none", 520, 648, 512, dict(tile_n=256, stages=6, split_k=1, swap_ab=0, cta_pair=1),
     dict(act="gelu_tanh", bias=True, residual=True, residual_pre_act=True)),
    ("e4m3", "token_channel", 200, 456, 512, dict(tile_n=224, stages=4, split_k=1, swap_ab=0),
     dict(act="silu", bias=True)),
    ("e4m3", "token_channel", 150, 392, 1024, dict(tile_n=128, stages=4, split_k=2, swap_ab=0),
     dict(act="silu", bias=True, residual=True)),
    ("e4m3", "block", 300, 640, 1024, dict(tile_n=256, stages=3, split_k=1, swap_ab=0, stream_k=1),
     dict(act="gelu_erf", bias=True, residual=True)),
    ("e4m3", "block", 600, 896, 768, dict(tile_n=256, stages=3, split_k=1, swap_ab=0, cta_pair=1),
     dict(act="silu", bias=True, residual=True)),
    ("int8", "token_channel", 130, 200, 640, dict(tile_n=64, stages=3, split_k=1, swap_ab=0),
     dict(residual=True)),
]


@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("dtype,scale,M,N,K,tuning,epi", STAGED_CASES)
def test_staged_tma_stores_match_direct_stores(dtype, scale, M, N, K, tuning, epi, out, monkeypatch):
    """Rows over M store Y through shared-memory boxes and TMA stores (the
    boxes clip at M and N); the direct stores from registers
    (EG_STAGED_STORE=0) give bit-identical outputs, and both meet the bound
    against the oracle."""
    p = inputs.make_problem(M, N, K, dtype, scale, seed=23, **epi)
    p.out = out
    y_staged, _ = run(p, tuning)
    monkeypatch.setenv("EG_STAGED_STORE", "0")
    y_direct, _ = run(p, tuning)
    monkeypatch.delenv("EG_STAGED_STORE")
    assert np.array_equal(bits(y_staged), bits(y_direct))
    ref = oracle.linear(p)
    if dtype == "int8" and out == "bf16":
        assert ulp_dist(bits(y_staged), ref).max() <= 1
    else:
        assert_close_out(bits(y_staged), ref, out)


def test_staged_stores_with_unaligned_output_rows_fall_back():
    """Y rows that are not 16-byte aligned: the plan stores directly."""
    p = inputs.make_problem(130, 203, 256, "bf16", act="relu", bias=False, seed=29)
    plan = make_plan(p, dict(tile_n=64, stages=3, split_k=1, swap_ab=0))
    d = to_device(p)
    Yw = torch.full((p.M, 205), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    Y = Yw[:, :p.N]
    plan.run(d["A"], d["W"], Y)
    torch.cuda.synchronize()
    assert plan.device_status() == eg.EG_OK
    assert_close_rms(bits(Y.cpu()), oracle.linear(p))
    assert (Yw[:, p.N:].view(torch.int16) == -1).all()
    plan.close()


@pytest.mark.parametrize("pair", [0, 1])
def test_block_fp8_wide_tiles_debug_accumulators(pair):
    p = inputs.make_problem(140 + 200 * pair, 384, 640, "e4m3", "block", seed=19)
    yacc, _ = run(p, dict(tile_n=256, stages=4, split_k=1, swap_ab=0, cta_pair=pair), debug=True)
    _, acc, _ = oracle.linear(p, want_acc=True)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    assert float(np.max(np.abs(yacc.numpy().astype(np.float64) - acc))) <= 1e-4 * rms


def test_block_fp8_wide_tiles_reject_cluster_reduce():
    with pytest.raises(eg.EgError) as ei:
        eg.Plan(256, 512, 1024, "e4m3", "block",
                tuning=dict(tile_n=256, stages=3, split_k=2, swap_ab=0, cluster_reduce=1))
    assert ei.value.status == eg.EG_ERR_UNSUPPORTED


# ------------------------------------------------- debug accumulators ---

@pytest.mark.parametrize("dtype,scale", [("bf16", "none"), ("e4m3", "token_channel"),
                                         ("e4m3", "block")])
def test_debug_float_accumulators(dtype, scale):
    p = inputs.make_problem(20, 256, 512, dtype, scale, seed=21)
    yacc, _ = run(p, debug=True)
    _, acc, _ = oracle.linear(p, want_acc=True)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    assert float(np.max(np.abs(yacc.numpy().astype(np.float64) - acc))) <= 1e-4 * rms


# ------------------------------------------------ graphs / unfused ------

def test_graph_mode_matches_direct_and_recaptures():
    p = inputs.make_problem(16, 512, 1024, "e4m3", "token_channel", act="silu", bias=True, seed=3)
    ref = oracle.linear(p)
    plan = make_plan(p, graph=True)
    d1, d2 = to_device(p), to_device(p)
    for _ in range(3):
        y1, _ = run(p, plan=plan, d=d1)
        assert plan.last_launch_count() == 1
    y2, _ = run(p, plan=plan, d=d2)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert_close_rms(bits(y2), ref)
    plan.close()


def _table_rows():
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "epilogue_tcgen05_tmem_gb300", "csrc", "eg_tuning_table.inc")
    return [tuple(int(x) for x in m.split(","))
            for m in re.findall(r"^\s*\{([-\d, ]+)\},", open(path).read(), flags=re.M)]


@pytest.mark.parametrize("M", [1, 16, 32])
def test_tuning_lookup_by_epilogue_class(M):
    """Plans take the table row of their own epilogue class: the plain
    FP8_Dynamic decode layer, its gated unit (W [2N, K]) and the layer behind
    the quantisation prologue each get their own swept row."""
    rows = _table_rows()
    keys = ("tile_n", "stages", "split_k", "swap_ab", "stream_k", "cluster_reduce", "cta_pair")

    def want(epi):
        for r in rows:
            if r[:6] == (1, 1, 12288, 4096, M, epi):
                return dict(zip(keys, r[6:]))
        return None
    for epi, kw in ((0, {}), (1, dict(gated=True)), (2, dict(quant_a=True))):
        w = want(epi)
        assert w is not None, epi
        plan = eg.Plan(M, 12288, 4096, "e4m3", "token_channel", "silu", **kw)
        assert plan.tuning == w, (epi, plan.tuning, w)
        plan.close()


def test_graph_cache_evicts_and_recaptures():
    """More distinct argument sets than the plan keeps graphs for: every
    call is still right, also when an evicted set comes back."""
    p = inputs.make_problem(8, 256, 512, "e4m3", "token_channel", act="silu", bias=True, seed=4)
    ref = oracle.linear(p)
    plan = make_plan(p, graph=True)
    ds = [to_device(p) for _ in range(11)]
    for rnd in range(2):
        for d in ds:
            d["Y"].fill_(0)
            y, _ = run(p, plan=plan, d=d)
            assert plan.last_launch_count() == 1
            assert_close_rms(bits(y), ref)
    plan.close()


@pytest.mark.parametrize("pre", [False, True])
def test_unfused_path(pre):
    p = inputs.make_problem(96, 512, 768, "bf16", act="gelu_tanh", bias=True, residual=True,
                            residual_pre_act=pre, seed=8)
    plan = make_plan(p)
    d = to_device(p)
    T1 = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
    T2 = torch.empty_like(T1)
    plan.run_unfused(d["A"], d["W"], d["Y"], T1, T2, d["s_a"], d["s_w"], d["bias"], d["residual"])
    torch.cuda.synchronize()
    assert plan.last_launch_count() == 3
    # the unfused path rounds two intermediates to bf16: allow those steps
    y = bits(d["Y"].cpu())
    ref = oracle.linear(p)
    assert_close_rms(y, ref, rel=3e-2, max_ulp_frac=1e-2)
    plan.run(d["A"], d["W"], d["Y"], d["s_a"], d["s_w"], d["bias"], d["residual"])
    assert plan.last_launch_count() == 1
    plan.close()


# ---------------------------------------------- failure detection -------

def test_device_wait_timeout_reported_without_hang():
    p = inputs.make_problem(8, 256, 512, "bf16", seed=1)
    plan = make_plan(p)
    d = to_device(p)
    plan.set_test_stall(5_000_000, True)           # 5 ms, load warp idle
    plan.run(d["A"], d["W"], d["Y"])
    assert plan.device_status() == eg.EG_ERR_DEVICE_TIMEOUT
    plan.set_test_stall(0, False)
    y, _ = run(p, plan=plan, d=d)
    assert_close_rms(bits(y), oracle.linear(p))
    plan.close()


@pytest.mark.parametrize("dtype,M,N,K,tuning", [
    ("e4m3", 8, 1024, 4096, dict(tile_n=16, stages=4, split_k=4, swap_ab=1)),
    ("int8", 4, 1024, 8192, dict(tile_n=16, stages=3, split_k=8, swap_ab=1)),
])
def test_timeout_in_some_ctas_then_split_k_plan_recovers(dtype, M, N, K, tuning):
    """Odd-numbered CTAs stall: the others finish their splits and count
    their arrivals, so every tile is left half counted (and, for INT8, slot
    0 of the workspace holds partial sums).  After the timeout is reported
    the plan's next run must match the oracle."""
    p = inputs.make_problem(M, N, K, dtype, "token_channel", act="silu", bias=dtype == "e4m3",
                            residual=dtype == "int8", seed=7)
    plan = make_plan(p, tuning)
    d = to_device(p)
    plan.set_test_stall(5_000_000, 2)              # 5 ms, odd CTAs' load warps idle
    plan.run(d["A"], d["W"], d["Y"], d["s_a"], d["s_w"], d["bias"], d["residual"])
    assert plan.device_status() == eg.EG_ERR_DEVICE_TIMEOUT
    plan.set_test_stall(0, 0)
    for _ in range(2):
        y, _ = run(p, plan=plan, d=d)
        ref = oracle.linear(p)
        if dtype == "int8":
            assert ulp_dist(bits(y), ref).max() <= 1
        else:
            assert_close_rms(bits(y), ref)
    plan.close()


def test_test_stall_rejects_unknown_modes():
    p = inputs.make_problem(8, 256, 512, "bf16", seed=1)
    plan = make_plan(p)
    assert eg.eg_plan_set_test_stall(plan.handle, 0, 3) == eg.EG_ERR_INVALID_ARG
    plan.close()


def test_run_argument_errors():
    p = inputs.make_problem(8, 64, 128, "bf16", bias=True, seed=1)
    plan = make_plan(p)
    d = to_device(p)
    bad = plan.args(d["A"], d["W"], d["Y"], bias=d["bias"])
    bad.A = bad.A + 2                                          # misaligned
    assert eg.eg_plan_run(plan.handle, bad, None) == eg.EG_ERR_INVALID_ARG
    alias = plan.args(d["A"], d["W"], d["Y"], bias=d["bias"])
    alias.Y = alias.A                                          # Y aliases A
    assert eg.eg_plan_run(plan.handle, alias, None) == eg.EG_ERR_INVALID_ARG
    nob = plan.args(d["A"], d["W"], d["Y"])
    assert eg.eg_plan_run(plan.handle, nob, None) == eg.EG_ERR_INVALID_ARG
    with pytest.raises(eg.EgError):
        make_plan(p, dict(tile_n=48, stages=4, split_k=1, swap_ab=0))
    with pytest.raises(eg.EgError):
        make_plan(p, dict(tile_n=64, stages=4, split_k=3, swap_ab=0))   # 2 K tiles only
    plan.close()


def test_programmatic_dependent_launch_chain():
    """Calls launched as programmatic dependents (weights streamed before the
    previous kernel finishes) give the same bits as plain launches, also when
    the previous kernel writes this call's activations."""
    p = inputs.make_problem(8, 1024, 2048, "e4m3", "token_channel", act="silu", bias=True, seed=6)
    plain = make_plan(p)
    plan_pdl = eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=True, pdl=True)
    d = to_device(p)
    y_ref, _ = run(p, plan=plain, d=d)
    A0 = d["A"].clone()
    for i in range(6):
        # the previous kernel on the stream rewrites A (same values)
        d["A"].copy_(A0)
        plan_pdl.run(d["A"], d["W"], d["Y"], d["s_a"], d["s_w"], d["bias"])
    torch.cuda.synchronize()
    assert plan_pdl.device_status() == eg.EG_OK
    assert torch.equal(d["Y"].cpu().view(torch.int16), y_ref.view(torch.int16))
    plain.close()
    plan_pdl.close()


def test_unaligned_output_rows_use_scalar_path():
    p = inputs.make_problem(5, 130, 256, "bf16", act="relu", bias=True, residual=True, seed=3)
    check_full(p, dict(tile_n=64, stages=3, split_k=1, swap_ab=0))
    check_full(p, dict(tile_n=16, stages=3, split_k=2, swap_ab=1))


def test_trace_timeline_and_launch_info():
    from epilogue_tcgen05_tmem_gb300 import trace as tr
    p = inputs.make_problem(4, 2048, 1024, "e4m3", "token_channel", act="silu", bias=True, seed=2)
    plan = make_plan(p)
    li = plan.launch_info
    assert 0 < li["grid"] <= li["units"] and li["block"] in (192, 320)
    buf = torch.zeros(li["grid"], eg.EG_TRACE_POINTS, dtype=torch.int64, device="cuda")
    plan.set_trace(buf)
    y, _ = run(p, plan=plan)
    t = buf.cpu().numpy()
    assert (t[:, 0] > 0).all() and (t[:, 7] > 0).all()
    assert tr.ordered(t)
    s = tr.summarize(t)
    assert s["end"]["p100"] >= s["start"]["p0"]
    plan.set_trace(None)
    assert_close_rms(bits(y), oracle.linear(p))
    plan.close()


@pytest.mark.parametrize("dtype,scale,M,N,K,tn,swap", [
    ("bf16", "none", 40, 512, 1024, 64, 0),
    ("bf16", "none", 7, 1000, 640, 16, 1),
    ("e4m3", "token_channel", 3, 1536, 2048, 16, 1),
    ("e4m3", "token_channel", 32, 2048, 4096, 32, 1),
    ("e4m3", "block", 8, 1024, 1024, 16, 1),
    ("e4m3", "block", 300, 384, 640, 128, 0),
])
@pytest.mark.parametrize("sk", [1, 2])
def test_balanced_split_k(dtype, scale, M, N, K, tn, swap, sk):
    """Balanced split-K (stream-K): CTAs share the tiles x K-tiles space in
    equal ranges; tiles split across CTAs reduce through the workspace."""
    p = inputs.make_problem(M, N, K, dtype, scale, act="silu", bias=True, residual=True, seed=12)
    t = dict(tile_n=tn, stages=4, split_k=1, swap_ab=swap, stream_k=sk)
    plan = make_plan(p, t)
    d = to_device(p)
    y1, _ = run(p, plan=plan, d=d)
    y2, _ = run(p, plan=plan, d=d)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    assert_close_rms(bits(y1), oracle.linear(p))
    plan.close()


@pytest.mark.parametrize("sk", [1, 2])
def test_balanced_split_k_int8_exact(sk):
    p = inputs.make_problem(16, 1024, 4096, "int8", "token_channel", residual=True, seed=14)
    t = dict(tile_n=16, stages=3, split_k=1, swap_ab=1, stream_k=sk)
    yacc, _ = run(p, t, debug=True)
    _, _, acc64 = oracle.linear(p, want_acc=True)
    assert np.array_equal(yacc.numpy().astype(np.int64), acc64)
    y, _ = run(p, t)
    assert ulp_dist(bits(y), oracle.linear(p)).max() <= 1


def test_plans_sharing_a_kernel_with_other_ring_depths():
    """Two plans of the same kernel instantiation with different stage
    counts: creating the shallower one must not break the deeper one."""
    p = inputs.make_problem(4, 512, 1024, "e4m3", "token_channel", act="silu", bias=True, seed=2)
    deep = make_plan(p, dict(tile_n=16, stages=6, split_k=2, swap_ab=1))
    shallow = make_plan(p, dict(tile_n=16, stages=2, split_k=2, swap_ab=1))
    ref = oracle.linear(p)
    for plan in (deep, shallow, deep):
        y, _ = run(p, plan=plan)
        assert_close_rms(bits(y), ref)
    deep.close()
    shallow.close()


# ------------------------------------------ split-K inside a cluster ----

CLUSTER_CASES = [
    # dtype, scale, M, N, K, tile_n, swap, split
    ("e4m3", "token_channel", 1, 1536, 2048, 16, 1, 4),
    ("e4m3", "token_channel", 5, 1000, 1024, 16, 1, 2),     # ragged N: partial last row tile
    ("e4m3", "token_channel", 16, 2048, 4096, 16, 1, 8),
    ("e4m3", "token_channel", 27, 1536, 2048, 32, 1, 4),    # ragged columns inside the tile
    ("e4m3", "token_channel", 40, 1024, 2048, 32, 1, 4),    # two column tiles, the last ragged
    ("bf16", "none", 200, 136, 512, 32, 0, 2),              # rows over M, ragged both ways
    ("e4m3", "block", 8, 1024, 1024, 16, 1, 4),
    ("e4m3", "block", 130, 384, 1024, 64, 0, 2),            # 8 epilogue warps
    ("e4m3", "token_channel", 130, 640, 2048, 256, 0, 2),   # 8 epilogue warps, TMEM path
    ("bf16", "none", 200, 384, 1024, 128, 0, 4),
]


@pytest.mark.parametrize("dtype,scale,M,N,K,tn,swap,S", CLUSTER_CASES)
def test_cluster_split_k_matches_workspace_path(dtype, scale, M, N, K, tn, swap, S):
    """Partial sums exchanged through distributed shared memory give the
    same bits as the workspace path with the same split, and meet the bound
    against the oracle."""
    p = inputs.make_problem(M, N, K, dtype, scale, act="silu", bias=True, residual=True, seed=31)
    base = dict(tile_n=tn, stages=4, split_k=S, swap_ab=swap)
    pc = make_plan(p, dict(base, cluster_reduce=1))
    li = pc.launch_info
    assert pc.workspace_bytes == 0
    assert li["grid"] == li["units"]
    assert li["grid"] % S == 0
    yc, _ = run(p, plan=pc)
    yc2, _ = run(p, plan=pc)
    pc.close()
    yw, _ = run(p, dict(base, cluster_reduce=0))
    assert torch.equal(yc.view(torch.int16), yc2.view(torch.int16)), "not deterministic"
    assert torch.equal(yc.view(torch.int16), yw.view(torch.int16)), "differs from the workspace path"
    assert_close_rms(bits(yc), oracle.linear(p))


@pytest.mark.parametrize("M,S", [(1, 4), (16, 8), (29, 2)])
def test_cluster_split_k_int8_exact(M, S):
    p = inputs.make_problem(M, 1000, 4096, "int8", "token_channel", residual=True, seed=33)
    t = dict(tile_n=16 if M <= 16 else 32, stages=4, split_k=S, swap_ab=1, cluster_reduce=1)
    yacc, _ = run(p, t, debug=True)
    _, _, acc64 = oracle.linear(p, want_acc=True)
    assert np.array_equal(yacc.numpy().astype(np.int64), acc64), "int32 accumulator not exact"
    y, _ = run(p, t)
    assert ulp_dist(bits(y), oracle.linear(p)).max() <= 1


def test_cluster_split_k_debug_float_accumulators():
    p = inputs.make_problem(12, 640, 2048, "e4m3", "token_channel", seed=35)
    t = dict(tile_n=16, stages=4, split_k=4, swap_ab=1)
    ya, _ = run(p, dict(t, cluster_reduce=1), debug=True)
    yb, _ = run(p, dict(t, cluster_reduce=0), debug=True)
    assert torch.equal(ya.view(torch.int32), yb.view(torch.int32))
    _, acc, _ = oracle.linear(p, want_acc=True)
    err = np.abs(ya.numpy().astype(np.float64) - acc)
    assert err.max() <= 1e-4 * np.sqrt(np.mean(acc * acc))


def test_cluster_split_k_full_size_decode():
    """The decode linear (K=4096, N=12288) with the cluster reduction, sampled
    outputs against the oracle, through graph replay with PDL."""
    for M in (1, 16, 32):
        p = inputs.workload("fp8_dynamic", M)
        plan = eg.Plan(p.M, p.N, p.K, p.dtype, p.scale, p.act, bias=True, graph=True, pdl=True,
                       tuning=dict(tile_n=16 if M <= 16 else 32, stages=4, split_k=4, swap_ab=1,
                                   cluster_reduce=1))
        d = to_device(p)
        for _ in range(3):
            y, _ = run(p, plan=plan, d=d)
        plan.close()
        _sampled(p, y)


@pytest.mark.parametrize("bad,status", [
    (dict(split_k=3), eg.EG_ERR_UNSUPPORTED),
    (dict(split_k=16), eg.EG_ERR_UNSUPPORTED),
    (dict(split_k=1, stream_k=1), eg.EG_ERR_UNSUPPORTED),
    (dict(stream_k=1), eg.EG_ERR_INVALID_ARG),
    (dict(tile_n=256, stages=2, split_k=2), eg.EG_ERR_UNSUPPORTED),   # buffer > operand ring
])
def test_cluster_split_k_rejected_tunings(bad, status):
    t = dict(dict(tile_n=16, stages=4, split_k=4, swap_ab=1, cluster_reduce=1), **bad)
    with pytest.raises(eg.EgError) as ei:
        eg.Plan(4, 1024, 4096, "e4m3", "token_channel", "silu", bias=True, tuning=t)
    assert ei.value.status == status


# ------------------------------------------------ mid-range token counts ---

@pytest.mark.parametrize("wl,M", [("fp8_dynamic", 48), ("fp8_dynamic", 700), ("w8a8_int8", 100),
                                  ("block_fp8", 300)])
def test_midrange_tokens_table_entries(wl, M):
    """Token counts between the decode buckets and the large-M rule use the
    swept mid-range rows (the first bucket at or above M); sampled outputs
    at the full layer sizes against the oracle."""
    p = inputs.workload(wl, M)
    plan = make_plan(p)
    assert plan.tuning["swap_ab"] == 0  # the mid-range rows all run rows over M
    y, _ = run(p, plan=plan)
    plan.close()
    _sampled(p, y, npts=1500, int8_ulp=(p.dtype == "int8"))


# ------------------------------------------------------ output narrowing ---

OUT_CASES = [
    # dtype, scale, M, N, K, tuning (None: table / default rule)
    ("bf16", "none", 64, 256, 512, None),
    ("bf16", "none", 40, 320, 1024, dict(tile_n=64, stages=4, split_k=3, swap_ab=1)),
    ("e4m3", "token_channel", 5, 1000, 1024, None),
    ("e4m3", "token_channel", 16, 2048, 4096, dict(tile_n=16, stages=4, split_k=4, swap_ab=1,
                                                  cluster_reduce=1)),
    ("e4m3", "token_channel", 130, 200, 640, dict(tile_n=64, stages=3, split_k=1, swap_ab=0)),
    ("int8", "token_channel", 7, 256, 1024, None),
    ("int8", "token_channel", 130, 200, 640, dict(tile_n=64, stages=3, split_k=1, swap_ab=0)),
    ("e4m3", "block", 8, 384, 1024, None),
    ("e4m3", "block", 200, 264, 640, dict(tile_n=128, stages=4, split_k=1, swap_ab=0)),
]


@pytest.mark.parametrize("out", ["f16", "e4m3"])
@pytest.mark.parametrize("dtype,scale,M,N,K,tuning", OUT_CASES)
def test_output_narrowing(out, dtype, scale, M, N, K, tuning):
    """fp16 output, and E4M3 output codes of v / s_y (s_y set so that the
    outputs span most of the E4M3 range), against the oracle."""
    p = inputs.make_problem(M, N, K, dtype, scale, act="silu", bias=True, residual=True, seed=17)
    if out == "e4m3":
        v = (oracle.linear(p).astype(np.uint32) << 16).view(np.float32)   # bf16 output
        p.s_y = float(np.abs(v).max()) / 200.0
    p.out = out
    y, _ = run(p, tuning)
    assert_close_out(bits(y), oracle.linear(p), out)


def test_output_narrowing_rejections():
    for flags in (eg.EG_OUT_F16 | eg.EG_OUT_E4M3, eg.EG_OUT_F16 | eg.EG_OUT_DEBUG_ACCUM):
        s, _ = eg.eg_plan_create(eg.make_problem(4, 256, 512, flags=flags))
        assert s == eg.EG_ERR_INVALID_ARG
    plan = eg.Plan(4, 256, 512, out="e4m3")
    A = torch.zeros(4, 512, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(256, 512, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(4, 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(eg.EgError) as ei:
        plan.run(A, W, Y)   # no s_y
    assert ei.value.status == eg.EG_ERR_INVALID_ARG
    plan.close()


# --------------------------------------------- gated linear unit (SwiGLU) ---

GATED_CASES = [
    # dtype, scale, M, N, K, tuning
    ("e4m3", "token_channel", 1, 1024, 2048, None),
    ("e4m3", "token_channel", 5, 1000, 1024, dict(tile_n=16, stages=4, split_k=3, swap_ab=1)),
    ("e4m3", "token_channel", 16, 512, 4096, dict(tile_n=16, stages=4, split_k=1, swap_ab=1,
                                                 stream_k=2)),
    ("e4m3", "token_channel", 40, 384, 1024, dict(tile_n=64, stages=3, split_k=2, swap_ab=1)),
    ("e4m3", "token_channel", 200, 264, 640, None),
    ("bf16", "none", 7, 300, 512, None),
    ("bf16", "none", 130, 256, 512, dict(tile_n=128, stages=3, split_k=2, swap_ab=0)),
    ("bf16", "none", 130, 200, 512, dict(tile_n=64, stages=4, split_k=1, swap_ab=0)),
]


@pytest.mark.parametrize("dtype,scale,M,N,K,tuning", GATED_CASES)
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
def test_gated_unit(dtype, scale, M, N, K, tuning, act):
    """y = act(gate) * up (+ R) over the two weight halves, against the
    oracle (SiLU: SwiGLU; GELU: GeGLU)."""
    p = inputs.make_gated_problem(M, N, K, dtype, scale, act=act, bias=True, residual=True, seed=23)
    y, _ = run(p, tuning)
    assert_close_rms(bits(y), oracle.linear_gated(p))


@pytest.mark.parametrize("out", ["f16", "e4m3"])
def test_gated_unit_narrow_outputs(out):
    p = inputs.make_gated_problem(8, 512, 1024, "e4m3", "token_channel", act="silu", seed=24)
    if out == "e4m3":
        v = (oracle.linear_gated(p).astype(np.uint32) << 16).view(np.float32)
        p.s_y = float(np.abs(v).max()) / 200.0
    p.out = out
    y, _ = run(p)
    assert_close_out(bits(y), oracle.linear_gated(p), out)


GATED_TWO_PASS_CASES = [
    # dtype, scale, M, N, K, tuning of the accumulator GEMM over the 2N rows
    ("int8", "token_channel", 1, 1024, 2048, None),
    ("int8", "token_channel", 5, 1000, 1024, dict(tile_n=16, stages=3, split_k=4, swap_ab=1)),
    ("int8", "token_channel", 24, 512, 1536, dict(tile_n=32, stages=3, split_k=2, swap_ab=1,
                                                 cluster_reduce=1)),
    ("int8", "token_channel", 150, 320, 640, dict(tile_n=64, stages=3, split_k=1, swap_ab=0)),
    ("e4m3", "block", 1, 512, 1024, None),
    ("e4m3", "block", 9, 384, 768, dict(tile_n=16, stages=3, split_k=2, swap_ab=1)),
    ("e4m3", "block", 300, 640, 1024, dict(tile_n=256, stages=3, split_k=1, swap_ab=0, stream_k=1)),
]


@pytest.mark.parametrize("dtype,scale,M,N,K,tuning", GATED_TWO_PASS_CASES)
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
def test_gated_unit_int8_and_block(dtype, scale, M, N, K, tuning, act):
    """INT8 and Block_FP8 gated units: the fused kernel's accumulators of the
    2N weight rows, then the combine kernel (two launches), against the
    oracle's gated unit; the accumulator GEMM runs swap-AB, split-K (through
    the workspace or a cluster), rows over M and balanced split-K."""
    p = inputs.make_gated_problem(M, N, K, dtype, scale, act=act, bias=True, residual=True, seed=27)
    plan = make_plan(p, tuning)
    y, _ = run(p, plan=plan)
    assert plan.last_launch_count() == 2
    plan.close()
    assert_close_rms(bits(y), oracle.linear_gated(p))


@pytest.mark.parametrize("out", ["f16", "e4m3"])
@pytest.mark.parametrize("dtype,scale", [("int8", "token_channel"), ("e4m3", "block")])
def test_gated_unit_int8_and_block_outputs(dtype, scale, out):
    p = inputs.make_gated_problem(8, 512, 1024, dtype, scale, act="silu", seed=28)
    if out == "e4m3":
        v = (oracle.linear_gated(p).astype(np.uint32) << 16).view(np.float32)
        p.s_y = float(np.abs(v).max()) / 200.0
    p.out = out
    y, _ = run(p)
    assert_close_out(bits(y), oracle.linear_gated(p), out)


@pytest.mark.parametrize("graph", [False, True])
def test_gated_unit_int8_quant_prologue(graph):
    """The INT8 gated unit behind the per-token quantisation prologue (bf16
    activations in; quantisation, accumulator GEMM and combine: three
    launches, programmatic dependents) gives the same bits as quantising
    first and running the unit on the codes, in direct and graph mode."""
    M, N, K = 4, 512, 1024
    p = inputs.make_gated_problem(M, N, K, "int8", "token_channel", act="silu", bias=True, seed=29)
    X = torch.from_numpy(inputs.activations_bf16(M, K, seed=29).view(np.int16)).cuda().view(torch.bfloat16)
    d = to_device(p)
    plan = eg.Plan(M, N, K, "int8", "token_channel", "silu", bias=True, gated=True, quant_a=True,
                   pdl=True, graph=graph)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        plan.run(X, d["W"], Y, None, d["s_w"], d["bias"])
    assert plan.last_launch_count() == 3
    torch.cuda.synchronize()
    assert plan.device_status() == eg.EG_OK
    plan.close()
    q, s = eg.quantize_rows(X, "int8")
    ref = make_plan(p)
    Y2 = torch.empty_like(Y)
    ref.run(q, d["W"], Y2, s, d["s_w"], d["bias"])
    torch.cuda.synchronize()
    ref.close()
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))


def test_gated_unit_rejections():
    with pytest.raises(eg.EgError) as ei:
        eg.Plan(4, 200, 512, "e4m3", "block", gated=True)   # up half off a weight block
    assert ei.value.status == eg.EG_ERR_UNSUPPORTED
    for kw in (dict(residual=True, residual_pre_act=True), dict(debug_accum=True)):
        with pytest.raises(eg.EgError) as ei:
            eg.Plan(4, 256, 512, "int8", "token_channel", gated=True, **kw)
        assert ei.value.status == eg.EG_ERR_INVALID_ARG
    with pytest.raises(eg.EgError) as ei:
        eg.Plan(4, 256, 512, "e4m3", "token_channel", gated=True,
                tuning=dict(tile_n=16, stages=4, split_k=4, swap_ab=1, cluster_reduce=1))
    assert ei.value.status == eg.EG_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype,scale,tn", [("bf16", "none", 64), ("e4m3", "token_channel", 64),
                                            ("e4m3", "block", 128)])
def test_balanced_split_k_with_data_parallel_waves(dtype, scale, tn):
    """More than two waves of tiles: whole tiles go data-parallel first and
    only the last one to two waves split their K range across CTAs."""
    M, N, K = (2560, 1024, 384) if tn == 64 else (4864, 1280, 512)
    p = inputs.make_problem(M, N, K, dtype, scale, act="silu", bias=True, residual=True, seed=44)
    t = dict(tile_n=tn, stages=3, split_k=1, swap_ab=0, stream_k=1)
    plan = make_plan(p, t)
    li = plan.launch_info
    tiles = ((M + 127) // 128) * ((N + tn - 1) // tn)
    assert tiles >= 2 * li["grid"], (tiles, li)
    d = to_device(p)
    y1, _ = run(p, plan=plan, d=d)
    y2, _ = run(p, plan=plan, d=d)
    plan.close()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    assert_close_rms(bits(y1), oracle.linear(p))


# ------------------------------------------------------------ CTA pairs ----

PAIR_CASES = [
    # M, N, K, tile_n: one pair row; ragged M/N/K (odd CTA partly empty);
    # M < 128 (odd CTA has no rows); more units than pairs (persistent)
    (256, 512, 512, 128),
    (300, 640, 1008, 256),
    (100, 384, 256, 128),
    (2048, 3072, 512, 256),
]


@pytest.mark.parametrize("dtype,scale", [("bf16", "none"), ("e4m3", "token_channel")])
@pytest.mark.parametrize("M,N,K,tn", PAIR_CASES)
def test_cta_pair(dtype, scale, M, N, K, tn):
    """Pair UMMAs over a 2-CTA cluster (256-row tiles, half the weight tile
    per CTA) meet the bound against the oracle and are deterministic."""
    p = inputs.make_problem(M, N, K, dtype, scale, act="silu", bias=True, residual=True, seed=41)
    plan = make_plan(p, dict(tile_n=tn, stages=4, split_k=1, swap_ab=0, cta_pair=1))
    li = plan.launch_info
    assert plan.tuning["cta_pair"] == 1
    assert li["grid"] % 2 == 0 and li["units"] == -(-M // 256) * -(-N // tn)
    d = to_device(p)
    y1, _ = run(p, plan=plan, d=d)
    y2, _ = run(p, plan=plan, d=d)
    assert canaries_intact(d)
    plan.close()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    assert_close_rms(bits(y1), oracle.linear(p))


def test_cta_pair_prefill_epilogue():
    """bf16 pair tiles with the prefill epilogue (bias + residual, then tanh
    GELU) and deeper rings."""
    p = inputs.make_problem(512, 768, 1024, "bf16", act="gelu_tanh", bias=True, residual=True,
                            residual_pre_act=True, seed=43)
    for stages in (5, 6):
        y, _ = run(p, dict(tile_n=256, stages=stages, split_k=1, swap_ab=0, cta_pair=1))
        assert_close_rms(bits(y), oracle.linear(p))


@pytest.mark.parametrize("t", [
    dict(tile_n=128, stages=4, split_k=1, swap_ab=1, cta_pair=1),
    dict(tile_n=128, stages=4, split_k=2, swap_ab=0, cta_pair=1),
    dict(tile_n=64, stages=4, split_k=1, swap_ab=0, cta_pair=1),
    dict(tile_n=128, stages=4, split_k=1, swap_ab=0, stream_k=1, cta_pair=1),
])
def test_cta_pair_unsupported_tunings(t):
    p = inputs.make_problem(256, 512, 512, "e4m3", "token_channel", seed=1)
    with pytest.raises(eg.EgError):
        make_plan(p, t)


def test_cta_pair_block_scales_need_wide_tiles():
    """Block-scale pairs exist only for 256-wide promotion tiles."""
    p = inputs.make_problem(256, 512, 512, "e4m3", "block", seed=1)
    with pytest.raises(eg.EgError):
        make_plan(p, dict(tile_n=128, stages=3, split_k=1, swap_ab=0, cta_pair=1))
    with pytest.raises(eg.EgError):
        make_plan(p, dict(tile_n=256, stages=3, split_k=2, swap_ab=0, cta_pair=1))


@pytest.mark.parametrize("dtype,scale", [("bf16", "none"), ("e4m3", "token_channel")])
@pytest.mark.parametrize("t", [dict(split_k=1, stream_k=0), dict(split_k=3, stream_k=0),
                               dict(split_k=1, stream_k=1)])
@pytest.mark.parametrize("tn", [128, 192, 224, 256])
def test_wide_tile_split_k(dtype, scale, t, tn):
    """Wide tiles without swap-AB (eight epilogue warps, each owning half of
    a TMEM lane quarter's columns; tile_n 192 and 224 with accumulator
    buffers 256 columns apart), unsplit, through the split-K workspace and
    balanced split-K; N = 700 leaves a ragged last tile column."""
    p = inputs.make_problem(300, 700, 2048, dtype, scale, act="gelu_tanh", bias=True,
                            residual=True, seed=45)
    y, _ = run(p, dict(tile_n=tn, stages=4, swap_ab=0, **t))
    assert_close_rms(bits(y), oracle.linear(p))


def test_prefill_full_size_sampled():
    """The bf16 prefill block at its full size (4096^3, bias + residual, then
    tanh GELU) with the table's tuning (CTA pairs, stages released two per
    commit), sampled outputs against the oracle, plus the single-CTA tiles
    with one stage per commit."""
    p = inputs.workload("prefill_bf16")
    plan = make_plan(p)
    assert plan.tuning["cta_pair"] == 1
    y, _ = run(p, plan=plan)
    plan.close()
    _sampled(p, y, npts=2000)
    y2, _ = run(p, dict(tile_n=256, stages=4, split_k=1, swap_ab=0))
    _sampled(p, y2, npts=500, seed=1)
