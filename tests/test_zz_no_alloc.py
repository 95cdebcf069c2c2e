"""eg_linear_noalloc: the fused linear layer without any device allocation.

Callers such as code running inside a memory pool or arena that owns the
whole device, or runtimes that forbid cudaMalloc once they are running,
cannot let the library allocate its split-K scratch.  eg_linear_noalloc
runs the same kernel with that scratch in a fixed array compiled into the
library.  These tests call it through the C ABI on split-K problems, on two
calls in a row (the second call finds the array holding the first call's
leftovers), and check that:

* its output is bit-identical to the plan-based entry point's
  (eg_plan_create + eg_plan_run): both run the same kernel with the same
  split order;
* both meet the parity bound against the oracle;
* the device's free memory does not change across a call.

This file is collected last on purpose; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import epilogue_tcgen05_tmem_gb300 as eg
from epilogue_tcgen05_tmem_gb300 import inputs
import oracle
from tests._gpu_helpers import assert_close_rms, bits, make_plan, to_device, ulp_dist

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from epilogue_tcgen05_tmem_gb300 import _build
    _build.build()
    eg.lib()


def _plan_output(p, tuning):
    plan = make_plan(p, tuning)
    d = to_device(p)
    plan.run(d["A"], d["W"], d["Y"], d["s_a"], d["s_w"], d["bias"], d["residual"])
    torch.cuda.synchronize()
    assert plan.device_status() == eg.EG_OK
    y = d["Y"].cpu()
    plan.close()
    return y


def _noalloc_call(p, tuning, d):
    flags = 0
    if p.bias is not None:
        flags |= eg.EG_EPI_BIAS
    if p.residual is not None:
        flags |= eg.EG_EPI_RESIDUAL_PRE_ACT if p.residual_pre_act else eg.EG_EPI_RESIDUAL
    prob = eg.make_problem(p.M, p.N, p.K, p.dtype, p.scale, p.act, flags)
    t = eg.make_tuning(**tuning)
    args = eg.eg_args(d["A"].data_ptr(), d["W"].data_ptr(),
                      None if d["s_a"] is None else d["s_a"].data_ptr(),
                      None if d["s_w"] is None else d["s_w"].data_ptr(),
                      None if d["bias"] is None else d["bias"].data_ptr(),
                      None if d["residual"] is None else d["residual"].data_ptr(),
                      d["Y"].data_ptr(), p.K, p.K, p.N, p.N)
    s = eg.eg_linear_noalloc(prob, t, args, torch.cuda.current_stream().cuda_stream)
    assert s == eg.EG_OK, eg.last_error_detail()


def _noalloc_output(p, tuning):
    d = to_device(p)
    _noalloc_call(p, tuning, d)
    torch.cuda.synchronize()
    return d["Y"].cpu()


def _check_pair(p, tuning):
    ref = oracle.linear(p)
    want = bits(_plan_output(p, tuning))
    got = bits(_noalloc_output(p, tuning))
    assert np.array_equal(got, want), "no-alloc output differs from the plan path's"
    if p.dtype == "int8":
        assert ulp_dist(got, ref).max() <= 1
    else:
        assert_close_rms(got, ref)


@pytest.mark.parametrize("tuning", [
    dict(tile_n=16, stages=4, split_k=4, swap_ab=1),
    dict(tile_n=16, stages=4, split_k=1, swap_ab=1, stream_k=1),
])
def test_noalloc_matches_plan_entry_two_calls(tuning):
    first = inputs.make_problem(8, 2048, 4096, "e4m3", "token_channel", act="silu", bias=True,
                                outlier_frac=0.01, seed=31)
    second = inputs.make_problem(8, 2048, 4096, "e4m3", "token_channel", act="silu", bias=True,
                                 outlier_frac=0.01, seed=32)
    for p in (first, second):
        _check_pair(p, tuning)


def test_noalloc_int8_split_k_two_calls():
    t = dict(tile_n=16, stages=3, split_k=8, swap_ab=1)
    for seed in (41, 42):
        p = inputs.make_problem(4, 1024, 8192, "int8", "token_channel", residual=True, seed=seed)
        _check_pair(p, t)


def test_noalloc_leaves_free_device_memory_unchanged():
    """The call's whole contract: no device allocation.  The first call on
    the device may load the library's module (and with it the scratch
    array); across every later call the device's free memory must not
    move."""
    t = dict(tile_n=16, stages=4, split_k=4, swap_ab=1)
    p = inputs.make_problem(8, 2048, 4096, "e4m3", "token_channel", act="silu", bias=True,
                            outlier_frac=0.01, seed=33)
    d = to_device(p)
    _noalloc_call(p, t, d)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc_call(p, t, d)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    assert_close_rms(bits(d["Y"].cpu()), oracle.linear(p))


def test_noalloc_rejects_problems_beyond_its_scratch():
    # a 32-way split of a 12288 x 4096 FP8 layer at tile_n 32 needs far
    # more split-K scratch than the fixed array holds
    p = inputs.make_problem(32, 12288, 4096, "e4m3", "token_channel", seed=1)
    prob = eg.make_problem(p.M, p.N, p.K, "e4m3", "token_channel")
    t = eg.make_tuning(tile_n=32, stages=4, split_k=32, swap_ab=1)
    d = to_device(p)
    args = eg.eg_args(d["A"].data_ptr(), d["W"].data_ptr(), d["s_a"].data_ptr(),
                      d["s_w"].data_ptr(), None, None, d["Y"].data_ptr(), p.K, p.K, 0, p.N)
    s = eg.eg_linear_noalloc(prob, t, args, None)
    assert s == eg.EG_ERR_UNSUPPORTED
    assert "scratch" in eg.last_error_detail()


@pytest.mark.parametrize("dtype,scale", [("int8", "token_channel"), ("e4m3", "block")])
def test_noalloc_rejects_two_kernel_gated_units(dtype, scale):
    """INT8 and Block_FP8 gated units need an [M][2N] accumulator buffer,
    which only a plan holds."""
    p = inputs.make_gated_problem(4, 256, 512, dtype, scale, act="silu", seed=2)
    prob = eg.make_problem(p.M, p.N, p.K, dtype, scale, "silu", eg.EG_EPI_GATED)
    d = to_device(p)
    args = eg.eg_args(d["A"].data_ptr(), d["W"].data_ptr(), d["s_a"].data_ptr(),
                      d["s_w"].data_ptr(), None, None, d["Y"].data_ptr(), p.K, p.K, 0, p.N)
    s = eg.eg_linear_noalloc(prob, None, args, None)
    assert s == eg.EG_ERR_UNSUPPORTED
    assert "accumulator buffer" in eg.last_error_detail()
