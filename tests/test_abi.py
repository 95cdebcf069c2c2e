"""The C ABI without a GPU: the library builds and loads, exports every
function include/eg.h declares, and rejects bad problems before touching a
device."""
import ctypes

import pytest
import torch

import epilogue_tcgen05_tmem_gb300 as eg
from epilogue_tcgen05_tmem_gb300 import _build
from tests._gpu_helpers import header_functions


@pytest.fixture(scope="module")
def L():
    _build.build()
    return eg.lib()


def test_exports_every_declared_function(L):
    names = header_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(eg.EXPORTED)


def test_status_strings(L):
    for s in range(7):
        assert eg.status_string(s).startswith("EG_")
    assert eg.status_string(99) == "EG_ERR_UNKNOWN"


BAD = [
    (dict(M=-1, N=8, K=64), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, dtype="bf16", scale="token_channel"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, dtype="e4m3", scale="none"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, dtype="int8", scale="block"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=192, dtype="e4m3", scale="block"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=60), eg.EG_ERR_INVALID_ARG),            # 120 bytes: not 16-aligned
    (dict(M=4, N=8, K=136, dtype="e4m3", scale="token_channel"), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=133152, dtype="int8", scale="token_channel"), eg.EG_ERR_UNSUPPORTED),
    (dict(M=4, N=8, K=64, flags=eg.EG_EPI_RESIDUAL | eg.EG_EPI_RESIDUAL_PRE_ACT), eg.EG_ERR_INVALID_ARG),
    (dict(M=4, N=8, K=64, flags=1 << 9), eg.EG_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("kw,status", BAD)
def test_invalid_problems_rejected_before_device(L, kw, status):
    kw = dict(kw)
    flags = kw.pop("flags", 0)
    p = eg.make_problem(flags=flags, **kw)
    s, h = eg.eg_plan_create(p)
    assert s == status and h is None
    assert eg.last_error_detail()


def test_invalid_activation(L):
    p = eg.make_problem(4, 8, 64)
    p.act = 9
    s, _ = eg.eg_plan_create(p)
    assert s == eg.EG_ERR_INVALID_ARG


def test_null_arguments(L):
    assert L.eg_plan_create(None, None, None) == eg.EG_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.eg_plan_create(None, None, ctypes.byref(h)) == eg.EG_ERR_INVALID_ARG
    assert L.eg_plan_destroy(None) == eg.EG_OK
    assert L.eg_plan_run(None, None, None) == eg.EG_ERR_INVALID_ARG
    assert L.eg_plan_device_status(None) == eg.EG_ERR_INVALID_ARG
    assert L.eg_plan_last_launch_count(None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_problem_without_device_reports_cuda_error(L):
    s, h = eg.eg_plan_create(eg.make_problem(4, 8, 64))
    assert s == eg.EG_ERR_CUDA and h is None
    assert "cuda" in eg.last_error_detail().lower()


def test_plan_class_raises_loudly(L):
    with pytest.raises(eg.EgError):
        eg.Plan(-1, 8, 64)
