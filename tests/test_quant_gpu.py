"""Per-token dynamic quantisation prologue on the GPU against the oracle:
codes and scales bit-exact; the quantise-then-GEMM plan against the oracle
run on the oracle's own quantisation."""
import numpy as np
import pytest
import torch

import epilogue_tcgen05_tmem_gb300 as eg
import oracle
from epilogue_tcgen05_tmem_gb300 import inputs
from tests._gpu_helpers import assert_close_rms, bits, ulp_dist

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from epilogue_tcgen05_tmem_gb300 import _build
    _build.build()
    eg.lib()


def _dev_bf16(xbits):
    return torch.from_numpy(np.ascontiguousarray(xbits)).view(torch.int16).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("dtype", ["e4m3", "int8"])
@pytest.mark.parametrize("M,K,outl", [(1, 4096, 0.01), (7, 4096, 0.01), (32, 12288, 0.0),
                                      (3, 5120, 0.0), (5, 200, 0.0), (4, 4100, 0.02),
                                      (300, 1024, 0.01)])
def test_quantize_rows_bit_exact(dtype, M, K, outl):
    xb = inputs.activations_bf16(M, K, seed=M + K, outlier_frac=outl)
    if M > 2:
        xb[1] = 0            # an all-zero row: s = 1, codes 0
    q, s = eg.quantize_rows(_dev_bf16(xb), dtype)
    torch.cuda.synchronize()
    qr, sr = oracle.quant_rows(xb, dtype)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32)), "scales"
    assert np.array_equal(q.cpu().numpy().view(np.uint8), qr), "codes"


def test_quantize_rows_strided_input():
    M, K, ld = 6, 512, 640
    full = inputs.activations_bf16(M, ld, seed=3)
    q, s = eg.quantize_rows(_dev_bf16(full)[:, :K], "e4m3")
    qr, sr = oracle.quant_rows(np.ascontiguousarray(full[:, :K]), "e4m3")
    assert np.array_equal(q.cpu().numpy(), qr) and np.array_equal(s.cpu().numpy(), sr)


def test_quantize_rows_argument_errors():
    x = torch.zeros(2, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(2, 64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(2, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert eg.eg_quantize_rows(x.data_ptr(), 2, 64, 64, eg.DTYPES["bf16"], q.data_ptr(), 64,
                               s.data_ptr(), st) == eg.EG_ERR_INVALID_ARG
    assert eg.eg_quantize_rows(x.data_ptr(), 2, 64, 32, eg.DTYPES["e4m3"], q.data_ptr(), 64,
                               s.data_ptr(), st) == eg.EG_ERR_INVALID_ARG
    assert eg.eg_quantize_rows(None, 2, 64, 64, eg.DTYPES["e4m3"], q.data_ptr(), 64,
                               s.data_ptr(), st) == eg.EG_ERR_INVALID_ARG
    assert eg.eg_quantize_rows(None, 0, 64, 64, eg.DTYPES["e4m3"], None, 64, None, st) == eg.EG_OK


def _layer(dtype, M, N, K, seed, act="silu", bias=True, residual=False):
    """The decode layer with bf16 activations: (activation bits, weights
    problem holding the oracle's quantisation of those activations)."""
    p = inputs.make_problem(M, N, K, dtype, "token_channel", act=act, bias=bias,
                            residual=residual, seed=seed, outlier_frac=0.01)
    xb = inputs.activations_bf16(M, K, seed=seed, outlier_frac=0.01)
    qa, sa = oracle.quant_rows(xb, dtype)
    p.A = qa.view(np.int8) if dtype == "int8" else qa
    p.s_a = sa
    return xb, p


@pytest.mark.parametrize("dtype,M,N,K", [("e4m3", 1, 1024, 4096), ("e4m3", 16, 2048, 4096),
                                         ("e4m3", 40, 640, 1024), ("int8", 8, 1024, 2048),
                                         ("int8", 32, 512, 12288)])
@pytest.mark.parametrize("graph", [False, True])
def test_quant_a_plan_against_oracle(dtype, M, N, K, graph):
    xb, p = _layer(dtype, M, N, K, seed=41, residual=(dtype == "int8"), bias=(dtype == "e4m3"),
                   act="silu" if dtype == "e4m3" else "none")
    plan = eg.Plan(M, N, K, dtype, "token_channel", p.act, bias=p.bias is not None,
                   residual=p.residual is not None, graph=graph, pdl=True, quant_a=True)
    X = _dev_bf16(xb)
    W = torch.from_numpy(np.ascontiguousarray(p.W)).cuda()
    sw = torch.from_numpy(p.s_w).cuda()
    b = None if p.bias is None else _dev_bf16(p.bias)
    R = None if p.residual is None else _dev_bf16(p.residual)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        plan.run(X, W, Y, None, sw, b, R)
    assert plan.last_launch_count() == 2
    torch.cuda.synchronize()
    assert plan.device_status() == eg.EG_OK
    plan.close()
    ref = oracle.linear(p)
    if dtype == "int8":
        assert ulp_dist(bits(Y.cpu()), ref).max() <= 1
    else:
        assert_close_rms(bits(Y.cpu()), ref)
    # bit-identical to quantising separately and running the plain plan
    q, s = eg.quantize_rows(X, dtype)
    plain = eg.Plan(M, N, K, dtype, "token_channel", p.act, bias=p.bias is not None,
                    residual=p.residual is not None)
    Y2 = torch.empty_like(Y)
    plain.run(q, W, Y2, s, sw, b, R)
    torch.cuda.synchronize()
    plain.close()
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))


def test_quant_a_rejections():
    with pytest.raises(eg.EgError) as ei:
        eg.Plan(4, 256, 512, "bf16", "none", quant_a=True)
    assert ei.value.status == eg.EG_ERR_INVALID_ARG
    with pytest.raises(eg.EgError) as ei:
        eg.Plan(4, 256, 512, "e4m3", "block", quant_a=True)
    assert ei.value.status == eg.EG_ERR_INVALID_ARG
    plan = eg.Plan(4, 256, 512, "e4m3", "token_channel", quant_a=True)
    X = torch.zeros(4, 512, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(256, 512, dtype=torch.uint8, device="cuda")
    sw = torch.ones(256, dtype=torch.float32, device="cuda")
    Y = torch.empty(4, 256, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(4, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(eg.EgError) as ei:
        plan.run_unfused(X, W, Y, T, T.clone(), None, sw)
    assert ei.value.status == eg.EG_ERR_UNSUPPORTED
    plan.close()
