"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently of its own
code: a value the pages print (tests/golden/page_facts.txt), the OCP E4M3
table, a library routine on a special case (torch float64 matmul, gelu, silu;
torch's float8/bfloat16 casts), a closed form, an invariant (swap-AB, split-K)
or brute force on tiny inputs.  They are chosen so that a dropped term, a
wrong sign, a wrong index or a transposed operand in the oracle fails at
least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from epilogue_tcgen05_tmem_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    out = {}
    with open(os.path.join(GOLDEN, "page_facts.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                out[k] = v
    return out


def _torch_decode(p, arr):
    """Decode input codes with torch's own casts (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(arr))
    if p.dtype == "bf16":
        return t.view(torch.bfloat16).to(torch.float64)
    if p.dtype == "e4m3":
        return t.view(torch.float8_e4m3fn).to(torch.float64)
    return t.to(torch.float64)


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(torch.float64)


# ------------------------------------------------------------------ codecs --

def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_e4m3_ocp_table():
    with open(os.path.join(GOLDEN, "e4m3_ocp.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for code, val in rows:
        got = oracle.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    assert np.array_equal(np.isnan(r), np.isnan(got))
    ok = ~np.isnan(r)
    assert np.array_equal(r[ok], got[ok])


def test_bf16_rne_matches_torch_on_float32_values():
    # Values exact in float32: torch's float32 -> bf16 cast is round to
    # nearest even in one step, so it must agree with the oracle exactly.
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]              # finite only
    ties = (u & 0xFFFF0000) | 0x8000                   # exact half-way cases
    vals = np.concatenate([u, ties]).view(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in vals], np.uint16)
    assert np.array_equal(ref, got)


def test_bf16_rne_direct_from_double():
    # Cases where rounding through float32 first would give another answer.
    assert oracle.bf16_from_double(1 + 2**-8) == 0x3F80              # tie -> even
    assert oracle.bf16_from_double(1 + 3 * 2**-8) == 0x3F82          # tie -> even (up)
    assert oracle.bf16_from_double(1 + 2**-8 + 2**-30) == 0x3F81     # just above a tie
    assert oracle.bf16_from_double(-(1 + 2**-8 + 2**-30)) == 0xBF81
    assert oracle.bf16_from_double(1 + 2**-8 - 2**-40) == 0x3F80
    assert oracle.bf16_from_double(3.0e38) == 0x7F62
    assert oracle.bf16_from_double(3.4e38) == 0x7F80                 # past max -> inf
    assert oracle.bf16_from_double(2**-133) == 0x0001                # smallest subnormal
    assert oracle.bf16_from_double(2**-134) == 0x0000                # tie -> even (zero)
    assert oracle.bf16_from_double(-0.0) == 0x8000
    assert oracle.bf16_from_double(float("nan")) & 0x7FC0 == 0x7FC0


# ------------------------------------------------------------- activations --

def test_activations_match_torch():
    x = torch.linspace(-12, 12, 4801, dtype=torch.float64)
    F = torch.nn.functional
    refs = {"gelu_erf": F.gelu(x), "gelu_tanh": F.gelu(x, approximate="tanh"),
            "silu": F.silu(x), "relu": F.relu(x), "none": x}
    for name, ref in refs.items():
        got = torch.tensor([oracle.act(name, float(v)) for v in x], dtype=torch.float64)
        # 1 + tanh(..) cancels for large negative x: bound the absolute error
        # by a few float64 ulps of |x| there
        tol = 1e-13 * ref.abs() + 1e-15 * (1 + x.abs())
        assert torch.all((got - ref).abs() <= tol), name


def test_activation_closed_forms():
    for a in ("relu", "gelu_erf", "gelu_tanh", "silu"):
        assert oracle.act(a, 0.0) == 0.0
    assert oracle.act("relu", -3.0) == 0.0 and oracle.act("relu", 3.0) == 3.0
    assert abs(oracle.act("gelu_erf", 10.0) - 10.0) < 1e-20
    assert abs(oracle.act("gelu_erf", -10.0)) < 1e-20
    assert abs(oracle.act("gelu_erf", 1.0) - 0.5 * (1 + math.erf(1 / math.sqrt(2)))) < 1e-15
    for v in (0.3, 1.7, 5.0):      # SiLU(v) - SiLU(-v) = v ; GELU(v) - GELU(-v) = v
        assert abs(oracle.act("silu", v) - oracle.act("silu", -v) - v) < 1e-14
        assert abs(oracle.act("gelu_erf", v) - oracle.act("gelu_erf", -v) - v) < 1e-14
        assert abs(oracle.act("gelu_tanh", v) - oracle.act("gelu_tanh", -v) - v) < 1e-14


def test_gelu_tanh_constant_printed_on_page():
    c0, c1 = (float(v) for v in _facts()["gelu_tanh_constants"])
    assert abs(c0 - math.sqrt(2 / math.pi)) < 1e-8
    # the oracle uses sqrt(2/pi) and 0.044715: check one point by the formula
    v = 1.3
    ref = 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + c1 * v ** 3)))
    assert abs(oracle.act("gelu_tanh", v) - ref) < 1e-15


# ----------------------------------------------------------- contraction --

def _small(dtype, scale, M=5, N=7, K=256, **kw):
    return inputs.make_problem(M, N, K, dtype, scale, seed=3, **kw)


@pytest.mark.parametrize("dtype,scale", [("bf16", "none"), ("e4m3", "token_channel"),
                                         ("int8", "token_channel"), ("e4m3", "block")])
def test_accumulator_matches_torch_matmul(dtype, scale):
    p = _small(dtype, scale, M=9, N=130, K=384)
    _, acc, acc64 = oracle.linear(p, want_acc=True)
    a, w = _torch_decode(p, p.A), _torch_decode(p, p.W)
    if scale == "block":
        sa = torch.from_numpy(p.s_a).double()
        sw = torch.from_numpy(p.s_w).double()
        ref = torch.zeros(p.M, p.N, dtype=torch.float64)
        for kb in range(p.K // 128):
            part = a[:, kb * 128:(kb + 1) * 128] @ w[:, kb * 128:(kb + 1) * 128].T
            scale_mn = sa[:, kb][:, None] * sw[torch.arange(p.N) // 128, kb][None, :]
            ref += scale_mn * part
    else:
        ref = a @ w.T
    err = (torch.from_numpy(acc) - ref).abs().max().item()
    assert err <= 1e-12 * max(ref.abs().max().item(), 1e-30)
    if dtype == "int8":
        exact = p.A.astype(np.int64) @ p.W.astype(np.int64).T
        assert np.array_equal(acc64, exact)


def test_transposed_operand_would_fail():
    # W[n][k] = n + 1 and A[m][k] = m + 1 give acc = K (m+1)(n+1); with
    # M != N != K an A.W or A^T.W reading gives other values or shapes.
    M, N, K = 3, 5, 8
    p = _small("bf16", "none", M, N, K)
    p.A = inputs.to_bf16_bits(np.repeat(np.arange(1, M + 1, dtype=np.float64)[:, None], K, 1))
    p.W = inputs.to_bf16_bits(np.repeat(np.arange(1, N + 1, dtype=np.float64)[:, None], K, 1))
    _, acc, _ = oracle.linear(p, want_acc=True)
    ref = K * np.outer(np.arange(1, M + 1), np.arange(1, N + 1))
    assert np.array_equal(acc, ref)


def test_identity_weight():
    K = 64
    p = _small("bf16", "none", 4, K, K)
    eye = inputs.to_bf16_bits(np.eye(K))
    p.W = eye
    _, acc, _ = oracle.linear(p, want_acc=True)
    assert np.array_equal(acc, _torch_decode(p, p.A).numpy())


@pytest.mark.parametrize("dtype", ["e4m3", "int8"])
def test_all_ones_token_channel_closed_form(dtype):
    M, N, K = 4, 6, 96
    p = _small(dtype, "token_channel", M, N, K)
    one = {"e4m3": 0x38, "int8": 1}[dtype]
    p.A = np.full((M, K), one, dtype=p.A.dtype)
    p.W = np.full((N, K), one, dtype=p.W.dtype)
    p.s_a = (2.0 ** -np.arange(M)).astype(np.float32)
    p.s_w = (2.0 ** np.arange(N) / 64).astype(np.float32)
    Y, acc, _ = oracle.linear(p, want_acc=True)
    assert np.all(acc == K)
    expect = K * np.outer(p.s_a.astype(np.float64), p.s_w.astype(np.float64))
    assert np.array_equal(_bf16(Y).numpy(), expect)   # powers of two: exact in bf16


def test_block_scale_indexing_closed_form():
    # codes all 1.0; s_a[m][kb] = 2^-m, s_w[nb][kb] = (kb+1) 2^nb
    M, N, K = 3, 384, 512
    KB, NB = K // 128, N // 128
    p = _small("e4m3", "block", M, N, K)
    p.A = np.full((M, K), 0x38, np.uint8)
    p.W = np.full((N, K), 0x38, np.uint8)
    p.s_a = np.repeat((2.0 ** -np.arange(M))[:, None], KB, 1).astype(np.float32)
    p.s_w = (np.arange(1, KB + 1)[None, :] * (2.0 ** np.arange(NB))[:, None]).astype(np.float32)
    _, acc, _ = oracle.linear(p, want_acc=True)
    nb = np.arange(N) // 128
    expect = 128.0 * (2.0 ** (nb[None, :] - np.arange(M)[:, None])) * (KB * (KB + 1) / 2)
    assert np.array_equal(acc, expect)


def test_int8_worst_case_fits_int32():
    M, N, K = 2, 3, 12288
    p = _small("int8", "token_channel", M, N, K)
    p.A = np.full((M, K), 127, np.int8)
    p.W = np.full((N, K), -127, np.int8)
    _, acc, acc64 = oracle.linear(p, want_acc=True)
    assert np.all(acc64 == -(127 ** 2) * K)
    assert 127 ** 2 * K < 2 ** 31


# ---------------------------------------------------------------- epilogue --

@pytest.mark.parametrize("act", ["none", "relu", "gelu_erf", "gelu_tanh", "silu"])
@pytest.mark.parametrize("pre", [False, True])
def test_epilogue_with_zero_accumulator(act, pre):
    """A = 0 reduces the layer to act(bias[n]) + R[m][n] (or act(bias + R)):
    checks bias indexing by n, residual by (m, n), the order flag and the
    activation, against torch float64 and the round-to-nearest error bound."""
    M, N, K = 5, 9, 64
    p = _small("bf16", "none", M, N, K, act=act, bias=True, residual=True,
               residual_pre_act=pre)
    p.A = np.zeros_like(p.A)
    Y = oracle.linear(p)
    b, r = _bf16(p.bias), _bf16(p.residual)
    F = torch.nn.functional
    f = {"none": lambda x: x, "relu": F.relu, "gelu_erf": F.gelu,
         "gelu_tanh": lambda x: F.gelu(x, approximate="tanh"), "silu": F.silu}[act]
    ref = f(b[None, :] + r) if pre else f(b)[None, :] + r
    got = _bf16(Y)
    assert torch.all((got - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-30)


def test_scale_bias_act_residual_chain_special_case():
    """Token/channel scale, bias, SiLU and residual together, against torch
    float64 on decoded inputs (W = identity, so acc = A exactly)."""
    M, K = 6, 128
    p = _small("e4m3", "token_channel", M, K, K, act="silu", bias=True, residual=True)
    p.W = np.where(np.eye(K, dtype=bool), 0x38, 0).astype(np.uint8)
    Y = oracle.linear(p)
    a = _torch_decode(p, p.A)
    v = a * torch.from_numpy(p.s_a).double()[:, None] * torch.from_numpy(p.s_w).double()[None, :]
    ref = torch.nn.functional.silu(v + _bf16(p.bias)[None, :]) + _bf16(p.residual)
    got = _bf16(Y)
    assert torch.all((got - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-30)


def test_bf16_no_epilogue_is_rounded_matmul():
    p = _small("bf16", "none", 17, 33, 320)
    Y = oracle.linear(p)
    ref = _torch_decode(p, p.A) @ _torch_decode(p, p.W).T
    got = _bf16(Y)
    assert torch.all((got - ref).abs() <= 2.0 ** -8 * ref.abs())


# --------------------------------------------------------------- invariants --

@pytest.mark.parametrize("dtype,scale", [("bf16", "none"), ("e4m3", "token_channel"),
                                         ("int8", "token_channel")])
def test_swap_ab_identity(dtype, scale):
    """(W A^T)^T = A W^T: the oracle run with the operands' roles swapped gives
    the transposed accumulator bit for bit."""
    p = _small(dtype, scale, 7, 11, 256)
    _, acc, _ = oracle.linear(p, want_acc=True)
    q = _small(dtype, scale, 11, 7, 256)
    q.A, q.W, q.s_a, q.s_w = p.W, p.A, p.s_w, p.s_a
    _, acc_t, _ = oracle.linear(q, want_acc=True)
    assert np.array_equal(acc, acc_t.T)


@pytest.mark.parametrize("dtype,scale,kunit", [("bf16", "none", 64), ("e4m3", "token_channel", 128),
                                               ("int8", "token_channel", 128), ("e4m3", "block", 128)])
@pytest.mark.parametrize("S", [1, 2, 3, 5])
def test_split_k_invariance(dtype, scale, kunit, S):
    p = _small(dtype, scale, 4, 6, 640)
    _, acc, acc64 = oracle.linear(p, want_acc=True)
    sacc, sacc64 = oracle.accum_splitk(p, S, kunit)
    if dtype == "int8":
        assert np.array_equal(acc64, sacc64)
    rms = math.sqrt(float(np.mean(acc ** 2)))
    assert np.max(np.abs(acc - sacc)) <= 1e-12 * rms


def test_naive_and_threaded_agree_bitwise():
    for dtype, scale in [("bf16", "none"), ("e4m3", "token_channel"),
                         ("int8", "token_channel"), ("e4m3", "block")]:
        p = _small(dtype, scale, 3, 130, 256, act="gelu_tanh", bias=True, residual=True)
        y1, a1, _ = oracle.linear(p, want_acc=True, nthreads=3)
        y2, a2, _ = oracle.linear(p, want_acc=True, naive=True)
        assert np.array_equal(y1, y2) and np.array_equal(a1, a2)


def test_points_match_full():
    p = _small("e4m3", "token_channel", 6, 50, 256, act="silu", bias=True)
    Y, acc, _ = oracle.linear(p, want_acc=True)
    ms = np.array([0, 5, 3, 2]); ns = np.array([0, 49, 17, 2])
    yp, ap = oracle.linear_points(p, ms, ns)
    assert np.array_equal(yp, Y[ms, ns]) and np.array_equal(ap, acc[ms, ns])


def test_brute_force_python_tiny():
    """Pure-Python loops with the math module, M,N,K tiny, all flags on."""
    for act in ("gelu_erf", "gelu_tanh", "silu", "relu"):
        for pre in (False, True):
            p = _small("bf16", "none", 2, 3, 4, act=act, bias=True, residual=True,
                       residual_pre_act=pre)
            Y = oracle.linear(p)
            dec = lambda b: float(torch.tensor([int(b)], dtype=torch.int32).to(torch.int16)
                                  .view(torch.bfloat16).double().item())
            for m in range(2):
                for n in range(3):
                    s = sum(dec(p.A[m, k]) * dec(p.W[n, k]) for k in range(4))
                    s += dec(p.bias[n])
                    r = dec(p.residual[m, n])
                    f = {"relu": lambda x: max(x, 0.0),
                         "gelu_erf": lambda x: 0.5 * x * (1 + math.erf(x / math.sqrt(2))),
                         "gelu_tanh": lambda x: 0.5 * x * (1 + math.tanh(
                             math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3))),
                         "silu": lambda x: x / (1 + math.exp(-x))}[act]
                    v = f(s + r) if pre else f(s) + r
                    got = dec(Y[m, n])
                    assert abs(got - v) <= 2.0 ** -8 * abs(v) + 1e-30


def test_degenerate_shapes():
    for M, N, K in [(0, 5, 64), (3, 0, 64), (1, 1, 64), (2, 3, 0)]:
        p = inputs.make_problem(M, N, K, "bf16", bias=True, seed=0)
        Y, acc, _ = oracle.linear(p, want_acc=True)
        assert Y.shape == (M, N)
        if K == 0 and M and N:
            assert np.all(acc == 0) and np.array_equal(Y, np.tile(p.bias, (M, 1)))


def test_oracle_rejects_bad_arguments():
    p = _small("e4m3", "block", 2, 130, 200)   # K % 128 != 0 for block scaling
    with pytest.raises(ValueError):
        oracle.linear(p)


# --------------------------------------- per-token dynamic quantisation ---

def _finite_e4m3_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_encoder_inverts_the_table():
    """Every finite code survives decode -> encode (the decoder is pinned to
    the OCP table above)."""
    for c in _finite_e4m3_codes():
        v = oracle.e4m3_to_double(c)
        assert oracle.e4m3_from_float(v) == c, hex(c)


def test_e4m3_encoder_ties_to_even_and_saturates():
    """Between consecutive finite magnitudes the midpoint goes to the code
    with an even mantissa, anything off the midpoint to the nearer code;
    magnitudes at or past 448 saturate; NaN stays NaN."""
    mags = sorted({oracle.e4m3_to_double(c) for c in range(0x7F)})
    for lo, hi in zip(mags, mags[1:]):
        c_lo, c_hi = oracle.e4m3_from_float(lo), oracle.e4m3_from_float(hi)
        mid = (lo + hi) / 2  # exact in float32 (a few significant bits)
        even = c_lo if (c_lo & 1) == 0 else c_hi
        assert oracle.e4m3_from_float(mid) == even
        assert oracle.e4m3_from_float(-mid) == (even | 0x80)
        assert oracle.e4m3_from_float(np.nextafter(np.float32(mid), np.float32(0))) == c_lo
        assert oracle.e4m3_from_float(np.nextafter(np.float32(mid), np.float32(1e9))) == c_hi
    for v in (448.0, 449.0, 464.0, 1e30, float("inf")):
        assert oracle.e4m3_from_float(v) == 0x7E and oracle.e4m3_from_float(-v) == 0xFE
    assert oracle.e4m3_from_float(float("nan")) & 0x7F == 0x7F


def test_e4m3_encoder_matches_torch_on_a_dense_sweep():
    """Library cross-check: torch's float -> float8_e4m3fn conversion (round
    to nearest even) on values inside the finite range."""
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 0.01, 20000), np.ldexp(rng.uniform(-1, 1, 5000), -7)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def _bf16_bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_quant_rows_closed_forms():
    # row 0: amax 2 -> s = 2/448; x/s = 224, -448, 112, 0 (exact E4M3 values)
    # row 1: zero row -> s = 1, codes 0
    # row 2: a constant row -> every code is +448
    x = _bf16_bits([[1.0, -2.0, 0.5, 0.0], [0.0, 0.0, 0.0, 0.0], [0.25, 0.25, 0.25, 0.25]])
    q, s = oracle.quant_rows(x, "e4m3")
    assert s[0] == np.float32(2.0) / np.float32(448.0) and s[1] == 1.0
    assert s[2] == np.float32(0.25) / np.float32(448.0)
    assert list(q[0]) == [0x76, 0xFE, 0x6E, 0x00] and list(q[1]) == [0, 0, 0, 0]
    assert list(q[2]) == [0x7E] * 4
    qi, si = oracle.quant_rows(x, "int8")
    assert si[0] == np.float32(2.0) / np.float32(127.0)
    # 1 / (2/127) = 63.5 in float32 -> ties to even -> 64
    assert list(qi[0].view(np.int8)) == [64, -127, 32, 0] and list(qi[1]) == [0, 0, 0, 0]


def test_quant_rows_int8_ties_to_even():
    """amax 127 gives s = 1, so x/s = x and the rounding of exact halves shows."""
    x = _bf16_bits([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 126.5, -126.5]])
    q, s = oracle.quant_rows(x, "int8")
    assert s[0] == 1.0
    assert list(q[0].view(np.int8)) == [127, 0, 2, 2, 0, -2, 126, -126]


@pytest.mark.parametrize("dtype", ["e4m3", "int8"])
def test_quant_rows_error_bound_and_range(dtype):
    """Each dequantised code is within half a step of its input (E4M3: half a
    unit of the third mantissa bit, relative; int8: s/2), up to the float32
    rounding of x / s; the row's amax element maps to the largest code."""
    rng = np.random.default_rng(9)
    xf = (rng.normal(0, 1, (6, 700)) * np.array([1, 10, 0.01, 1e-3, 100, 3])[:, None]).astype(np.float32)
    x = _bf16_bits(xf)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q, s = oracle.quant_rows(x, dtype)
    for m in range(x.shape[0]):
        if dtype == "e4m3":
            deq = np.array([oracle.e4m3_to_double(int(c)) for c in q[m]]) * s[m]
            assert np.all(np.abs(deq - xv[m]) <= np.abs(xv[m]) * 2.0 ** -4 + s[m] * 2.0 ** -10 + 1e-30)
            assert np.max(np.abs(deq)) == pytest.approx(448.0 * s[m], rel=1e-6)
        else:
            deq = q[m].view(np.int8).astype(np.float64) * s[m]
            # half a step, plus the float32 rounding of x / s (|x/s| <= 127)
            assert np.all(np.abs(deq - xv[m]) <= s[m] * (0.5 + 127 * 2.0 ** -23))
            assert np.max(np.abs(q[m].view(np.int8).astype(int))) == 127


# --------------------------------------------------- output narrowing ---

def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)])) and np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_f16_rounding_matches_numpy_from_float64():
    """Library cross-check: numpy's float64 -> float16 conversion rounds to
    nearest even in one step (no float32 in between)."""
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 3e4, 5000),
                        rng.normal(0, 1e-5, 5000), np.ldexp(rng.uniform(-1, 1, 5000), -20),
                        np.array([65504.0, 65519.99, 65520.0, 1e6, -65520.0, 0.0, -0.0])])
    with np.errstate(over="ignore"):   # 1e6 overflows to infinity, as intended
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_from_double(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_f16_ties_to_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: even mantissa (1.0) wins;
    # 1 + 3 * 2^-11 is halfway between 1 + 2^-10 and 1 + 2^-9: 1 + 2^-9 wins
    assert oracle.f16_from_double(1 + 2.0 ** -11) == 0x3C00
    assert oracle.f16_from_double(1 + 3 * 2.0 ** -11) == 0x3C02
    assert oracle.f16_from_double(2.0 ** -25) == 0x0000          # half the smallest subnormal
    assert oracle.f16_from_double(3 * 2.0 ** -25) == 0x0002


@pytest.mark.parametrize("out", ["f16", "e4m3"])
def test_output_format_closed_form(out):
    """A = W = 1, token/channel scales 1: v = K exactly, so Y is the format's
    encoding of K (E4M3: of K / s_y)."""
    K = 256
    p = inputs.make_problem(2, 3, K, "e4m3", "token_channel", seed=1)
    p.A = np.full((2, K), 0x38, np.uint8)   # e4m3 1.0
    p.W = np.full((3, K), 0x38, np.uint8)
    p.s_a = np.ones(2, np.float32)
    p.s_w = np.ones(3, np.float32)
    p.out = out
    p.s_y = 2.0
    y = oracle.linear(p)
    if out == "f16":
        assert np.all(y == np.float16(K).view(np.uint16))
    else:
        assert y.dtype == np.uint8 and np.all(y == oracle.e4m3_from_float(K / 2.0))
        assert oracle.e4m3_to_double(int(y[0, 0])) * 2.0 == K


def test_output_formats_agree_with_bf16_path():
    """The same epilogue value rounded three ways: the fp16 and E4M3 outputs
    decode to within half a step of the bf16 output's exact value."""
    p = inputs.make_problem(5, 40, 512, "e4m3", "token_channel", act="gelu_tanh", bias=True,
                            residual=True, seed=4)
    _, acc, _ = oracle.linear(p, want_acc=True)
    yb = oracle.linear(p)
    p.out = "f16"
    yh = oracle.linear(p)
    p.out, p.s_y = "e4m3", 0.0625
    ye = oracle.linear(p)
    vb = (yb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    vh = yh.view(np.float16).astype(np.float64)
    ve = np.vectorize(oracle.e4m3_to_double)(ye.astype(int)) * 0.0625
    # bf16 keeps 8 significant bits, fp16 11, E4M3 4: each within its own
    # half step of the exact value, so within the sum of the two half steps
    assert np.all(np.abs(vh - vb) <= np.abs(vb) * (2.0 ** -8 + 2.0 ** -11) + 2.0 ** -24)
    assert np.all(np.abs(ve - vb) <= np.abs(vb) * (2.0 ** -8 + 2.0 ** -4) + 0.0625 * 2.0 ** -9)


def test_output_format_flags_rejected_together():
    p = inputs.make_problem(2, 3, 64, "bf16", seed=1)
    pr = oracle._problem(p, oracle.OUT_F16 | oracle.OUT_E4M3)
    A, W, sa, sw, b, r = oracle._arrays(p)
    Y = np.zeros((2, 3), np.uint16)
    import ctypes
    assert oracle.lib().orc_linear(ctypes.byref(pr), oracle._ptr(A), oracle._ptr(W), None, None,
                                   None, None, oracle._ptr(Y), None, None, 1) == -1


# ------------------------------------------------ gated linear unit (SwiGLU) ---

def test_gated_zero_weights_is_act_of_bias_times_bias():
    """W = 0: g = bias[n], u = bias[N + n], so y = act(bias_g) * bias_u (+ R)."""
    p = inputs.make_gated_problem(3, 40, 64, "bf16", act="silu", bias=True, residual=True, seed=2)
    p.W = np.zeros_like(p.W)
    y = oracle.linear_gated(p)
    bg = np.array([oracle.bf16_to_double(int(b)) for b in p.bias[:40]])
    bu = np.array([oracle.bf16_to_double(int(b)) for b in p.bias[40:]])
    r = np.array([[oracle.bf16_to_double(int(v)) for v in row] for row in p.residual])
    want = np.array([[oracle.bf16_from_double(oracle.act("silu", bg[n]) * bu[n] + r[m, n])
                      for n in range(40)] for m in range(3)], np.uint16)
    assert np.array_equal(y, want)


def test_gated_scales_pick_each_half():
    """A = W = 1 with distinct per-row weight scales: g = K sa sw[n],
    u = K sa sw[N + n]; a halves mix-up changes the result."""
    M, N, K = 2, 3, 128
    p = inputs.make_gated_problem(M, N, K, "e4m3", "token_channel", act="silu", seed=3)
    p.A = np.full((M, K), 0x38, np.uint8)
    p.W = np.full((2 * N, K), 0x38, np.uint8)
    p.s_a = np.array([1.0, 0.5], np.float32)
    p.s_w = np.array([0.01, 0.02, -0.03, 0.2, 0.3, 0.4], np.float32)
    y = oracle.linear_gated(p)
    for m in range(M):
        for n in range(N):
            g = K * float(p.s_a[m]) * float(p.s_w[n])
            u = K * float(p.s_a[m]) * float(p.s_w[N + n])
            assert y[m, n] == oracle.bf16_from_double(oracle.act("silu", g) * u)


def test_gated_halves_not_swapped():
    """A strongly negative gate closes the unit (g = -80: y ~ -4e-33),
    whereas the swapped unit would give silu(2.5) * (-80) ~ -186."""
    M, N, K = 1, 1, 128
    p = inputs.make_gated_problem(M, N, K, "bf16", act="silu", seed=4)
    one = np.uint16(0x3F80)  # bf16 1.0
    p.A = np.full((M, K), one, np.uint16)
    p.W = np.zeros((2, K), np.uint16)
    p.W[0, :] = np.uint16(0xBF20)  # -0.625 * 128 = -80 -> gate
    p.W[1, :] = np.uint16(0x3CA0)  # 0.01953125 * 128 = 2.5 -> up
    y = oracle.linear_gated(p)
    v = oracle.bf16_to_double(int(y[0, 0]))
    assert y[0, 0] == oracle.bf16_from_double(oracle.act("silu", -80.0) * 2.5)
    assert abs(v) < 1e-20 and abs(oracle.act("silu", 2.5) * -80.0) > 100


def test_gated_rejects_pre_activation_residual():
    p = inputs.make_gated_problem(2, 8, 64, "bf16", act="silu", residual=True, seed=5)
    p.residual_pre_act = True
    with pytest.raises(ValueError):
        oracle.linear_gated(p)
