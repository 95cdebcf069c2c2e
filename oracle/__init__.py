"""CPU oracle for the fused scaled linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  It shares no code with the CUDA
path and never imports it.  The arithmetic lives in plain C
(``eg_oracle.c``, float64, no FMA contraction); this module only builds that
library with gcc and marshals numpy arrays into it.

Every function of the C library is pinned by ``tests/test_oracle_pins.py``
against facts fixed by the pages and by mathematics (closed forms, library
routines on special cases, brute force, split-K and swap-AB invariants, the
E4M3 code table, round-to-nearest-even tie cases).  Parity is pinned for all
of it; nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "eg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"bf16": 0, "e4m3": 1, "int8": 2}
SCALES = {"none": 0, "token_channel": 1, "block": 2}
ACTS = {"none": 0, "relu": 1, "gelu_erf": 2, "gelu_tanh": 3, "silu": 4}
BIAS, RESIDUAL, RESIDUAL_PRE_ACT, OUT_F16, OUT_E4M3 = 1, 2, 4, 8, 16


class _Problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_int32),
                ("act", ctypes.c_int32), ("flags", ctypes.c_uint32), ("s_y", ctypes.c_float)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, float64, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                               os.path.getmtime(os.path.join(_HERE, "eg_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            vp = ctypes.c_void_p
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_double.restype = ctypes.c_double
            L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_double.restype = ctypes.c_double
            L.orc_bf16_from_double.argtypes = [ctypes.c_double]
            L.orc_bf16_from_double.restype = ctypes.c_uint16
            L.orc_act.argtypes = [ctypes.c_int32, ctypes.c_double]
            L.orc_act.restype = ctypes.c_double
            L.orc_linear.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            L.orc_linear_naive.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            L.orc_linear_points.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_int64, vp, vp, ctypes.c_int]
            L.orc_accum_splitk.argtypes = [P, vp, vp, vp, vp, ctypes.c_int64,
                                           ctypes.c_int64, vp, vp]
            L.orc_default_threads.argtypes = []
            L.orc_linear_gated.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            L.orc_linear_gated.restype = ctypes.c_int
            L.orc_quant_rows.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int32, vp, ctypes.c_int64, vp]
            L.orc_quant_rows.restype = ctypes.c_int
            L.orc_e4m3_from_float.argtypes = [ctypes.c_float]
            L.orc_e4m3_from_float.restype = ctypes.c_uint8
            L.orc_e4m3_from_double.argtypes = [ctypes.c_double]
            L.orc_e4m3_from_double.restype = ctypes.c_uint8
            L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_double.restype = ctypes.c_double
            L.orc_f16_from_double.argtypes = [ctypes.c_double]
            L.orc_f16_from_double.restype = ctypes.c_uint16
            for f in ("orc_linear", "orc_linear_naive", "orc_linear_points",
                      "orc_accum_splitk", "orc_default_threads"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def _problem(p, flags):
    return _Problem(p.M, p.N, p.K, DTYPES[p.dtype], SCALES[p.scale], ACTS[p.act], flags,
                    float(getattr(p, "s_y", 1.0)))


def _flags(p):
    f = 0
    if p.bias is not None:
        f |= BIAS
    if p.residual is not None:
        f |= RESIDUAL_PRE_ACT if p.residual_pre_act else RESIDUAL
    out = getattr(p, "out", "bf16")
    if out == "f16":
        f |= OUT_F16
    elif out == "e4m3":
        f |= OUT_E4M3
    return f


_ELT = {"bf16": np.uint16, "e4m3": np.uint8, "int8": np.int8}


def _arrays(p):
    e = _ELT[p.dtype]
    return (_c(p.A, e), _c(p.W, e), _c(p.s_a, np.float32), _c(p.s_w, np.float32),
            _c(p.bias, np.uint16), _c(p.residual, np.uint16))


def linear(p, nthreads: int = 0, want_acc: bool = False, naive: bool = False):
    """Y (bf16 bits [M,N]: fp16 bits, or E4M3 codes as uint8, when ``p.out``
    says so); with want_acc also the float64 accumulator and, for INT8, the
    exact int64 accumulator.  ``p`` is any object with the fields
    of a problem (M, N, K, dtype, scale, act, A, W, s_a, s_w, bias, residual,
    residual_pre_act)."""
    A, W, sa, sw, b, r = _arrays(p)
    Y = np.zeros((p.M, p.N), np.uint16)
    acc = np.zeros((p.M, p.N), np.float64) if want_acc else None
    acc64 = np.zeros((p.M, p.N), np.int64) if (want_acc and p.dtype == "int8") else None
    pr = _problem(p, _flags(p))
    if naive:
        rc = lib().orc_linear_naive(ctypes.byref(pr), _ptr(A), _ptr(W), _ptr(sa), _ptr(sw),
                                    _ptr(b), _ptr(r), _ptr(Y), _ptr(acc), _ptr(acc64))
    else:
        rc = lib().orc_linear(ctypes.byref(pr), _ptr(A), _ptr(W), _ptr(sa), _ptr(sw),
                              _ptr(b), _ptr(r), _ptr(Y), _ptr(acc), _ptr(acc64), nthreads)
    if rc:
        raise ValueError("oracle rejected the problem")
    if getattr(p, "out", "bf16") == "e4m3":
        Y = Y.astype(np.uint8)
    if want_acc:
        return Y, acc, acc64
    return Y


def linear_points(p, ms, ns, nthreads: int = 0):
    """(Y bits, float64 acc) at the given output coordinates."""
    A, W, sa, sw, b, r = _arrays(p)
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    Y = np.zeros(len(ms), np.uint16)
    acc = np.zeros(len(ms), np.float64)
    pr = _problem(p, _flags(p))
    rc = lib().orc_linear_points(ctypes.byref(pr), _ptr(A), _ptr(W), _ptr(sa), _ptr(sw),
                                 _ptr(b), _ptr(r), _ptr(ms), _ptr(ns), len(ms),
                                 _ptr(Y), _ptr(acc), nthreads)
    if rc:
        raise ValueError("oracle rejected the points")
    if getattr(p, "out", "bf16") == "e4m3":
        Y = Y.astype(np.uint8)
    return Y, acc


def accum_splitk(p, S: int, kunit: int):
    A, W, sa, sw, _, _ = _arrays(p)
    acc = np.zeros((p.M, p.N), np.float64)
    acc64 = np.zeros((p.M, p.N), np.int64) if p.dtype == "int8" else None
    pr = _problem(p, 0)
    rc = lib().orc_accum_splitk(ctypes.byref(pr), _ptr(A), _ptr(W), _ptr(sa), _ptr(sw),
                                S, kunit, _ptr(acc), _ptr(acc64))
    if rc:
        raise ValueError("oracle rejected the split")
    return acc, acc64


def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(bits)


def e4m3_to_double(code: int) -> float:
    return lib().orc_e4m3_to_double(code)


def bf16_from_double(v: float) -> int:
    return lib().orc_bf16_from_double(v)


def act(name: str, v: float) -> float:
    return lib().orc_act(ACTS[name], v)


def default_threads() -> int:
    return lib().orc_default_threads()


def quant_rows(x_bits, dtype: str):
    """Per-token dynamic quantisation of bf16 activations (bits [M, K]):
    (codes uint8 [M, K] -- E4M3 codes or int8 two's complement -- and
    float32 scales [M])."""
    x = np.ascontiguousarray(x_bits, np.uint16)
    M, K = x.shape
    q = np.zeros((M, K), np.uint8)
    sc = np.zeros(M, np.float32)
    rc = lib().orc_quant_rows(_ptr(x), M, K, K, DTYPES[dtype], _ptr(q), K, _ptr(sc))
    if rc:
        raise ValueError("oracle rejected the quantisation")
    return q, sc


def e4m3_from_float(v: float) -> int:
    return lib().orc_e4m3_from_float(v)


def e4m3_from_double(v: float) -> int:
    return lib().orc_e4m3_from_double(v)


def f16_to_double(bits: int) -> float:
    return lib().orc_f16_to_double(bits)


def f16_from_double(v: float) -> int:
    return lib().orc_f16_from_double(v)


def linear_gated(p, nthreads: int = 0):
    """Gated output Y [M, N] (bf16 bits, or the format ``p.out`` names) of a
    problem whose W holds 2N rows (gate half, then up half); ``p.N`` is the
    output width N, s_w / bias cover the 2N rows."""
    A, W, sa, sw, b, r = _arrays(p)
    Y = np.zeros((p.M, p.N), np.uint16)
    pr = _problem(p, _flags(p))
    rc = lib().orc_linear_gated(ctypes.byref(pr), _ptr(A), _ptr(W), _ptr(sa), _ptr(sw),
                                _ptr(b), _ptr(r), _ptr(Y), nthreads)
    if rc:
        raise ValueError("oracle rejected the gated problem")
    if getattr(p, "out", "bf16") == "e4m3":
        Y = Y.astype(np.uint8)
    return Y
