"""GB300 (sm_103a) fused scaled linear layer: thin Python binding of the C ABI.

Every function here marshals arguments into ``libeg.so`` (``include/eg.h``);
every step of the computation runs in that library's CUDA kernels.  There is
no fallback: when the library is missing or fails to load, the calls raise.
Build it with ``__graft_entry__.build()`` (or ``python -m
epilogue_tcgen05_tmem_gb300._build``).

Names follow the C ABI: ``eg_plan_create``, ``eg_plan_run``,
``eg_plan_run_unfused``, ``eg_plan_destroy``, ... and a small ``Plan`` class
that takes torch tensors and passes their device pointers.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libeg.so")

# eg_status
EG_OK, EG_ERR_INVALID_ARG, EG_ERR_UNSUPPORTED, EG_ERR_NO_MEMORY, EG_ERR_CUDA, \
    EG_ERR_DEVICE_TIMEOUT, EG_ERR_NOT_TUNED = range(7)
# eg_in_dtype / eg_scale_mode / eg_act
DTYPES = {"bf16": 0, "e4m3": 1, "int8": 2}
SCALES = {"none": 0, "token_channel": 1, "block": 2}
ACTS = {"none": 0, "relu": 1, "gelu_erf": 2, "gelu_tanh": 3, "silu": 4}
EG_EPI_BIAS, EG_EPI_RESIDUAL, EG_EPI_RESIDUAL_PRE_ACT, EG_OUT_DEBUG_ACCUM, EG_RUN_GRAPH, \
    EG_RUN_PDL, EG_RUN_QUANT_A, EG_OUT_F16, EG_OUT_E4M3, EG_EPI_GATED = \
    1, 2, 4, 8, 16, 32, 64, 128, 256, 512
OUTS = {"bf16": 0, "f16": EG_OUT_F16, "e4m3": EG_OUT_E4M3}

EXPORTED = ("eg_plan_create", "eg_plan_workspace_bytes", "eg_plan_get_tuning", "eg_plan_run",
            "eg_plan_run_unfused", "eg_plan_device_status", "eg_plan_destroy",
            "eg_plan_last_launch_count", "eg_plan_set_test_stall", "eg_plan_get_launch",
            "eg_plan_set_trace", "eg_status_string", "eg_last_error_detail",
            "eg_linear_noalloc", "eg_quantize_rows")
EG_TRACE_POINTS = 16
TRACE_POINT_NAMES = ("start", "setup", "first_tma", "first_operands", "last_commit",
                     "first_acc", "epilogue_done", "end", "pre_issued", "last_load",
                     "last_acc", "partial_out", "arrived", "reduced", "store_begin",
                     "unused15")


class eg_problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_int32), ("act", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class eg_tuning(ctypes.Structure):
    _fields_ = [("tile_n", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("swap_ab", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("cluster_reduce", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32)]

    def as_dict(self):
        return {"tile_n": self.tile_n, "stages": self.stages, "split_k": self.split_k,
                "swap_ab": self.swap_ab, "stream_k": self.stream_k,
                "cluster_reduce": self.cluster_reduce, "cta_pair": self.cta_pair}


class eg_args(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("W", ctypes.c_void_p), ("s_a", ctypes.c_void_p),
                ("s_w", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p),
                ("Y", ctypes.c_void_p), ("lda", ctypes.c_int64), ("ldw", ctypes.c_int64),
                ("ldr", ctypes.c_int64), ("ldy", ctypes.c_int64), ("s_y", ctypes.c_void_p)]


class eg_launch_info(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("units", ctypes.c_int32),
                ("blocks_per_sm", ctypes.c_int32), ("regs_per_thread", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class EgError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status
        self.detail = detail


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libeg.so; raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                                  "(run __graft_entry__.build())")
            L = ctypes.CDLL(LIB_PATH)
            vp = ctypes.c_void_p
            L.eg_plan_create.argtypes = [ctypes.POINTER(eg_problem), ctypes.POINTER(eg_tuning),
                                         ctypes.POINTER(vp)]
            L.eg_plan_workspace_bytes.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
            L.eg_plan_get_tuning.argtypes = [vp, ctypes.POINTER(eg_tuning)]
            L.eg_plan_run.argtypes = [vp, ctypes.POINTER(eg_args), vp]
            L.eg_plan_run_unfused.argtypes = [vp, ctypes.POINTER(eg_args), vp, vp, vp]
            L.eg_plan_device_status.argtypes = [vp]
            L.eg_plan_destroy.argtypes = [vp]
            L.eg_plan_last_launch_count.argtypes = [vp]
            L.eg_plan_last_launch_count.restype = ctypes.c_int32
            L.eg_plan_set_test_stall.argtypes = [vp, ctypes.c_uint64, ctypes.c_int32]
            L.eg_plan_get_launch.argtypes = [vp, ctypes.POINTER(eg_launch_info)]
            L.eg_plan_set_trace.argtypes = [vp, vp, ctypes.c_int32]
            L.eg_linear_noalloc.argtypes = [ctypes.POINTER(eg_problem), ctypes.POINTER(eg_tuning),
                                            ctypes.POINTER(eg_args), vp]
            L.eg_linear_noalloc.restype = ctypes.c_int
            L.eg_quantize_rows.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int32, vp, ctypes.c_int64, vp, vp]
            L.eg_quantize_rows.restype = ctypes.c_int
            for f in ("eg_plan_create", "eg_plan_workspace_bytes", "eg_plan_get_tuning",
                      "eg_plan_run", "eg_plan_run_unfused", "eg_plan_device_status",
                      "eg_plan_destroy", "eg_plan_set_test_stall", "eg_plan_get_launch",
                      "eg_plan_set_trace"):
                getattr(L, f).restype = ctypes.c_int
            L.eg_status_string.argtypes = [ctypes.c_int]
            L.eg_status_string.restype = ctypes.c_char_p
            L.eg_last_error_detail.argtypes = []
            L.eg_last_error_detail.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().eg_status_string(s).decode()


def last_error_detail() -> str:
    return lib().eg_last_error_detail().decode()


def _check(status: int):
    if status != EG_OK:
        raise EgError(status, last_error_detail())


def make_problem(M, N, K, dtype="bf16", scale="none", act="none", flags=0) -> eg_problem:
    return eg_problem(M, N, K, DTYPES[dtype], SCALES[scale], ACTS[act], flags)


def make_tuning(tile_n, stages, split_k, swap_ab, stream_k=0, cluster_reduce=0,
                cta_pair=0) -> eg_tuning:
    return eg_tuning(tile_n, stages, split_k, int(bool(swap_ab)), stream_k, int(bool(cluster_reduce)),
                     int(bool(cta_pair)))


# ------------------------------------------------------ C-ABI functions ---

def eg_plan_create(problem: eg_problem, tuning: eg_tuning | None = None):
    """Returns (status, plan handle or None)."""
    h = ctypes.c_void_p()
    s = lib().eg_plan_create(ctypes.byref(problem),
                             ctypes.byref(tuning) if tuning is not None else None,
                             ctypes.byref(h))
    return s, (h.value if s == EG_OK else None)


def eg_plan_run(plan, args: eg_args, stream: int | None) -> int:
    return lib().eg_plan_run(plan, ctypes.byref(args), stream)


def eg_plan_run_unfused(plan, args: eg_args, t1: int, t2: int, stream: int | None) -> int:
    return lib().eg_plan_run_unfused(plan, ctypes.byref(args), t1, t2, stream)


def eg_linear_noalloc(problem: eg_problem, tuning: eg_tuning | None, args: eg_args,
                      stream: int | None) -> int:
    """One call that allocates no device memory (see include/eg.h): for
    callers that cannot allocate while they run the layer."""
    return lib().eg_linear_noalloc(ctypes.byref(problem),
                                   ctypes.byref(tuning) if tuning is not None else None,
                                   ctypes.byref(args), stream)


def eg_quantize_rows(x: int, M: int, K: int, ldx: int, dtype: int, q: int, ldq: int, s: int,
                     stream: int | None) -> int:
    return lib().eg_quantize_rows(x, M, K, ldx, dtype, q, ldq, s, stream)


def quantize_rows(x, dtype: str, stream=None):
    """Per-token quantisation of bf16 activations x [M, K] (torch CUDA
    tensor): returns (codes [M, K] uint8 for E4M3 / int8, scales [M] float32)."""
    import torch
    M, K = x.shape
    q = torch.empty(M, K, dtype=torch.uint8 if dtype == "e4m3" else torch.int8, device=x.device)
    sc = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(eg_quantize_rows(x.data_ptr(), M, K, x.stride(0), DTYPES[dtype], q.data_ptr(), K,
                            sc.data_ptr(), Plan._stream(stream)))
    return q, sc


def eg_plan_destroy(plan) -> int:
    return lib().eg_plan_destroy(plan)


def eg_plan_device_status(plan) -> int:
    return lib().eg_plan_device_status(plan)


def eg_plan_get_tuning(plan) -> eg_tuning:
    t = eg_tuning()
    _check(lib().eg_plan_get_tuning(plan, ctypes.byref(t)))
    return t


def eg_plan_workspace_bytes(plan) -> int:
    n = ctypes.c_size_t()
    _check(lib().eg_plan_workspace_bytes(plan, ctypes.byref(n)))
    return n.value


def eg_plan_last_launch_count(plan) -> int:
    return lib().eg_plan_last_launch_count(plan)


def eg_plan_set_test_stall(plan, wait_limit_ns: int, stall_producer: int) -> int:
    """stall_producer: 0 off, 1 (or True) every CTA, 2 odd-numbered CTAs only."""
    return lib().eg_plan_set_test_stall(plan, wait_limit_ns, int(stall_producer))


# -------------------------------------------------------------- Plan -------

def _ptr(t):
    return None if t is None else t.data_ptr()


class Plan:
    """A plan for one problem; ``run`` takes torch CUDA tensors.

    A [M,K] and W [N,K] hold the input codes (torch.bfloat16, torch.uint8 for
    e4m3 codes or torch.int8), s_a/s_w float32, bias [N] and residual [M,N]
    bf16, Y [M,N] bf16 (float32/int32 in debug mode; ``out="f16"``: fp16;
    ``out="e4m3"``: uint8 codes of v / s_y, s_y a one-element float32
    tensor).  With ``quant_a`` A is bf16 and each run quantises it per token
    first (s_a is not used).  With ``gated`` (SwiGLU when act is silu) W is
    [2N, K], gate half then up half, and s_w / bias cover the 2N rows.
    """

    def __init__(self, M, N, K, dtype="bf16", scale="none", act="none", bias=False,
                 residual=False, residual_pre_act=False, debug_accum=False, graph=False,
                 pdl=False, tuning: dict | None = None, quant_a=False, out="bf16",
                 gated=False):
        flags = 0
        if bias:
            flags |= EG_EPI_BIAS
        if residual:
            flags |= EG_EPI_RESIDUAL_PRE_ACT if residual_pre_act else EG_EPI_RESIDUAL
        if debug_accum:
            flags |= EG_OUT_DEBUG_ACCUM
        if graph:
            flags |= EG_RUN_GRAPH
        if pdl:
            flags |= EG_RUN_PDL
        if quant_a:
            flags |= EG_RUN_QUANT_A
        flags |= OUTS[out]
        if gated:
            flags |= EG_EPI_GATED
        self.problem = make_problem(M, N, K, dtype, scale, act, flags)
        t = make_tuning(**tuning) if tuning is not None else None
        s, h = eg_plan_create(self.problem, t)
        _check(s)
        self.handle = h
        self.M, self.N, self.K = M, N, K

    @property
    def tuning(self) -> dict:
        return eg_plan_get_tuning(self.handle).as_dict()

    @property
    def workspace_bytes(self) -> int:
        return eg_plan_workspace_bytes(self.handle)

    @property
    def launch_info(self) -> dict:
        li = eg_launch_info()
        _check(lib().eg_plan_get_launch(self.handle, ctypes.byref(li)))
        return li.as_dict()

    def set_trace(self, buf=None):
        """Record a per-CTA timeline into ``buf`` (int64 CUDA tensor of
        [ctas, EG_TRACE_POINTS]); None turns tracing off."""
        if buf is None:
            _check(lib().eg_plan_set_trace(self.handle, None, 0))
        else:
            _check(lib().eg_plan_set_trace(self.handle, buf.data_ptr(), buf.shape[0]))

    def args(self, A, W, Y, s_a=None, s_w=None, bias=None, residual=None, s_y=None) -> eg_args:
        return eg_args(_ptr(A), _ptr(W), _ptr(s_a), _ptr(s_w), _ptr(bias), _ptr(residual),
                       _ptr(Y), A.stride(0) if A is not None else 0,
                       W.stride(0) if W is not None else 0,
                       residual.stride(0) if residual is not None else 0, Y.stride(0), _ptr(s_y))

    @staticmethod
    def _stream(stream):
        if stream is None:
            import torch
            return torch.cuda.current_stream().cuda_stream
        return stream

    def run(self, A, W, Y, s_a=None, s_w=None, bias=None, residual=None, stream=None, s_y=None):
        _check(eg_plan_run(self.handle, self.args(A, W, Y, s_a, s_w, bias, residual, s_y),
                           self._stream(stream)))
        return Y

    def run_args(self, args: eg_args, stream=None):
        _check(eg_plan_run(self.handle, args, self._stream(stream)))

    def run_unfused(self, A, W, Y, T1, T2, s_a=None, s_w=None, bias=None, residual=None,
                    stream=None):
        _check(eg_plan_run_unfused(self.handle, self.args(A, W, Y, s_a, s_w, bias, residual),
                                   _ptr(T1), _ptr(T2), self._stream(stream)))
        return Y

    def device_status(self) -> int:
        return eg_plan_device_status(self.handle)

    def last_launch_count(self) -> int:
        return eg_plan_last_launch_count(self.handle)

    def set_test_stall(self, wait_limit_ns: int, stall_producer: int):
        _check(eg_plan_set_test_stall(self.handle, wait_limit_ns, stall_producer))

    def close(self):
        if getattr(self, "handle", None):
            eg_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
