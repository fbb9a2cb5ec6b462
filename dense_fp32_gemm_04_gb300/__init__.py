"""GB300 (sm_103a) single-precision GEMM: C = alpha * A @ B + beta * C, row-major FP32.

Python binding over the library's C ABI (``include/sgemm.h``), by ctypes.
Everything here is argument marshalling: pointers, leading dimensions and the
CUDA stream go to ``sgemm_run`` unchanged; every step of the computation runs
in the library's CUDA kernels. PyTorch only supplies device memory and
streams. There is no fallback: if the compiled library is missing, the calls
raise.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import inputs  # noqa: F401  (seeded synthetic operands; no GEMM arithmetic)

_PKG = os.path.dirname(os.path.abspath(__file__))
# SGEMM_GB300_DEBUG_CHECKS=1 loads the debug build, whose kernels check the indices
# of their accesses (python -m dense_fp32_gemm_04_gb300._build --debug builds it).
LIB_PATH = os.path.join(_PKG, "_lib", "libsgemm_gb300_debug.so" if os.environ.get("SGEMM_GB300_DEBUG_CHECKS") == "1"
                        else "libsgemm_gb300.so")

SGEMM_OK = 0
SGEMM_ERR_INVALID_VALUE = 1
SGEMM_ERR_ARCH = 2
SGEMM_ERR_ALLOC = 3
SGEMM_ERR_LAUNCH = 4
SGEMM_ERR_TIMEOUT = 5
SGEMM_ERR_CUDA = 6
SGEMM_ERR_NOT_SUPPORTED = 7
SGEMM_ERR_INDEX = 8

MATH_FP32 = 0
MATH_TF32 = 1

KERNEL_NONE, KERNEL_SCALE, KERNEL_FFMA, KERNEL_TF32 = 0, 1, 2, 3

OPT_FORCE_CONFIG = 1
OPT_FORCE_SPLITS = 2
OPT_WAIT_TIMEOUT_NS = 3
OPT_INJECT_SKIP = 4
OPT_LOG = 5
OPT_SKEW_NS = 6
OPT_FORCE_TRANSPOSE_A = 7
OPT_FORCE_STREAMK = 8
OPT_FORCE_TF32_KERNEL = 9
OPT_FORCE_REPACK_C = 10
OPT_CLUSTER_SPLIT = 11


class Plan(ctypes.Structure):
    """Mirror of ``sgemm_plan_t``."""

    _fields_ = [(n, ctypes.c_int) for n in (
        "kernel", "config", "bm", "bn", "bk", "stages", "threads", "ctas_per_sm", "splits",
        "tiles_m", "tiles_n", "units", "grid", "repack_a", "repack_b", "vec_c", "math_mode",
        "launches")] + [("workspace_bytes", ctypes.c_longlong), ("transpose_a", ctypes.c_int),
                        ("sk_tiles", ctypes.c_int), ("sk_grid", ctypes.c_int), ("repack_c", ctypes.c_int),
                        ("cluster_split", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


_lock = threading.Lock()
_lib = None

_I, _F, _P, _LL = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_longlong
_SIGNATURES = {
    "sgemm_create": ([ctypes.POINTER(_P)], _I),
    "sgemm_create_for_device": ([_I, ctypes.POINTER(_P)], _I),
    "sgemm_destroy": ([_P], _I),
    "sgemm_run": ([_P, _I, _I, _I, _F, _P, _I, _P, _I, _F, _P, _I, _P], _I),
    "sgemm_run_host": ([_P, _I, _I, _I, _F, _P, _I, _P, _I, _F, _P, _I, _P], _I),
    "sgemm_set_math_mode": ([_P, _I], _I),
    "sgemm_get_math_mode": ([_P, ctypes.POINTER(_I)], _I),
    "sgemm_set_option": ([_P, _I, _LL], _I),
    "sgemm_check_device_status": ([_P, _P, ctypes.POINTER(_I)], _I),
    "sgemm_plan": ([_I, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(Plan)], _I),
    "sgemm_last_plan": ([_P, ctypes.POINTER(Plan)], _I),
    "sgemm_reserve": ([_P, _LL], _I),
    "sgemm_config_count": ([], _I),
    "sgemm_config_info": ([_I, ctypes.POINTER(Plan)], _I),
    "sgemm_status_string": ([_I], ctypes.c_char_p),
    "sgemm_run_splitk_static": ([_I, _I, _I, _F, _P, _I, _P, _I, _F, _P, _I, _I, _P, _P], _I),
    "sgemm_run_min2": ([_P, _I, _I, _I, _F, _P, _I, _P, _I, _F, _P, _I, _P, _P, _P], _I),
    "sgemm_ladder_run": ([_I, _I, _I, _I, _F, _P, _P, _F, _P, _P], _I),
}

STATIC_SCRATCH_BYTES = 32 << 20


def library():
    """The loaded C library (loads it on first use; raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library not built ({LIB_PATH} missing); run __graft_entry__.build() "
                    "or python -m dense_fp32_gemm_04_gb300._build")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().sgemm_status_string(status).decode()


def _check(status: int, what: str):
    if status != SGEMM_OK:
        raise SgemmError(status, what)


def plan(M, N, K, lda=None, ldb=None, ldc=None, align_flags=7, num_sms=152, math_mode=MATH_FP32) -> Plan:
    """Host-only: the plan ``sgemm_run`` would use on a GPU with ``num_sms`` SMs (no GPU needed)."""
    p = Plan()
    lda = max(1, K) if lda is None else lda
    ldb = max(1, N) if ldb is None else ldb
    ldc = max(1, N) if ldc is None else ldc
    _check(library().sgemm_plan(M, N, K, lda, ldb, ldc, align_flags, num_sms, math_mode, ctypes.byref(p)),
           "sgemm_plan")
    return p


def run_splitk_static(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, splits, device_status=None, stream=None) -> int:
    """Split-K SGEMM that allocates nothing (static 32 MiB scratch); raw device pointers.

    For callers that cannot call cudaMalloc. Returns the C-ABI status (no
    exception). ``stream`` is a torch stream, a raw handle or None (current
    torch stream).
    """
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return library().sgemm_run_splitk_static(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, splits,
                                             device_status, s)


def ladder_run(rung, A, B, C, alpha=1.0, beta=0.0, stream=None) -> int:
    """One rung of the pages' kernel ladder (context kernels) on packed torch CUDA tensors; returns the status."""
    import torch

    M, K = A.shape
    N = B.shape[1]
    for t, r, c, name in ((A, M, K, "A"), (B, K, N, "B"), (C, M, N, "C")):
        if not t.is_contiguous() or tuple(t.shape) != (r, c) or t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a packed {r} x {c} float32 CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return library().sgemm_ladder_run(rung, M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), s)


def configs():
    """The tile-config table rows, as plans."""
    lib = library()
    out = []
    for i in range(lib.sgemm_config_count()):
        p = Plan()
        _check(lib.sgemm_config_info(i, ctypes.byref(p)), "sgemm_config_info")
        out.append(p)
    return out


def _matrix_arg(t, rows, cols, name):
    """(pointer, leading dimension) of a row-major 2-D float32 CUDA tensor."""
    import torch

    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.float32 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (use run_host for host operands)")
    if tuple(t.shape) != (rows, cols):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {(rows, cols)}")
    if rows > 0 and cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with unit column stride")
    ld = t.stride(0) if rows > 1 else max(1, cols)
    return t.data_ptr(), max(ld, 1)


class Sgemm:
    """A library handle bound to one CUDA device (owns workspace and staging buffers)."""

    def __init__(self, device: int = None):
        import torch

        if device is None:
            device = torch.cuda.current_device()
        self.device = device
        h = ctypes.c_void_p()
        _check(library().sgemm_create_for_device(device, ctypes.byref(h)), "sgemm_create_for_device")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            library().sgemm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def _stream(self, stream):
        import torch

        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))

    def run(self, A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """C = alpha * A @ B + beta * C in place, asynchronously on ``stream`` (torch CUDA tensors)."""
        M, K = A.shape
        N = B.shape[1]
        pa, lda = _matrix_arg(A, M, K, "A")
        pb, ldb = _matrix_arg(B, K, N, "B")
        pc, ldc = _matrix_arg(C, M, N, "C")
        _check(library().sgemm_run(self._h, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, self._stream(stream)),
               "sgemm_run")
        return C

    def run_min2(self, A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """C = alpha * A @ B + beta * C in place, plus the two smallest elements of C.

        Returns device tensors ``(vals[2], ij[4])`` = values and {row0, col0, row1, col1}.
        """
        import torch

        M, K = A.shape
        N = B.shape[1]
        pa, lda = _matrix_arg(A, M, K, "A")
        pb, ldb = _matrix_arg(B, K, N, "B")
        pc, ldc = _matrix_arg(C, M, N, "C")
        vals = torch.empty(2, dtype=torch.float32, device=C.device)
        ij = torch.empty(4, dtype=torch.int32, device=C.device)
        _check(library().sgemm_run_min2(self._h, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, vals.data_ptr(),
                                        ij.data_ptr(), self._stream(stream)), "sgemm_run_min2")
        return vals, ij

    def run_ptr(self, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
        """Direct C-ABI call with raw device pointers; returns the status (no exception)."""
        return library().sgemm_run(self._h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, self._stream(stream))

    def run_host(self, A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """Host-operand variant (numpy arrays or CPU tensors, ideally pinned); C updated in place."""
        import numpy as np

        def host(x, rows, cols, name):
            if isinstance(x, np.ndarray):
                if x.dtype != np.float32 or x.ndim != 2 or x.shape != (rows, cols):
                    raise TypeError(f"{name} must be a {rows} x {cols} float32 array")
                if rows > 0 and cols > 1 and x.strides[1] != 4:
                    raise ValueError(f"{name} must have unit column stride")
                return x.ctypes.data, (x.strides[0] // 4 if rows > 1 else max(1, cols))
            import torch

            if not isinstance(x, torch.Tensor) or x.is_cuda or x.dtype != torch.float32 or x.dim() != 2:
                raise TypeError(f"{name} must be a host float32 matrix")
            if tuple(x.shape) != (rows, cols):
                raise ValueError(f"{name} has the wrong shape")
            if rows > 0 and cols > 1 and x.stride(1) != 1:
                raise ValueError(f"{name} must have unit column stride")
            return x.data_ptr(), (x.stride(0) if rows > 1 else max(1, cols))

        M, K = A.shape
        N = B.shape[1]
        pa, lda = host(A, M, K, "A")
        pb, ldb = host(B, K, N, "B")
        pc, ldc = host(C, M, N, "C")
        _check(library().sgemm_run_host(self._h, M, N, K, alpha, pa, max(lda, 1), pb, max(ldb, 1), beta, pc,
                                        max(ldc, 1), self._stream(stream)), "sgemm_run_host")
        return C

    def set_math_mode(self, mode: int):
        _check(library().sgemm_set_math_mode(self._h, mode), "sgemm_set_math_mode")

    def math_mode(self) -> int:
        m = ctypes.c_int()
        _check(library().sgemm_get_math_mode(self._h, ctypes.byref(m)), "sgemm_get_math_mode")
        return m.value

    def set_option(self, option: int, value: int):
        _check(library().sgemm_set_option(self._h, option, int(value)), "sgemm_set_option")

    def check_device_status(self, stream=None):
        """Synchronize ``stream`` and return (status, raw device code); clears the code."""
        code = ctypes.c_int()
        st = library().sgemm_check_device_status(self._h, self._stream(stream), ctypes.byref(code))
        return st, code.value

    def reserve(self, workspace_bytes: int):
        """Grow the device workspace now (so that later calls can be captured into a CUDA graph)."""
        _check(library().sgemm_reserve(self._h, int(workspace_bytes)), "sgemm_reserve")

    def last_plan(self) -> Plan:
        p = Plan()
        _check(library().sgemm_last_plan(self._h, ctypes.byref(p)), "sgemm_last_plan")
        return p
