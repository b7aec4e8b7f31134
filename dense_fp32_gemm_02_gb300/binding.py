"""ctypes binding of libsgemm.so (argument marshalling only).

Every computing function here hands pointers, sizes and a stream to the C ABI
in include/sgemm.h; no arithmetic of the GEMM happens in Python.  Importing
this module raises ImportError when the library has not been built (there is
no fallback path).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_DEBUG_BOUNDS_PATH, LIB_PATH

# SGEMM_LIBRARY=debug_bounds loads the range-checked test build instead of the
# library (a test switch; the library is always one of this package's builds)
library_path = LIB_DEBUG_BOUNDS_PATH if os.environ.get("SGEMM_LIBRARY") == "debug_bounds" \
    else LIB_PATH

if not os.path.exists(library_path):
    raise ImportError(
        f"{os.path.basename(library_path)} is not built at {library_path}; run "
        "`python -c 'import __graft_entry__ as g; g.build()'` or "
        "`python -m dense_fp32_gemm_02_gb300.build`")

lib = ctypes.CDLL(library_path)

_i, _f, _p = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
_ull, _ll, _d = ctypes.c_ulonglong, ctypes.c_longlong, ctypes.c_double

lib.sgemm.argtypes = [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]
lib.sgemm.restype = _i
lib.sgemm_host.argtypes = [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]
lib.sgemm_host.restype = _i
lib.sgemm_ex.argtypes = [_i, _i, _i, _f, _p, _i, _ll, _p, _i, _ll, _f, _p, _i, _ll, _i, _p, _ll,
                         _i, _p]
lib.sgemm_ex.restype = _i
lib.sgemm_noalloc.argtypes = [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]
lib.sgemm_noalloc.restype = _i
lib.sgemm_3xtf32.argtypes = [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]
lib.sgemm_3xtf32.restype = _i
lib.sgemm_host_3xtf32.argtypes = [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]
lib.sgemm_host_3xtf32.restype = _i
lib.sgemm_status_string.argtypes = [_i]
lib.sgemm_status_string.restype = ctypes.c_char_p
lib.sgemm_version.argtypes = []
lib.sgemm_version.restype = _i
lib.sgemm_last_cuda_error.argtypes = []
lib.sgemm_last_cuda_error.restype = _i
lib.sgemm_device_status.argtypes = [_p]
lib.sgemm_device_status.restype = _i
lib.sgemm_set_wait_timeout_ns.argtypes = [_ull]
lib.sgemm_set_wait_timeout_ns.restype = _i
lib.sgemm_selftest_wait_timeout.argtypes = [_ull, _p]
lib.sgemm_selftest_wait_timeout.restype = _i
lib.sgemm_profile_enable.argtypes = [_i]
lib.sgemm_profile_enable.restype = _i
lib.sgemm_profile_collect.argtypes = [ctypes.POINTER(_d), ctypes.POINTER(_ll),
                                      ctypes.POINTER(_d), ctypes.POINTER(_ll)]
lib.sgemm_profile_collect.restype = _i
lib.sgemm_kernel_launch_count.argtypes = []
lib.sgemm_kernel_launch_count.restype = _ll
lib.sgemm_config_string.argtypes = [_i, _i, _i]
lib.sgemm_config_string.restype = ctypes.c_char_p
lib.sgemm_last_kernel.argtypes = []
lib.sgemm_last_kernel.restype = ctypes.c_char_p
lib.sgemm_variant_count.argtypes = []
lib.sgemm_variant_count.restype = _i
lib.sgemm_variant_name.argtypes = [_i]
lib.sgemm_variant_name.restype = ctypes.c_char_p
lib.sgemm_set_variant.argtypes = [_i]
lib.sgemm_set_variant.restype = _i
lib.sgemm_set_3xtf32_kernel.argtypes = [_i]
lib.sgemm_set_3xtf32_kernel.restype = _i
lib.sgemm_debug_drop_release.argtypes = [_i]
lib.sgemm_debug_drop_release.restype = _i
lib.sgemm_debug_bounds_checks.argtypes = []
lib.sgemm_debug_bounds_checks.restype = _i

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = 1
SGEMM_ERR_UNSUPPORTED_DEVICE = 2
SGEMM_ERR_CUDA = 3
SGEMM_ERR_TIMEOUT = 4
SGEMM_ERR_ALLOC = 5
SGEMM_ERR_TOO_LARGE = 6
SGEMM_ERR_BOUNDS = 7


class SgemmError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        msg = lib.sgemm_status_string(status).decode()
        if status in (SGEMM_ERR_CUDA, SGEMM_ERR_ALLOC):
            msg += f" (cuda error {lib.sgemm_last_cuda_error()})"
        super().__init__(msg)


def check(status: int) -> int:
    if status != SGEMM_OK:
        raise SgemmError(status)
    return status


def status_string(status: int) -> str:
    return lib.sgemm_status_string(status).decode()


def version() -> int:
    return lib.sgemm_version()


# ------------------------------------------------------------------ tensors
def _ld(t, width: int) -> int:
    """Row pitch (elements) of a 2-D row-major tensor/array view."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.numel() > 0 and t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    ld = t.stride(0) if (t.size(0) > 1 and t.numel() > 0) else 0
    return max(ld, width, 1)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _shapes(A, B, C):
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A {tuple(A.shape)}, B {tuple(B.shape)}")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    return M, N, K


def _cuda_f32(*named):
    """TypeError unless every (name, tensor) pair holds a CUDA float32 tensor;
    ValueError unless they all sit on one device."""
    import torch
    for name, t in named:
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA float32 tensor")
    if len({t.device for _, t in named}) > 1:
        raise ValueError(", ".join(n for n, _ in named) + " must be on one device")


def sgemm_into(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C <- alpha*A@B + beta*C on CUDA float32 tensors (row-major, any row pitch).
    Asynchronous on `stream` (default: torch's current stream of C's device)."""
    import torch
    _cuda_f32(("A", A), ("B", B), ("C", C))
    M, N, K = _shapes(A, B, C)
    with torch.cuda.device(C.device):
        st = lib.sgemm(M, N, K, float(alpha), A.data_ptr(), _ld(A, K), B.data_ptr(), _ld(B, N),
                       float(beta), C.data_ptr(), _ld(C, N), _stream_handle(stream, C.device))
    check(st)
    return C


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}


def _batched(t, name):
    """(2-D view of batch 0, batch count, batch stride in elements) of a 2-D or
    3-D tensor; a 2-D tensor is one matrix used by every batch (stride 0)."""
    if t.dim() == 2:
        return t, 1, 0
    if t.dim() != 3:
        raise ValueError(f"{name} must be 2-D or 3-D")
    return t[0], t.size(0), (t.stride(0) if t.size(0) > 1 else 0)


def sgemm_ex_into(A, B, C, alpha: float = 1.0, beta: float = 0.0, bias=None, act: str = "none",
                  stream=None):
    """C[b] <- act(alpha*A[b]@B[b] + beta*C[b] + bias[b]) on CUDA float32 tensors.
    C is 3-D (batch, M, N) or 2-D (one batch); A and B are 3-D with the same
    batch or 2-D (shared by all batches); bias is None, a length-N vector
    (shared) or (batch, N).  Asynchronous on `stream`."""
    import torch
    _cuda_f32(("A", A), ("B", B), ("C", C), *((("bias", bias),) if bias is not None else ()))
    if act not in ACTIVATIONS:
        raise ValueError(f"act must be one of {sorted(ACTIVATIONS)}, got {act!r}")
    C0, batch, sc = _batched(C, "C")
    A0, ba, sa = _batched(A, "A")
    B0, bb, sb = _batched(B, "B")
    for name, t, n in (("A", A, ba), ("B", B, bb)):
        if t.dim() == 3 and n != batch:
            raise ValueError(f"{name} has {n} batches, C has {batch}")
    M, N, K = _shapes(A0, B0, C0)
    bias_ptr, sbias = None, 0
    if bias is not None:
        if bias.dim() == 1 and bias.size(0) == N:
            sbias = 0
        elif bias.dim() == 2 and tuple(bias.shape) == (batch, N):
            sbias = bias.stride(0) if batch > 1 else 0
        else:
            raise ValueError(f"bias must be ({N},) or ({batch}, {N})")
        if bias.size(-1) > 1 and bias.stride(-1) != 1:
            raise ValueError("bias rows must be contiguous")
        bias_ptr = bias.data_ptr()
    with torch.cuda.device(C.device):
        st = lib.sgemm_ex(M, N, K, float(alpha), A0.data_ptr(), _ld(A0, K), sa, B0.data_ptr(),
                          _ld(B0, N), sb, float(beta), C0.data_ptr(), _ld(C0, N), sc, batch,
                          bias_ptr, sbias, ACTIVATIONS[act], _stream_handle(stream, C.device))
    check(st)
    return C


def sgemm_3xtf32_into(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """Like sgemm_into(), on the tensor cores by the 3xTF32 split (same FP32
    tolerance, not bitwise equal to sgemm_into)."""
    import torch
    _cuda_f32(("A", A), ("B", B), ("C", C))
    M, N, K = _shapes(A, B, C)
    with torch.cuda.device(C.device):
        st = lib.sgemm_3xtf32(M, N, K, float(alpha), A.data_ptr(), _ld(A, K), B.data_ptr(),
                              _ld(B, N), float(beta), C.data_ptr(), _ld(C, N),
                              _stream_handle(stream, C.device))
    check(st)
    return C


def sgemm_noalloc_into(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """Like sgemm_into(), through the entry point that allocates no device
    memory (its workspace is a fixed array; see include/sgemm.h)."""
    import torch
    _cuda_f32(("A", A), ("B", B), ("C", C))
    M, N, K = _shapes(A, B, C)
    with torch.cuda.device(C.device):
        st = lib.sgemm_noalloc(M, N, K, float(alpha), A.data_ptr(), _ld(A, K), B.data_ptr(),
                               _ld(B, N), float(beta), C.data_ptr(), _ld(C, N),
                               _stream_handle(stream, C.device))
    check(st)
    return C


# floats in the fixed scratch array of sgemm_noalloc (see include/sgemm.h)
NOALLOC_SCRATCH_FLOATS = 8 * 1024 * 1024


def sgemm(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """alpha*A@B + beta*C.  With C=None a new tensor is returned (beta must be 0);
    otherwise C is updated in place and returned."""
    import torch
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty((A.shape[0], B.shape[1]), dtype=torch.float32, device=A.device)
    return sgemm_into(A, B, C, alpha, beta, stream)


def sgemm_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None, device=None,
               tensor_cores: bool = False):
    """The host-buffer entry point: A, B, C are CPU float32 tensors (pinned for
    speed).  C is overwritten with alpha*A@B + beta*C; synchronous.  Copies and
    compute are pipelined over row blocks.  tensor_cores=True uses the 3xTF32
    path (sgemm_host_3xtf32)."""
    import torch
    for name, t in (("A", A), ("B", B), ("C", C)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.is_cuda:
            raise TypeError(f"{name} must be a CPU float32 tensor")
    M, N, K = _shapes(A, B, C)
    device = torch.device(device) if device is not None else \
        torch.device("cuda", torch.cuda.current_device())
    fn = lib.sgemm_host_3xtf32 if tensor_cores else lib.sgemm_host
    with torch.cuda.device(device):
        st = fn(M, N, K, float(alpha), A.data_ptr(), _ld(A, K), B.data_ptr(), _ld(B, N),
                float(beta), C.data_ptr(), _ld(C, N), _stream_handle(stream, device))
    check(st)
    return C


# ------------------------------------------------------------------ control
def device_status(stream=None, device=None) -> int:
    """Synchronise and read/clear the device error word: 0 or SGEMM_ERR_TIMEOUT."""
    import torch
    device = device or torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        return lib.sgemm_device_status(_stream_handle(stream, device))


def set_wait_timeout_ns(ns: int) -> None:
    check(lib.sgemm_set_wait_timeout_ns(int(ns)))


def selftest_wait_timeout(ns: int, stream=None, device=None) -> int:
    import torch
    device = device or torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        return lib.sgemm_selftest_wait_timeout(int(ns), _stream_handle(stream, device))


def profile_enable(on: bool = True) -> None:
    check(lib.sgemm_profile_enable(1 if on else 0))


def profile_collect() -> dict:
    mm, pm = ctypes.c_double(0), ctypes.c_double(0)
    mn, pn = ctypes.c_longlong(0), ctypes.c_longlong(0)
    check(lib.sgemm_profile_collect(ctypes.byref(mm), ctypes.byref(mn), ctypes.byref(pm),
                                    ctypes.byref(pn)))
    return {"main_ms": mm.value, "main_launches": mn.value,
            "pack_ms": pm.value, "pack_launches": pn.value}


def kernel_launch_count() -> int:
    return lib.sgemm_kernel_launch_count()


def config_string(M: int, N: int, K: int) -> str:
    return lib.sgemm_config_string(M, N, K).decode()


def last_kernel() -> str:
    """Configuration of the last main kernel this thread's calls launched."""
    return lib.sgemm_last_kernel().decode()


def variants() -> list:
    """Descriptions of the compiled kernel variants, by index."""
    return [lib.sgemm_variant_name(i).decode() for i in range(lib.sgemm_variant_count())]


def set_variant(variant_id: int) -> None:
    """Force a kernel variant for later calls (-1: automatic choice)."""
    check(lib.sgemm_set_variant(int(variant_id)))


def set_3xtf32_kernel(pair) -> None:
    """3xTF32 main kernel for later calls: the CTA pair (True), the single-CTA
    kernel (False) or the automatic choice per shape (None, the default)."""
    check(lib.sgemm_set_3xtf32_kernel(-1 if pair is None else (1 if pair else 0)))


def debug_drop_release(on: bool) -> None:
    """Failure-detection test switch: while on, plain sgemm() calls run the
    test build of the default kernel in which one release is left out, so a
    bounded wait expires and the kernel's abort path runs (include/sgemm.h)."""
    check(lib.sgemm_debug_drop_release(1 if on else 0))
