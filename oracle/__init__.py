"""CPU oracle for the row-major FP32 GEMM  C = alpha*A*B + beta*C.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg import this package; the product path never does, and it
shares no code with the CUDA library.

The arithmetic lives in ``oracle_sgemm.c`` (plain C, double accumulation, one
final rounding to float; see that file's header for the definition it follows
and the readings taken where the pages are silent).  This module only compiles
it with the host C compiler, loads it with ctypes and splits rows over threads
(ctypes releases the GIL during the call, so the threads run in parallel).

Public functions take numpy float32 2-D arrays whose rows are contiguous; a
leading dimension larger than the logical width is expressed by passing a
column slice of a wider array (``storage[:, :K]``).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_sgemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"liboracle_sgemm_{platform.machine()}.so")
_ABI_VERSION = 2

# -ffp-contract=off: no fused multiply-add contraction; no -ffast-math; no -march:
# the same source gives the same bits on x86-64 and aarch64.
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (idempotent). Returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CC", "gcc"), *CFLAGS, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load_library(path: str):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    if lib.oracle_abi_version() != _ABI_VERSION:
        raise RuntimeError(f"stale oracle build at {path}; rebuild it")
    ll, f32 = ctypes.c_longlong, ctypes.c_float
    p = ctypes.c_void_p
    lib.oracle_sgemm_rows.argtypes = [ll, ll, ll, f32, p, ll, p, ll, f32, p, ll,
                                      p, ll, p, p]
    lib.oracle_sgemm_rows.restype = ctypes.c_int
    lib.oracle_sgemm_cols.argtypes = [ll, ll, ll, f32, p, ll, p, ll, f32, p, ll,
                                      p, ll, ll, ll, p, p]
    lib.oracle_sgemm_cols.restype = ctypes.c_int
    lib.oracle_sgemm_ex_rows.argtypes = [ll, ll, ll, f32, p, ll, p, ll, f32, p, ll,
                                         p, ctypes.c_int, p, ll, p, p]
    lib.oracle_sgemm_ex_rows.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _check_matrix(x, name):
    if x is None:
        return None, 0
    if not isinstance(x, np.ndarray) or x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D numpy float32 array")
    if x.size > 0 and x.shape[1] > 1 and x.strides[1] != 4:
        raise ValueError(f"{name} rows must be contiguous")
    ld = x.strides[0] // 4 if (x.shape[0] > 1 and x.size > 0) else 0
    return x, max(ld, x.shape[1], 1)


def _ptr(x):
    return None if x is None else x.ctypes.data


def _threads(threads):
    if threads is None:
        threads = os.cpu_count() or 1
    return max(1, int(threads))


def _dims(A, B, C_in, beta):
    A, lda = _check_matrix(A, "A")
    B, ldb = _check_matrix(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    if beta != 0.0:
        C_in, ldc = _check_matrix(C_in, "C_in")
        if C_in.shape != (M, N):
            raise ValueError(f"C_in must be {(M, N)}, got {C_in.shape}")
    else:
        C_in, ldc = None, max(1, N)
    return A, lda, B, ldb, C_in, ldc, M, N, K


def sgemm_rows(A, B, C_in, alpha, beta, rows, threads=None, with_bound=True, lib=None):
    """Rows ``rows`` of alpha*A@B + beta*C_in.  Returns (out, bound):
    out is float32 [len(rows), N]; bound is float64 of the same shape (or None)."""
    A, lda, B, ldb, C_in, ldc, M, N, K = _dims(A, B, C_in, beta)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    nrows = rows.shape[0]
    out = np.empty((nrows, N), dtype=np.float32)
    bound = np.empty((nrows, N), dtype=np.float64) if with_bound else None
    lib = lib or _load()
    nt = min(_threads(threads), max(1, nrows))
    chunks = np.array_split(np.arange(nrows), nt)

    def run(idx):
        if idx.size == 0:
            return 0
        r0, r1 = int(idx[0]), int(idx[-1]) + 1
        sub_rows = rows[r0:r1]
        o = out[r0:r1]
        b = bound[r0:r1] if bound is not None else None
        return lib.oracle_sgemm_rows(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                                     float(beta), _ptr(C_in), ldc,
                                     sub_rows.ctypes.data, r1 - r0, _ptr(o), _ptr(b))

    with ThreadPoolExecutor(max_workers=nt) as ex:
        codes = list(ex.map(run, chunks))
    if any(codes):
        raise RuntimeError(f"oracle_sgemm_rows failed with codes {set(codes)}")
    return out, bound


def sgemm_cols(A, B, C_in, alpha, beta, cols, threads=None, with_bound=True, lib=None):
    """Columns ``cols`` of alpha*A@B + beta*C_in over all M rows.  Returns (out, bound)
    with out float32 [M, len(cols)] and bound float64 of the same shape (or None)."""
    A, lda, B, ldb, C_in, ldc, M, N, K = _dims(A, B, C_in, beta)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    ncols = cols.shape[0]
    out = np.empty((M, ncols), dtype=np.float32)
    bound = np.empty((M, ncols), dtype=np.float64) if with_bound else None
    lib = lib or _load()
    nt = min(_threads(threads), max(1, M))
    chunks = np.array_split(np.arange(M), nt)

    def run(idx):
        if idx.size == 0:
            return 0
        r0, r1 = int(idx[0]), int(idx[-1]) + 1
        o = out[r0:r1]
        b = bound[r0:r1] if bound is not None else None
        return lib.oracle_sgemm_cols(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                                     float(beta), _ptr(C_in), ldc,
                                     cols.ctypes.data, ncols, r0, r1, _ptr(o), _ptr(b))

    with ThreadPoolExecutor(max_workers=nt) as ex:
        codes = list(ex.map(run, chunks))
    if any(codes):
        raise RuntimeError(f"oracle_sgemm_cols failed with codes {set(codes)}")
    return out, bound


def sgemm(A, B, C_in, alpha, beta, threads=None, with_bound=True, lib=None):
    """Whole alpha*A@B + beta*C_in.  Returns (out float32 [M,N], bound float64 [M,N])."""
    M = A.shape[0]
    return sgemm_rows(A, B, C_in, alpha, beta, np.arange(M, dtype=np.int64),
                      threads=threads, with_bound=with_bound, lib=lib)


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}


def sgemm_ex_rows(A, B, C_in, alpha, beta, bias=None, act="none", rows=None, threads=None,
                  with_bound=True, lib=None):
    """Rows ``rows`` (all when None) of act(alpha*A@B + beta*C_in + bias) for one
    batch; ``bias`` is a float32 vector of length N or None.  Returns (out, bound)."""
    A, lda, B, ldb, C_in, ldc, M, N, K = _dims(A, B, C_in, beta)
    if bias is not None:
        if not isinstance(bias, np.ndarray) or bias.dtype != np.float32 or bias.shape != (N,):
            raise TypeError(f"bias must be a float32 vector of length {N}")
        bias = np.ascontiguousarray(bias)
    code = ACTIVATIONS[act]
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    nrows = rows.shape[0]
    out = np.empty((nrows, N), dtype=np.float32)
    bound = np.empty((nrows, N), dtype=np.float64) if with_bound else None
    lib = lib or _load()
    nt = min(_threads(threads), max(1, nrows))
    chunks = np.array_split(np.arange(nrows), nt)

    def run(idx):
        if idx.size == 0:
            return 0
        r0, r1 = int(idx[0]), int(idx[-1]) + 1
        o = out[r0:r1]
        b = bound[r0:r1] if bound is not None else None
        return lib.oracle_sgemm_ex_rows(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                                        float(beta), _ptr(C_in), ldc, _ptr(bias), code,
                                        rows[r0:r1].ctypes.data, r1 - r0, _ptr(o), _ptr(b))

    with ThreadPoolExecutor(max_workers=nt) as ex:
        codes = list(ex.map(run, chunks))
    if any(codes):
        raise RuntimeError(f"oracle_sgemm_ex_rows failed with codes {set(codes)}")
    return out, bound


def sgemm_batched(As, Bs, Cs, alpha, beta, biases=None, act="none", rows=None, threads=None,
                  with_bound=True, lib=None):
    """One fused GEMM per batch: As, Bs, Cs are sequences of 2-D float32 arrays (Cs
    entries may be None when beta == 0), biases a sequence of vectors or None.
    Returns (out [batch, len(rows), N], bound of the same shape)."""
    batch = len(As)
    if len(Bs) != batch or (Cs is not None and len(Cs) != batch):
        raise ValueError("As, Bs and Cs must have one entry per batch")
    outs, bounds = [], []
    for b in range(batch):
        o, bd = sgemm_ex_rows(As[b], Bs[b], None if Cs is None else Cs[b], alpha, beta,
                              None if biases is None else biases[b], act, rows, threads,
                              with_bound, lib)
        outs.append(o)
        bounds.append(bd)
    return np.stack(outs), (np.stack(bounds) if with_bound else None)
