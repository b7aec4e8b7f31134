"""Host-side checks of the C ABI that need no GPU.

The library must load on a machine without a GPU, export every function that
include/sgemm.h declares, and reject invalid arguments before touching CUDA.
"""
import ctypes
import os
import re

import pytest

from dense_fp32_gemm_02_gb300 import build as sgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    path = sgbuild.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(sgemm\w*)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("sgemm", "sgemm_host", "sgemm_status_string", "sgemm_version"):
        assert required in names, names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in include/*.h but not exported: {missing}"


def test_library_exports_nothing_undeclared():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", sgbuild.LIB_PATH], capture_output=True,
                         text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = {l.split()[-1] for l in out.stdout.splitlines() if " T " in l}
    assert exported <= set(declared_functions()), exported - set(declared_functions())


def test_status_strings_and_version(lib):
    lib.sgemm_status_string.restype = ctypes.c_char_p
    for st in range(7):
        s = lib.sgemm_status_string(st).decode()
        assert s.startswith("SGEMM_")
    assert b"unknown" in lib.sgemm_status_string(99)
    assert lib.sgemm_version() >= 10000


def _call(lib, M, N, K, A=1, lda=None, B=1, ldb=None, C=1, ldc=None, alpha=1.0, beta=0.0,
          entry="sgemm"):
    f = getattr(lib, entry)
    f.argtypes = [ctypes.c_int] * 3 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    lda = max(1, K) if lda is None else lda
    ldb = max(1, N) if ldb is None else ldb
    ldc = max(1, N) if ldc is None else ldc
    # fake, never-dereferenced but 16-byte aligned addresses (validation happens first)
    ptr = lambda v: None if v is None else 0x100000 * v
    return f(M, N, K, alpha, ptr(A), lda, ptr(B), ldb, beta, ptr(C), ldc, None)


INVALID = [
    dict(M=-1, N=4, K=4),
    dict(M=4, N=-1, K=4),
    dict(M=4, N=4, K=-1),
    dict(M=4, N=4, K=8, lda=7),
    dict(M=4, N=8, K=4, ldb=7),
    dict(M=4, N=8, K=4, ldc=7),
    dict(M=4, N=4, K=4, A=None),
    dict(M=4, N=4, K=4, B=None),
    dict(M=4, N=4, K=4, C=None),
    dict(M=4, N=4, K=0, lda=0),
]


# every entry point with the sgemm() argument list
ENTRIES = ["sgemm", "sgemm_host", "sgemm_3xtf32", "sgemm_host_3xtf32", "sgemm_noalloc"]


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("kw", INVALID)
def test_invalid_arguments_rejected_without_gpu(lib, kw, entry):
    assert _call(lib, entry=entry, **kw) == 1  # SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("entry", ["sgemm", "sgemm_3xtf32", "sgemm_noalloc"])
@pytest.mark.parametrize("M,N,K", [(2 ** 31 - 1, 1, 1), (1, 2 ** 31 - 65535, 1), (1, 1, 2 ** 31 - 1000)])
def test_sizes_past_the_limit_rejected_without_gpu(lib, M, N, K, entry):
    """Sizes within 2^16 of 2^31 would overflow the kernels' 32-bit rounding
    up to whole tiles: SGEMM_ERR_TOO_LARGE before any CUDA call."""
    assert _call(lib, M, N, K, A=16, B=16, C=16, entry=entry) == 6


def test_misaligned_pointer_rejected(lib):
    f = lib.sgemm
    f.argtypes = [ctypes.c_int] * 3 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert f(4, 4, 4, 1.0, 0x100001, 4, 0x200000, 4, 0.0, 0x300000, 4, None) == 1
    assert f(4, 4, 4, 1.0, 0x100000, 4, 0x200000, 4, 0.0, 0x300002, 4, None) == 1


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("kw", [dict(M=0, N=4, K=4), dict(M=4, N=0, K=4),
                                dict(M=0, N=0, K=0, A=None, B=None, C=None)])
def test_empty_output_is_a_no_op_without_gpu(lib, kw, entry):
    # nothing to compute: success without any CUDA call, pointers not read
    assert _call(lib, entry=entry, **kw) == 0


def test_variant_selection_validates(lib):
    lib.sgemm_variant_name.restype = ctypes.c_char_p
    n = lib.sgemm_variant_count()
    assert n >= 1
    assert lib.sgemm_variant_name(n) == b"" and lib.sgemm_variant_name(-1) == b""
    assert lib.sgemm_set_variant(n) == 1 and lib.sgemm_set_variant(-2) == 1
    assert lib.sgemm_set_variant(n - 1) == 0 and lib.sgemm_set_variant(-1) == 0


def test_default_library_is_not_the_range_checked_build(lib):
    assert lib.sgemm_debug_bounds_checks() == 0
    lib.sgemm_status_string.restype = ctypes.c_char_p
    assert b"SGEMM_ERR_BOUNDS" in lib.sgemm_status_string(7)


def test_drop_release_switch_validates(lib):
    assert lib.sgemm_debug_drop_release(2) == 1 and lib.sgemm_debug_drop_release(-1) == 1
    assert lib.sgemm_debug_drop_release(1) == 0 and lib.sgemm_debug_drop_release(0) == 0


def test_timeout_setter_validates(lib):
    lib.sgemm_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
    assert lib.sgemm_set_wait_timeout_ns(10) == 1
    assert lib.sgemm_set_wait_timeout_ns(2_000_000_000) == 0


def test_binding_loads_and_reports_config():
    from dense_fp32_gemm_02_gb300 import binding
    assert binding.version() == ctypes.CDLL(sgbuild.LIB_PATH).sgemm_version()
    assert "tile=" in binding.config_string(8192, 8192, 8192)
    names = binding.variants()
    assert len(names) >= 1 and all("tile=" in n for n in names)
    assert binding.config_string(8192, 8192, 8192) in names
    with pytest.raises(binding.SgemmError) as e:
        binding.check(1)
    assert "INVALID_ARG" in str(e.value)


def _call_ex(lib, M=4, N=4, K=4, batch=2, stride_a=16, stride_b=16, stride_c=16, bias=None,
             stride_bias=0, act=0, C=3):
    f = lib.sgemm_ex
    ll = ctypes.c_longlong
    f.argtypes = [ctypes.c_int] * 3 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ll,
                                       ctypes.c_void_p, ctypes.c_int, ll, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_int, ll, ctypes.c_int,
                                       ctypes.c_void_p, ll, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    # fake, never-dereferenced, 16-byte aligned addresses (validation comes first)
    ptr = lambda v: None if v is None else 0x100000 * v
    return f(M, N, K, 1.0, ptr(1), max(1, K), stride_a, ptr(2), max(1, N), stride_b, 0.0,
             ptr(C), max(1, N), stride_c, batch, bias, stride_bias, act, None)


@pytest.mark.parametrize("kw", [
    dict(batch=-1), dict(stride_a=-1), dict(stride_b=-4), dict(stride_c=-16),
    dict(stride_bias=-1, bias=0x400000), dict(act=3), dict(act=-1),
    dict(bias=0x400001),                       # bias not 4-byte aligned
    dict(stride_c=15),                         # batches of C overlap: (M-1)*ldc + N = 16
    dict(M=-1), dict(C=None),
])
def test_ex_invalid_arguments_rejected_without_gpu(lib, kw):
    assert _call_ex(lib, **kw) == 1  # SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(batch=0), dict(M=0), dict(N=0, stride_c=0),
                                dict(batch=0, C=None, stride_c=0)])
def test_ex_empty_is_a_no_op_without_gpu(lib, kw):
    assert _call_ex(lib, **kw) == 0


def test_ex_single_batch_needs_no_c_stride(lib):
    # batch 1: stride_c is irrelevant, so 0 is accepted (rejected only if it were
    # needed); validation happens before any CUDA call, so on a machine without a
    # GPU the call gets as far as the device check
    st = _call_ex(lib, batch=1, stride_c=0, stride_a=0, stride_b=0)
    assert st != 1


@pytest.mark.parametrize("M,N,K,tile", [
    (8192, 8192, 8192, "256x128"),     # no padding either way: the default
    (4096, 4096, 4096, "256x128"),
    (16384, 16384, 512, "256x128"),
    (4097, 3001, 1023, "128x256"),     # 17 x 256 rows pad more than 33 x 128
    (300, 8192, 512, "128x256"),       # 512 rows against 384
    (4096, 300, 64, "256x128"),        # 300 columns: 384 against 512
])
def test_shape_heuristic_takes_the_tile_orientation_that_pads_less(M, N, K, tile):
    """Between the 256x128 tile and the same tile turned (128x256) the one that
    pads C less is chosen, the 256x128 one on a tie."""
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    name = binding.config_string(M, N, K)
    assert f"tile={tile}x64" in name and name in binding.variants()[:2]


def test_3xtf32_kernel_choice_validates(lib):
    lib.sgemm_set_3xtf32_kernel.argtypes = [ctypes.c_int]
    for v in (-1, 0, 1, -1):
        assert lib.sgemm_set_3xtf32_kernel(v) == 0
    assert lib.sgemm_set_3xtf32_kernel(2) == 1 and lib.sgemm_set_3xtf32_kernel(-2) == 1


def test_every_declared_function_is_documented_in_the_header():
    """Each declaration sits directly under a comment, or directly under
    another declaration of the same documented group (e.g. the variant
    functions), and the header names the page that defines the operation."""
    for h in HEADERS:
        text = open(h).read()
        comments = [(m.start(), m.end()) for m in re.finditer(r"/\*.*?\*/", text, flags=re.S)]

        def outside_comments(pos):
            return all(not (a <= pos < b) for a, b in comments)

        documented = {}
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(sgemm\w*)\s*\(", text, flags=re.M):
            if not outside_comments(m.start()):
                continue
            start = m.start()
            last_comment_end = max((b for a, b in comments if b <= start), default=-1)
            semis = [i for i in range(start) if text[i] == ";" and outside_comments(i)]
            last_semi = semis[-1] if semis else -1
            if last_comment_end > last_semi and not text[last_comment_end:start].strip():
                documented[m.group(1)] = True
            elif (last_semi > last_comment_end and not text[last_semi + 1:start].strip()
                  and text[last_semi + 1:start].count("\n") <= 1):   # the next line: same group
                documented[m.group(1)] = documented.get(prev, False)
            else:
                documented[m.group(1)] = False
            prev = m.group(1)
        missing = sorted(n for n, ok in documented.items() if not ok)
        assert not missing, f"{os.path.basename(h)}: no comment above {missing}"
    header = open(os.path.join(ROOT, "include", "sgemm.h")).read()
    flat = re.sub(r"\s*\n\s*\*?\s*", " ", header)     # comment lines joined
    assert "How to implement matrix multiplication efficiently" in flat
    assert "Naive GEMM and prerequisites" in flat
