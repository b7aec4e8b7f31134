"""The five measured workloads at full size, in the launch configuration the
benchmark times (one sgemm() call through the C ABI), checked against the
oracle on the outputs each workload names (all of them, or seeded rows and
columns), plus the all-ones x all-twos closed form over every full output and
integer-valued inputs checked bit for bit over every full output on both entry
points (the FFMA kernels and the 3xTF32 tensor-core path)."""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import WORKLOADS, sample_indices, workload_inputs
from _helpers import assert_within_bound, to_device

pytestmark = pytest.mark.gpu

# workloads of the plain GEMM entry points (the batched / fused ones go through
# sgemm_ex and are checked in test_sgemm_ex_gpu.py)
PLAIN = [n for n, w in WORKLOADS.items() if not w.extended]


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding  # noqa: F401
    yield


@pytest.mark.parametrize("name", PLAIN)
def test_workload_matches_oracle(name):
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    w = WORKLOADS[name]
    A, B, C = workload_inputs(w)
    dA, dB = to_device(A), to_device(B)
    dC = to_device(C) if C is not None else torch.full((w.M, w.N), float("nan"), device="cuda")
    binding.sgemm_into(dA, dB, dC, w.alpha, w.beta)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    rows, cols = sample_indices(w)
    c_in = C if w.beta != 0 else None
    if rows is None and cols is None:
        ref, bound = oracle.sgemm(A, B, c_in, w.alpha, w.beta)
        got = dC.cpu().numpy()
        assert_within_bound(got, ref, bound, name)
    if rows is not None:
        ref, bound = oracle.sgemm_rows(A, B, c_in, w.alpha, w.beta, rows)
        got = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
        assert_within_bound(got, ref, bound, name + " rows")
    if cols is not None:
        ref, bound = oracle.sgemm_cols(A, B, c_in, w.alpha, w.beta, cols)
        got = dC[:, torch.from_numpy(cols).cuda()].cpu().numpy()
        assert_within_bound(got, ref, bound, name + " cols")
    assert torch.isfinite(dC).all()


@pytest.mark.parametrize("name", PLAIN)
def test_workload_shape_ones_times_twos_exact(name):
    """A = 1, B = 2 at every workload shape (row pitches included): every
    element of C equals 2K exactly (closed form of the tiling exercise page)."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    w = WORKLOADS[name]
    lda, ldb, ldc = w.lds()
    A = torch.ones((w.M, lda), device="cuda")[:, :w.K]
    B = torch.full((w.K, ldb), 2.0, device="cuda")[:, :w.N]
    C = torch.full((w.M, ldc), float("nan"), device="cuda")[:, :w.N]
    binding.sgemm_into(A, B, C, 1.0, 0.0)
    torch.cuda.synchronize()
    assert bool((C == 2.0 * w.K).all())
    del A, B, C
    torch.cuda.empty_cache()


# Integer-valued inputs at every workload shape (row pitches included), on
# both entry points.  Entries of A, B and C_in are integers in [-4, 4], so every
# partial sum of K <= 8192 products is an integer below 2^24 in magnitude and
# exact in fp32 whatever the summation order, and with alpha = 1.5, beta = 0.5
# the result is a multiple of 1/2 below 2^22, exact as well.  The whole C must
# then equal the oracle's bit for bit: the closed form of the exercise page's
# all-ones x all-twos check ("3.3 Shared memory and tiling - exercises",
# skeleton), extended to inputs that tell every row, column and k apart.  On
# the 3xTF32 path an integer splits exactly (hi = x, lo = 0), so it too must
# be bit-exact.
INT_CASES = [(n, path) for n in PLAIN for path in ("ffma", "3xtf32")]
_int_case_cache = {}


def _integer_case(name):
    """(A, B, C_in, oracle C) of the integer-valued inputs at a workload's shape;
    the oracle's whole C is kept for the next test (the other entry point)."""
    if name not in _int_case_cache:
        _int_case_cache.clear()
        from dense_fp32_gemm_02_gb300.workloads import make_inputs
        w = WORKLOADS[name]
        lda, ldb, ldc = w.lds()
        A, B, C = make_inputs(w.M, w.N, w.K, "int4", "int4", "int4", seed=w.seed + 77,
                              lda=lda, ldb=ldb, ldc=ldc)
        ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5, with_bound=False)
        _int_case_cache[name] = (A, B, C, ref)
    return _int_case_cache[name]


@pytest.mark.parametrize("name,path", INT_CASES)
def test_integer_inputs_bit_exact_whole_matrix(name, path):
    """Integer-valued inputs at a workload's full size, alpha=1.5, beta=0.5:
    the whole C is bit-exact against the oracle."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    A, B, C, ref = _integer_case(name)
    dC = to_device(C)
    gemm = binding.sgemm_into if path == "ffma" else binding.sgemm_3xtf32_into
    gemm(to_device(A), to_device(B), dC, 1.5, 0.5)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    got = dC.cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        i, j = bad[0]
        raise AssertionError(f"{name} {path}: {len(bad)} elements differ; first at ({i}, {j}): "
                             f"got {got[i, j]!r}, oracle {ref[i, j]!r}")
    del dC
    torch.cuda.empty_cache()
