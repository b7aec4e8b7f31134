"""The five measured workloads at full size, in the launch configuration the
benchmark times (one sgemm() call through the C ABI), checked against the
oracle on the outputs each workload names (all of them, or seeded rows and
columns), plus the all-ones x all-twos closed form over every full output."""
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


def test_integer_inputs_bit_exact_at_ragged_full_size():
    """Integer inputs at the ragged workload's full size, alpha=1.5, beta=0.5:
    whole-matrix bit-exact against the oracle."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    from dense_fp32_gemm_02_gb300.workloads import make_inputs
    w = WORKLOADS["sgemm_ragged_4097x3001x1023"]
    lda, ldb, ldc = w.lds()
    A, B, C = make_inputs(w.M, w.N, w.K, "int4", "int4", "int4", seed=77, lda=lda, ldb=ldb,
                          ldc=ldc)
    dC = to_device(C)
    binding.sgemm_into(to_device(A), to_device(B), dC, 1.5, 0.5)
    torch.cuda.synchronize()
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5, with_bound=False)
    assert np.array_equal(dC.cpu().numpy(), ref)
