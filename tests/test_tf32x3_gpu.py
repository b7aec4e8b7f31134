"""Parity of the 3xTF32 tensor-core entry point (sgemm_3xtf32) against the CPU
oracle, with the same FP32 tolerance as the FFMA path.  Integer-valued inputs
split exactly (lo part zero) and every partial sum is an exact integer, so
those cases must match bit for bit."""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import WORKLOADS, make_inputs, sample_indices, workload_inputs
from _helpers import assert_within_bound, to_device

pytestmark = pytest.mark.gpu

# workloads of the plain GEMM entry points (the batched / fused ones go through
# sgemm_ex and are checked in test_sgemm_ex_gpu.py)
PLAIN = [n for n, w in WORKLOADS.items() if not w.extended]


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding  # noqa: F401
    yield


def run3(A, B, C, alpha, beta, offsets=(0, 0, 0)):
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N = A.shape[0], B.shape[1]
    dA = to_device(A, offset_elems=offsets[0])
    dB = to_device(B, offset_elems=offsets[1])
    dC = to_device(C if C is not None else np.full((M, N), np.nan, np.float32),
                   offset_elems=offsets[2])
    binding.sgemm_3xtf32_into(dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    return dC


def test_single_tile_integer_exact():
    A, B, C = make_inputs(128, 256, 32, "int4", "int4", "int4", seed=1)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    got = run3(A, B, C, 1.5, 0.5).cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 300, 5), (129, 257, 33), (300, 513, 100),
                                   (256, 512, 1024), (1000, 77, 129)])
def test_integer_inputs_bit_exact(M, N, K):
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=M + N + K)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    got = run3(A, B, C, 1.5, 0.5).cpu().numpy()
    assert np.array_equal(got, ref), (M, N, K)


@pytest.mark.parametrize("M,N,K", [(300, 200, 100), (129, 257, 513), (640, 640, 640),
                                   (5, 1100, 260), (1031, 777, 1500)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, 0.5), (-0.75, 1.0)])
def test_random_parity_within_bound(M, N, K, alpha, beta):
    A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=M * 7 + K)
    c_in = C if beta != 0 else None
    ref, bound = oracle.sgemm(A, B, c_in, alpha, beta)
    got = run3(A, B, c_in, alpha, beta).cpu().numpy()
    assert_within_bound(got, ref, bound, f"3xtf32 {M}x{N}x{K}")


def test_leading_dimensions_misalignment_and_padding():
    M, N, K = 203, 157, 141
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=7, lda=K + 3, ldb=N + 5,
                          ldc=N + 2)
    ref, bound = oracle.sgemm(A, B, C, 1.0, 1.0)
    dC = run3(A, B, C, 1.0, 1.0, offsets=(1, 3, 1))
    got = dC.cpu().numpy()
    assert np.isfinite(got).all()
    assert_within_bound(got, ref, bound, "3xtf32 ld/offsets")
    full = dC.as_strided((M, N + 2), (N + 2, 1)).cpu().numpy()
    assert np.isnan(full[:, N:]).all()


def test_bitwise_deterministic():
    import torch
    A, B, C = make_inputs(700, 900, 800, "normal", "normal", "normal", seed=3)
    g1 = run3(A, B, C, 1.0, 1.0).cpu()
    g2 = run3(A, B, C, 1.0, 1.0).cpu()
    assert torch.equal(g1, g2)


@pytest.mark.parametrize("name", PLAIN)
def test_workloads_match_oracle(name):
    import torch
    w = WORKLOADS[name]
    A, B, C = workload_inputs(w)
    dC = run3(A, B, C, w.alpha, w.beta)
    rows, cols = sample_indices(w)
    c_in = C if w.beta != 0 else None
    if rows is None and cols is None:
        ref, bound = oracle.sgemm(A, B, c_in, w.alpha, w.beta)
        assert_within_bound(dC.cpu().numpy(), ref, bound, name)
    if rows is not None:
        ref, bound = oracle.sgemm_rows(A, B, c_in, w.alpha, w.beta, rows)
        assert_within_bound(dC[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, bound, name)
    if cols is not None:
        ref, bound = oracle.sgemm_cols(A, B, c_in, w.alpha, w.beta, cols)
        assert_within_bound(dC[:, torch.from_numpy(cols).cuda()].cpu().numpy(), ref, bound, name)


@pytest.mark.parametrize("M,N,K", [(300, 513, 100), (1031, 777, 1500), (4100, 3001, 515),
                                   (2048, 2048, 64), (4096, 4096, 64)])
def test_cta_pair_kernel_matches_oracle(M, N, K):
    """The CTA-pair main kernel (sgemm_set_3xtf32_kernel(1)): integer inputs bit-exact
    and random inputs within the bound, on ragged pair tiles, fewer tiles than pairs
    (2048^2: 64), several waves (4100 x 3001: 204 pair tiles over 76 pairs) and a
    half-width last wave (4096^2: 256 tiles, the last 28 cut in halves)."""
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_3xtf32_kernel(True)
    try:
        A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=M + 3 * N)
        ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
        got = run3(A, B, C, 1.5, 0.5).cpu().numpy()
        assert np.array_equal(got, ref), (M, N, K)
        A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=M + 5 * N)
        ref, bound = oracle.sgemm(A, B, C, -0.75, 1.0)
        got = run3(A, B, C, -0.75, 1.0).cpu().numpy()
        assert_within_bound(got, ref, bound, f"pair {M}x{N}x{K}")
    finally:
        binding.set_3xtf32_kernel(None)
