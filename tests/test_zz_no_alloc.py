"""The entry point that allocates no device memory (sgemm_noalloc).

Some callers cannot allocate device memory: a host framework that has handed
all of it to its own allocator, or a latency-critical path where an allocation
could synchronise the device or fail.  sgemm_noalloc serves them by keeping its
workspace in a fixed device array.  These tests call it through the C ABI and
compare it with the CPU oracle and with the ordinary sgemm() entry point, on two
calls in a row (the second call finds the first call's data still in the shared
array), and check that a problem too large for the array is refused without any
work.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs
from _helpers import assert_within_bound, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding  # noqa: F401  (fails loudly if not built)
    yield


CASES = [
    # (M, N, K, alpha, beta, seed, B offset in floats: 1 forces the re-pitched copy of B)
    (300, 257, 129, 1.5, 0.5, 1, 0),
    (1030, 700, 515, -1.0, 1.0, 2, 1),
]


def test_no_alloc_matches_sgemm_on_two_calls_in_a_row():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    for (M, N, K, alpha, beta, seed, b_off) in CASES:
        A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=seed)
        dA = to_device(A)
        dB = to_device(B, offset_elems=b_off)
        c_ref = to_device(C)
        c_new = to_device(C)
        binding.sgemm_into(dA, dB, c_ref, alpha, beta)              # existing entry point
        binding.sgemm_noalloc_into(dA, dB, c_new, alpha, beta)      # no-allocation entry point
        torch.cuda.synchronize()
        assert binding.device_status() == binding.SGEMM_OK
        ref, bound = oracle.sgemm(A, B, C, alpha, beta)
        got_ref = c_ref.cpu().numpy()
        got_new = c_new.cpu().numpy()
        assert np.isfinite(got_new).all()
        # against the CPU oracle first, so a fault both entry points share
        # (packing, tensor maps, edge tiles) cannot hide
        assert_within_bound(got_new, ref, bound, f"no-alloc vs oracle {M}x{N}x{K}")
        assert_within_bound(got_new, got_ref, bound, f"no-alloc vs sgemm {M}x{N}x{K}")


def test_no_alloc_refuses_a_problem_larger_than_its_scratch():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    # K * M = 16 Mi floats > 8 Mi floats of scratch.  The buffers are real and
    # full-size, so nothing could be read or written out of bounds regardless.
    M = N = K = 4096
    A = torch.ones((M, K), device="cuda")
    B = torch.ones((K, N), device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    with pytest.raises(binding.SgemmError) as e:
        binding.sgemm_noalloc_into(A, B, C, 1.0, 0.0)
    assert e.value.status == binding.SGEMM_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())          # refused before any work
