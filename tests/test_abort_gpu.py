"""The main kernel's own abort path, made to run without any fault.

A missing barrier arrival shows up only if something checks for it: exercise 5
of "3.3 Shared memory and tiling - exercises" removes a synchronisation and
watches the result go wrong.  Here the library's test switch
(sgemm_debug_drop_release) runs a build of the default persistent kernel in
which consumer warp 0 of CTA 0 leaves out one release of a ring stage.  With a
2 ms wait limit the issuer's bounded wait for that stage expires while no copy
into it is in flight, and the kernel must:
  * report SGEMM_ERR_TIMEOUT through sgemm_device_status;
  * leave the output tile CTA 0 was computing unwritten (NaN sentinel), also
    when that tile is shared with other CTAs through stream-K pieces;
  * write every other tile correctly (checked against the oracle);
  * leave the context usable: the next ordinary call matches the oracle.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs
from _helpers import assert_within_bound, to_device

pytestmark = pytest.mark.gpu

DEFAULT_TIMEOUT_NS = 2_000_000_000

# (M, N, K, what CTA 0 computes) -- the test kernel tiles C in 256 x 128 tiles
# of 64-deep k-slabs over one CTA per SM, whole tiles first, then the leftover
# tiles' slabs spread evenly (stream-K).  In both shapes CTA 0 works on tile 0
# alone (rows 0-255, columns 0-127) and has at least five slabs, so its third
# slab's missing release stops the refill of the fifth.
CASES = [
    (4096, 1280, 512, "a whole tile of 8 slabs (160 tiles: 152 whole, 8 by stream-K)"),
    (1024, 1024, 2048, "a stream-K piece of tile 0 (32 tiles of 32 slabs, all by stream-K)"),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding
    yield
    binding.debug_drop_release(False)
    binding.set_wait_timeout_ns(DEFAULT_TIMEOUT_NS)


@pytest.mark.parametrize("M,N,K,what", CASES)
def test_expired_wait_in_the_main_kernel_aborts_cleanly(M, N, K, what):
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    props = torch.cuda.get_device_properties(0)
    if props.multi_processor_count < 152:
        pytest.skip("the work split of these shapes assumes 152 SMs")
    A, B, _ = make_inputs(M, N, K, "upm1", "upm1", None, seed=M + N + K)
    ref, bound = oracle.sgemm(A, B, None, 1.0, 0.0)
    dA, dB = to_device(A), to_device(B)
    dC = torch.full((M, N), float("nan"), device="cuda")
    assert binding.device_status() == binding.SGEMM_OK
    binding.set_wait_timeout_ns(2_000_000)
    binding.debug_drop_release(True)
    try:
        binding.sgemm_into(dA, dB, dC, 1.0, 0.0)
        status = binding.device_status()
    finally:
        binding.debug_drop_release(False)
        binding.set_wait_timeout_ns(DEFAULT_TIMEOUT_NS)
    assert status == binding.SGEMM_ERR_TIMEOUT, what
    got = dC.cpu().numpy()
    aborted = np.zeros((M, N), dtype=bool)
    aborted[:256, :128] = True
    assert np.isnan(got[aborted]).all(), f"{what}: the aborted tile was written"
    written = np.where(aborted, ref, got)
    assert_within_bound(written, ref, bound, f"{what}: tiles of the other CTAs")
    # the context is usable and the next ordinary call is correct
    dC.fill_(float("nan"))
    binding.sgemm_into(dA, dB, dC, 1.0, 0.0)
    assert binding.device_status() == binding.SGEMM_OK
    assert_within_bound(dC.cpu().numpy(), ref, bound, f"{what}: the next ordinary call")
