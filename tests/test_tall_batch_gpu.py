"""Parity of strided batches that run as one tall GEMM, against the oracle,
through the C ABI (sgemm_ex).

A batch with no bias or activation, one A per batch, M a multiple of 256 up to
4096, K a multiple of 64 and the batches of C one under the other (batch stride
M * ldc) runs through the plain kernel as one (batch*M) x N GEMM whose copies of
B start at the tile's batch: B's batches one under the other, shared, or re-pitched
that way when their rows break the TMA's 16-byte rule.  These tests cover each
of those B layouts, a padded ldc, stream-K tiles that straddle batches, and the
near misses that keep the batched kernel.  Batches of A are laid out with NaN
between them, so a copy from the wrong batch shows up in the result; the
padding columns of C hold a sentinel that must survive.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs
from _helpers import assert_within_bound

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding  # noqa: F401  (fails loudly if not built)
    yield


def _inputs(batch, M, N, K, dist, dist_c, seed):
    As, Bs, Cs = [], [], []
    for b in range(batch):
        A, B, C = make_inputs(M, N, K, dist, dist, dist_c, seed=seed * 1000 + b)
        As.append(A)
        Bs.append(B)
        Cs.append(C)
    return As, Bs, Cs


def _planes(mats, gap, fill=float("nan")):
    """Device tensor (batch, rows, cols) whose batches sit `gap` floats apart
    (batch stride rows*cols + gap), the gaps filled with `fill`."""
    import torch
    batch = len(mats)
    rows, cols = mats[0].shape
    plane = rows * cols + gap
    flat = torch.full((batch * plane + 4,), fill, dtype=torch.float32, device="cuda")
    for b, m in enumerate(mats):
        flat[b * plane:b * plane + rows * cols] = torch.from_numpy(
            np.ascontiguousarray(m).reshape(-1)).cuda()
    return flat.as_strided((batch, rows, cols), (plane, cols, 1))


def _run(As, Bs, Cs, alpha, beta, *, a_gap=4, b_layout="contiguous", ldc_pad=0, c_gap=0):
    """Run sgemm_ex on the batches; returns (C as (batch, M, N), the whole
    padded C buffer as (batch, M, ldc))."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    batch = len(As)
    M, N = As[0].shape[0], Bs[0].shape[1]
    dA = _planes(As, a_gap)
    if b_layout == "shared":
        dB = torch.from_numpy(Bs[0]).cuda()
    elif b_layout == "contiguous":
        dB = _planes(Bs, 0)
    else:                                   # batches of B `b_layout` floats apart
        dB = _planes(Bs, int(b_layout))
    ldc = N + ldc_pad
    plane = M * ldc + c_gap
    flat = torch.full((batch * plane + 4,), SENTINEL, dtype=torch.float32, device="cuda")
    full = flat.as_strided((batch, M, ldc), (plane, ldc, 1))
    for b in range(batch):
        full[b, :, :N] = torch.from_numpy(Cs[b]).cuda()
    dC = full[:, :, :N]
    binding.sgemm_ex_into(dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    return dC.cpu().numpy(), full.cpu().numpy()


def _check(got, full, As, Bs, Cs, alpha, beta, what, exact):
    ref, bound = oracle.sgemm_batched(As, Bs, Cs, alpha, beta, None, "none")
    N = Bs[0].shape[1]
    for b in range(len(As)):
        if exact:
            assert np.array_equal(got[b], ref[b]), f"{what}: batch {b} not bit-exact"
        else:
            assert_within_bound(got[b], ref[b], bound[b], f"{what}: batch {b}")
    assert (full[:, :, N:] == SENTINEL).all(), f"{what}: padding columns of C written"


# (batch, M, N, K, B layout, ldc padding): every case meets the tall-batch
# conditions.  N = 200 keeps B's rows 16-byte aligned (B read in place), N = 203
# does not (B re-pitched, batches one under the other); "3" puts 3 floats
# between B's batches.
TALL_CASES = [
    (3, 512, 200, 128, "contiguous", 0),
    (3, 512, 200, 128, "shared", 0),
    (2, 256, 203, 192, "contiguous", 0),
    (3, 768, 203, 64, "3", 0),
    (2, 512, 136, 256, "contiguous", 5),
    # 48 tiles over 152 SMs: every tile by stream-K, its k range spread over
    # several CTAs
    (3, 512, 1000, 512, "contiguous", 0),
    # 5 x 3 x 8 = 120 tiles of 16 slabs
    (5, 768, 1000, 1024, "contiguous", 3),
    # 2 x 8 x 10 = 160 tiles: one whole wave and 8 tiles by stream-K
    (2, 2048, 1250, 256, "shared", 0),
    # the tallest batch taken: 16 tile rows
    (2, 4096, 136, 64, "contiguous", 0),
]


@pytest.mark.parametrize("case", TALL_CASES, ids=lambda c: "x".join(map(str, c)))
def test_tall_batch_integer_bit_exact(case):
    # integers in [-4, 4] and integer C: every sum is exact, in any order
    batch, M, N, K, b_layout, ldc_pad = case
    As, Bs, Cs = _inputs(batch, M, N, K, "int4", "int4", seed=21 + M + N)
    if b_layout == "shared":
        Bs = [Bs[0]] * batch
    got, full = _run(As, Bs, Cs, 1.5, 0.5, b_layout=b_layout, ldc_pad=ldc_pad)
    _check(got, full, As, Bs, Cs, 1.5, 0.5, f"tall {case}", exact=True)


@pytest.mark.parametrize("b_layout", ["contiguous", "shared"])
def test_tall_batch_random_parity(b_layout):
    batch, M, N, K = 4, 768, 515, 1024
    As, Bs, Cs = _inputs(batch, M, N, K, "upm1", "normal", seed=22)
    if b_layout == "shared":
        Bs = [Bs[0]] * batch
    got, full = _run(As, Bs, Cs, 0.75, -0.5, b_layout=b_layout)
    _check(got, full, As, Bs, Cs, 0.75, -0.5, f"tall random {b_layout}", exact=False)


def test_tall_batch_beta_zero_ignores_nan_c():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    batch, M, N, K = 3, 256, 264, 320
    As, Bs, _ = _inputs(batch, M, N, K, "int4", "int4", seed=23)
    dA = _planes(As, 4)
    dB = _planes(Bs, 0)
    dC = torch.full((batch, M, N), float("nan"), device="cuda")
    binding.sgemm_ex_into(dA, dB, dC, 2.0, 0.0)
    torch.cuda.synchronize()
    ref, _ = oracle.sgemm_batched(As, Bs, None, 2.0, 0.0, None, "none")
    got = dC.cpu().numpy()
    for b in range(batch):
        assert np.array_equal(got[b], ref[b]), f"batch {b} not bit-exact"


# Near misses: each breaks one tall-batch condition and runs the batched
# kernel; the results are the same.
NEAR_MISSES = {
    "c_gap": dict(M=512, K=128, c_gap=4),           # C batches not one under the other
    "m_ragged": dict(M=300, K=128),                  # M not whole tiles
    "m_over_16_tiles": dict(M=4352, K=64),           # 17 tile rows per batch
    "k_ragged": dict(M=512, K=100),                  # K not whole slabs
    "b_gap_aligned": dict(M=512, K=128, b_layout="4"),   # B read in place at its own stride
}


@pytest.mark.parametrize("name", sorted(NEAR_MISSES))
def test_near_misses_keep_batched_kernel_results(name):
    kw = dict(NEAR_MISSES[name])
    M, K = kw.pop("M"), kw.pop("K")
    batch, N = 3, 200
    As, Bs, Cs = _inputs(batch, M, N, K, "int4", "int4", seed=24)
    got, full = _run(As, Bs, Cs, 1.5, 0.5, **kw)
    _check(got, full, As, Bs, Cs, 1.5, 0.5, name, exact=True)


def test_tall_batch_reproducible():
    batch, M, N, K = 3, 512, 1000, 512      # every tile by stream-K
    As, Bs, Cs = _inputs(batch, M, N, K, "upm1", "normal", seed=25)
    g1, _ = _run(As, Bs, Cs, 1.0, 0.25)
    g2, _ = _run(As, Bs, Cs, 1.0, 0.25)
    assert np.array_equal(g1, g2)
