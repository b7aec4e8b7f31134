"""Parity of sgemm_ex (strided batched GEMM with a fused bias and activation)
against the oracle, through the C ABI.

Every batch is checked element by element against the oracle's fused GEMM
(act(alpha*A@B + beta*C + bias) in double, one rounding) within the oracle's
bound; integer-valued inputs, where every intermediate is exact, must match bit
for bit.  Batches are laid out with NaN between them, so a read of the wrong
batch or past a batch shows up in the result.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import (WORKLOADS, make_inputs, sample_indices,
                                                workload_bias, workload_inputs)
from _helpers import assert_within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding  # noqa: F401  (fails loudly if not built)
    yield


def _stack(mats, gap, device="cuda"):
    """Device tensor (batch, rows, cols) whose batches sit `gap` NaN floats
    apart (batch stride rows*cols + gap)."""
    import torch
    batch = len(mats)
    rows, cols = mats[0].shape
    plane = rows * cols + gap
    flat = torch.full((batch * plane + 4,), float("nan"), dtype=torch.float32, device=device)
    for b, m in enumerate(mats):
        flat[b * plane:b * plane + rows * cols] = torch.from_numpy(
            np.ascontiguousarray(m).reshape(-1)).to(device)
    return flat.as_strided((batch, rows, cols), (plane, cols, 1))


def _inputs(batch, M, N, K, dist="upm1", dist_c="normal", seed=0):
    As, Bs, Cs = [], [], []
    for b in range(batch):
        A, B, C = make_inputs(M, N, K, dist, dist, dist_c, seed=seed * 1000 + b)
        As.append(A)
        Bs.append(B)
        Cs.append(C)
    return As, Bs, Cs


def _run(As, Bs, Cs, alpha, beta, biases, act, share_a=False, share_b=False, gap=4,
         bias_shared=False):
    # the same gap after every batch of A, B and C: with gap 4 a batch stride is
    # 16-byte aligned exactly when the matrix size is a multiple of 4 floats, so
    # the shapes below cover both the direct and the re-pitched B and both
    # epilogue paths
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    dA = torch.from_numpy(As[0]).cuda() if share_a else _stack(As, gap)
    dB = torch.from_numpy(Bs[0]).cuda() if share_b else _stack(Bs, gap)
    Cin = Cs if Cs[0] is not None else [np.full((As[0].shape[0], Bs[0].shape[1]), np.nan,
                                                np.float32)] * len(As)
    dC = _stack(Cin, gap)
    dbias = None
    if biases is not None:
        dbias = (torch.from_numpy(biases[0]).cuda() if bias_shared
                 else torch.from_numpy(np.stack(biases)).cuda())
    binding.sgemm_ex_into(dA, dB, dC, alpha, beta, bias=dbias, act=act)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    return dC.cpu().numpy()


def _check(got, As, Bs, Cs, alpha, beta, biases, act, what, exact=False):
    ref, bound = oracle.sgemm_batched(As, Bs, Cs if Cs[0] is not None else None, alpha, beta,
                                      biases, act)
    for b in range(len(As)):
        if exact:
            assert np.array_equal(got[b], ref[b]), f"{what}: batch {b} not bit-exact"
        else:
            assert_within_bound(got[b], ref[b], bound[b], f"{what}: batch {b}")


@pytest.mark.parametrize("act", ["none", "relu"])
@pytest.mark.parametrize("batch", [1, 3])
def test_integer_grid_bit_exact(act, batch):
    # integers in [-4, 4] and integer bias/C: exact in any summation order;
    # batch 1 runs the unbatched fused-epilogue kernel, 3 the batched one
    M, N, K = 300, 257, 129
    As, Bs, Cs = _inputs(batch, M, N, K, "int4", "int4", seed=1)
    rng = np.random.default_rng(2)
    biases = [rng.integers(-50, 51, N).astype(np.float32) for _ in range(batch)]
    got = _run(As, Bs, Cs, 1.5, 0.5, biases, act)
    _check(got, As, Bs, Cs, 1.5, 0.5, biases, act, f"integer {act}", exact=True)


@pytest.mark.parametrize("shape", [(2, 513, 385, 200), (3, 300, 257, 129), (5, 64, 72, 1023),
                                   (1, 1030, 700, 515), (1, 2048, 1100, 1056)])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_random_parity(shape, act):
    batch, M, N, K = shape
    As, Bs, Cs = _inputs(batch, M, N, K, seed=3 + M)
    rng = np.random.default_rng(4 + N)
    biases = [rng.standard_normal(N).astype(np.float32) for _ in range(batch)]
    got = _run(As, Bs, Cs, 0.75, -0.5, biases, act)
    _check(got, As, Bs, Cs, 0.75, -0.5, biases, act, f"{shape} {act}")


def test_no_bias_beta_zero_ignores_nan_c():
    batch, M, N, K = 4, 200, 136, 96
    As, Bs, _ = _inputs(batch, M, N, K, seed=5)
    got = _run(As, Bs, [None] * batch, 1.0, 0.0, None, "gelu")
    assert np.isfinite(got).all()
    _check(got, As, Bs, [None] * batch, 1.0, 0.0, None, "gelu", "beta 0, NaN C")


@pytest.mark.parametrize("share", ["a", "b"])
def test_shared_operand_across_batches(share):
    batch, M, N, K = 3, 260, 190, 150
    As, Bs, Cs = _inputs(batch, M, N, K, seed=6)
    if share == "a":
        As = [As[0]] * batch
    else:
        Bs = [Bs[0]] * batch
    rng = np.random.default_rng(7)
    bias = rng.standard_normal(N).astype(np.float32)
    got = _run(As, Bs, Cs, 1.0, 1.0, [bias] * batch, "relu", share_a=share == "a",
               share_b=share == "b", bias_shared=True)
    _check(got, As, Bs, Cs, 1.0, 1.0, [bias] * batch, "relu", f"shared {share}")


def test_unaligned_batch_strides_and_pitches():
    # gaps of an odd number of floats: B planes are not 16-byte aligned, so B
    # goes through the re-pitching copy; C batches are not either, so the
    # epilogue takes its scalar path
    batch, M, N, K = 3, 131, 97, 77
    As, Bs, Cs = _inputs(batch, M, N, K, seed=8)
    rng = np.random.default_rng(9)
    biases = [rng.standard_normal(N).astype(np.float32) for _ in range(batch)]
    got = _run(As, Bs, Cs, 1.25, 0.5, biases, "gelu", gap=3)
    _check(got, As, Bs, Cs, 1.25, 0.5, biases, "gelu", "odd strides")


def test_many_small_batches():
    batch, M, N, K = 257, 64, 64, 64
    As, Bs, Cs = _inputs(batch, M, N, K, "int4", "int4", seed=10)
    got = _run(As, Bs, Cs, 1.0, -1.0, None, "relu")
    _check(got, As, Bs, Cs, 1.0, -1.0, None, "relu", "257 batches", exact=True)


@pytest.mark.parametrize("case", ["k0", "alpha0"])
def test_quick_returns_apply_bias_and_activation(case):
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    batch, M, N = 2, 70, 33
    K = 0 if case == "k0" else 16
    As, Bs, Cs = _inputs(batch, M, N, max(K, 1), seed=11)
    As = [a[:, :K] for a in As]
    Bs = [b[:K] for b in Bs]
    rng = np.random.default_rng(12)
    biases = [rng.standard_normal(N).astype(np.float32) for _ in range(batch)]
    alpha = 0.0 if case == "alpha0" else 1.0
    dA = torch.zeros((batch, M, max(K, 1)), device="cuda")[:, :, :K]
    dB = torch.zeros((batch, max(K, 1), N), device="cuda")[:, :K]
    dC = torch.from_numpy(np.stack(Cs)).cuda()
    binding.sgemm_ex_into(dA, dB, dC, alpha, 0.5, bias=torch.from_numpy(np.stack(biases)).cuda(),
                          act="gelu")
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    ref, bound = oracle.sgemm_batched(As, Bs, Cs, alpha, 0.5, biases, "gelu")
    for b in range(batch):
        assert_within_bound(got[b], ref[b], bound[b], f"{case} batch {b}")


def test_single_batch_plain_matches_sgemm_bitwise():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    A, B, C = make_inputs(700, 530, 300, "upm1", "upm1", "normal", seed=13)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c1 = torch.from_numpy(C).cuda()
    c2 = c1.clone()
    binding.sgemm_into(dA, dB, c1, 1.5, 0.5)
    binding.sgemm_ex_into(dA, dB, c2, 1.5, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_deterministic_run_to_run():
    batch, M, N, K = 3, 600, 500, 700
    As, Bs, Cs = _inputs(batch, M, N, K, seed=14)
    rng = np.random.default_rng(15)
    biases = [rng.standard_normal(N).astype(np.float32) for _ in range(batch)]
    g1 = _run(As, Bs, Cs, 1.0, 0.25, biases, "gelu")
    g2 = _run(As, Bs, Cs, 1.0, 0.25, biases, "gelu")
    assert np.array_equal(g1, g2)


def test_overlapping_c_batches_rejected():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    A = torch.zeros((2, 8, 8), device="cuda")
    B = torch.zeros((2, 8, 8), device="cuda")
    flat = torch.zeros(8 * 8 + 8, device="cuda")
    C = flat.as_strided((2, 8, 8), (8, 8, 1))      # batch 1 starts inside batch 0
    with pytest.raises(binding.SgemmError) as e:
        binding.sgemm_ex_into(A, B, C, 1.0, 0.0)
    assert e.value.status == binding.SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.extended])
def test_full_size_workload_sampled_rows(name):
    """The batched and fused workloads at full size, in the configuration the
    benchmark times: sampled rows (every column) of the first, a middle and the
    last batch against the oracle."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    w = WORKLOADS[name]
    A, B, C = workload_inputs(w)
    bias = workload_bias(w)
    if w.batch == 1:
        A, B = A[None], B[None]
        C = None if C is None else C[None]
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = (torch.from_numpy(C).cuda() if C is not None
          else torch.full((w.batch, w.M, w.N), float("nan"), device="cuda"))
    dbias = None if bias is None else torch.from_numpy(bias).cuda()
    binding.sgemm_ex_into(dA, dB, dC, w.alpha, w.beta, bias=dbias, act=w.act)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    rows, _ = sample_indices(w)
    for b in sorted({0, w.batch // 2, w.batch - 1}):
        ref, bound = oracle.sgemm_ex_rows(A[b], B[b], None if C is None else C[b], w.alpha,
                                          w.beta, None if bias is None else bias[b], w.act, rows)
        got = dC[b][torch.from_numpy(rows).cuda()].cpu().numpy()
        assert_within_bound(got, ref, bound, f"{name} batch {b}")
    assert torch.isfinite(dC).all()


def test_batch_count_past_the_grid_limit():
    """70,000 batches: past the 65,535 blocks a launch may have along z, so
    the per-batch A transpose runs in two launches and the per-batch B copy
    (rows of 5 floats, re-pitched) walks its batches in a grid-stride loop.
    Integer inputs; up to 129 batches, those next to each launch's z range among
    them, checked bit for bit against the oracle."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    batch, M, N, K = 70000, 3, 5, 7
    rng = np.random.default_rng(31)
    A = rng.integers(-4, 5, (batch, M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (batch, K, N)).astype(np.float32)
    C = rng.integers(-4, 5, (batch, M, N)).astype(np.float32)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    binding.sgemm_ex_into(dA, dB, dC, 1.5, 0.5)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    got = dC.cpu().numpy()
    # the batches on both sides of each launch's z range, the first and the
    # last, and a seeded sample of the rest (one oracle call per batch)
    picks = sorted({0, 1, 65533, 65534, 65535, 65536, 65537, batch - 2, batch - 1}
                   | set(rng.choice(batch, 120, replace=False).tolist()))
    ref, _ = oracle.sgemm_batched([A[b] for b in picks], [B[b] for b in picks],
                                  [C[b] for b in picks], 1.5, 0.5, None, "none", threads=1,
                                  with_bound=False)
    assert np.array_equal(got[picks], ref)
