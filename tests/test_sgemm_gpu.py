"""GPU parity of the SGEMM path against the CPU oracle (small and ragged shapes,
edge cases, failure detection).  Every call goes through the C ABI."""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs
from _helpers import assert_within_bound, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    from dense_fp32_gemm_02_gb300 import binding  # noqa: F401  (fails loudly if not built)
    yield


@pytest.fixture(params=["auto", "tma"])
def kernel(request):
    """Run a test twice: with the library's own choice (problems too small for
    the persistent kernel take the direct small-problem kernel) and with the
    persistent TMA kernel forced (variant 0), so both stay covered at small
    and ragged shapes."""
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(0 if request.param == "tma" else -1)
    yield request.param
    binding.set_variant(-1)


SIZES_MN = [1, 7, 33, 64, 127, 128, 129, 255, 257]
SIZES_K = [1, 5, 16, 17, 33, 100]


@pytest.mark.parametrize("K", SIZES_K)
def test_integer_inputs_bit_exact_over_shape_grid(K, kernel):
    """Integer inputs in [-4, 4]: every partial sum is an exact integer, so any
    summation order gives the oracle's bits.  alpha=1.5, beta=0.5 with integer
    C keeps the epilogue exact too."""
    for M in SIZES_MN:
        for N in SIZES_MN:
            A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=M * 1000 + N * 10 + K)
            ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
            got = run_gpu(A, B, C, 1.5, 0.5).cpu().numpy()
            assert np.array_equal(got, ref), (M, N, K)


@pytest.mark.parametrize("M,N,K", [(300, 200, 100), (129, 257, 513), (1000, 33, 77),
                                   (5, 1100, 260), (640, 640, 640)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, 0.5), (-0.75, 1.0), (2.0, -3.0)])
def test_random_parity_within_bound(M, N, K, alpha, beta, kernel):
    A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=M + N + K)
    ref, bound = oracle.sgemm(A, B, C if beta != 0 else None, alpha, beta)
    got = run_gpu(A, B, C if beta != 0 else None, alpha, beta).cpu().numpy()
    assert_within_bound(got, ref, bound, f"{M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("pads,offsets", [((3, 5, 2), (0, 0, 0)), ((0, 0, 0), (1, 1, 1)),
                                          ((4, 4, 4), (0, 2, 3)), ((1, 0, 7), (3, 0, 0))])
def test_leading_dimensions_and_alignment(pads, offsets, kernel):
    """Row pitches above the minimum with NaN padding, and base addresses that
    are 4-byte but not 16-byte aligned: the TMA rule is met by the packing
    pass; NaN padding must never reach the result; C padding stays untouched."""
    M, N, K = 203, 157, 141
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=7,
                          lda=K + pads[0], ldb=N + pads[1], ldc=N + pads[2])
    ref, bound = oracle.sgemm(A, B, C, 1.0, 1.0)
    dC = run_gpu(A, B, C, 1.0, 1.0, offsets=offsets)
    got = dC.cpu().numpy()
    assert np.isfinite(got).all()
    assert_within_bound(got, ref, bound, f"pads={pads} offsets={offsets}")
    if pads[2]:
        full = dC.as_strided((M, N + pads[2]), (N + pads[2], 1)).cpu().numpy()
        assert np.isnan(full[:, N:]).all(), "C padding columns were written"


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("ldc_pad,c_off", [(0, 0), (2, 1), (3, 3), (4, 2)])
def test_staged_epilogue_rows_not_16_byte_aligned(variant, ldc_pad, c_off):
    """Rows of C that do not all start 16-byte aligned (odd row pitch, or a
    base 4 or 12 bytes past a 16-byte boundary), with beta != 0 and a short K,
    take the staged epilogue on both tile orientations: the whole C within the
    bound, the padding columns beyond N untouched, and integer inputs bit-exact."""
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 515, 1003, 300
    binding.set_variant(variant)
    try:
        for dist, exact in (("upm1", False), ("int4", True)):
            A, B, C = make_inputs(M, N, K, dist, dist, "int4" if exact else "normal",
                                  seed=variant * 10 + ldc_pad, ldc=N + ldc_pad)
            ref, bound = oracle.sgemm(A, B, C, 1.5, 0.5)
            dC = run_gpu(A, B, C, 1.5, 0.5, offsets=(0, 0, c_off))
            got = dC.cpu().numpy()
            if exact:
                assert np.array_equal(got, ref), (variant, ldc_pad, c_off)
            else:
                assert_within_bound(got, ref, bound, f"variant {variant} ldc+{ldc_pad} off {c_off}")
            if ldc_pad:
                full = dC.as_strided((M, N + ldc_pad), (N + ldc_pad, 1)).cpu().numpy()
                assert np.isnan(full[:, N:]).all(), "C padding columns were written"
    finally:
        binding.set_variant(-1)


@pytest.mark.parametrize("M,N,K", [
    (64, 64, 128),      # 4 tiles of 32x32: split in two (two k steps each)
    (33, 95, 200),      # 12 tiles, ragged: split in four
    (256, 256, 256),    # the 256^3 workload: 64 tiles x 4 CTAs
    (7, 5, 1000),       # one tile: split in eight
    (100, 130, 4099),   # 20 tiles, K not a multiple of 32: split in eight
])
def test_small_problem_k_split_over_clusters(M, N, K):
    """Small problems whose 32x32 tiles fill at most half the SMs split the k
    range over a cluster's CTAs, CTA 0 adding the others' partial sums in a
    fixed order: integer inputs bit-exact (any order is exact), random inputs
    within the bound, misaligned operands and padded pitches included, and
    bitwise the same on a second call."""
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=M + N + K, lda=K + 3, ldc=N + 1)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    got = run_gpu(A, B, C, 1.5, 0.5, offsets=(1, 2, 3)).cpu().numpy()
    assert np.array_equal(got, ref), (M, N, K)
    A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=M * N + K)
    ref, bound = oracle.sgemm(A, B, C, -0.75, 1.25)
    first = run_gpu(A, B, C, -0.75, 1.25).cpu().numpy()
    second = run_gpu(A, B, C, -0.75, 1.25).cpu().numpy()
    assert_within_bound(first, ref, bound, f"split-K {M}x{N}x{K}")
    assert np.array_equal(first, second), "split-K result changed between calls"
    assert binding.device_status() == binding.SGEMM_OK


# Shapes whose chosen orientation of the default tile makes fewer tiles than a
# quarter of the SMs run the 128x128x48 tile (variant 9): twice the tiles, so
# stream-K cuts each into half as many pieces.  All of these are above the
# small-problem kernel's threshold and have more than 32 rows and columns.
FEW_TILE_SHAPES = [(1024, 1024, 1024), (768, 768, 768), (64, 3001, 1023), (256, 3001, 1023),
                   (512, 512, 2048), (130, 700, 4000)]


@pytest.mark.parametrize("M,N,K", FEW_TILE_SHAPES)
def test_few_tile_shapes_take_the_128x128_tile_and_match_oracle(M, N, K):
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = min(-(-M // 256) * -(-N // 128), -(-M // 128) * -(-N // 256))
    name = binding.config_string(M, N, K)
    if 4 * tiles < sms:
        assert "tile=128x128x48" in name, name
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=M + 7 * N + K)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    got = run_gpu(A, B, C, 1.5, 0.5).cpu().numpy()
    assert np.array_equal(got, ref), (M, N, K)
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=M + 7 * N + K + 1)
    ref, bound = oracle.sgemm(A, B, C, -0.75, 1.25)
    got = run_gpu(A, B, C, -0.75, 1.25).cpu().numpy()
    assert_within_bound(got, ref, bound, f"few tiles {M}x{N}x{K}")


def test_config_string_reports_the_work_split_on_this_device():
    """With a device current, the configuration text says when the work split
    leaves the stream-K tail out: 16384x16384x512 is 8192 tiles of 256x128, 54
    waves of 152 with 0.2 % of the slots idle; 8192^3 (2048 tiles, 3.8 % idle)
    keeps the tail."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the split of these shapes assumes 152 SMs")
    assert "whole tiles only" in binding.config_string(16384, 16384, 512)
    assert "whole tiles only" not in binding.config_string(8192, 8192, 8192)


def test_edge_rows_and_columns_not_written_outside_block(kernel):
    """Guard band: C is a window inside a NaN-filled buffer; nothing outside the
    M x N window may change."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 130, 70, 40
    A, B, _ = make_inputs(M, N, K, "upm1", "upm1", None, seed=3)
    big = torch.full((M + 4, N + 40), float("nan"), device="cuda")
    win = big[2:2 + M, 3:3 + N]
    binding.sgemm_into(to_device(A), to_device(B), win, 1.0, 0.0)
    torch.cuda.synchronize()
    ref, bound = oracle.sgemm(A, B, None, 1.0, 0.0)
    assert_within_bound(win.cpu().numpy(), ref, bound, "window")
    h = big.cpu().numpy()
    mask = np.ones_like(h, dtype=bool)
    mask[2:2 + M, 3:3 + N] = False
    assert np.isnan(h[mask]).all()


def test_beta_zero_does_not_read_c(kernel):
    M, N, K = 150, 140, 130
    A, B, _ = make_inputs(M, N, K, "upm1", "upm1", None, seed=5)
    C = np.full((M, N), np.nan, np.float32)
    ref, bound = oracle.sgemm(A, B, None, 1.0, 0.0)
    got = run_gpu(A, B, C, 1.0, 0.0).cpu().numpy()
    assert np.isfinite(got).all()
    assert_within_bound(got, ref, bound, "beta=0")


@pytest.mark.parametrize("K,alpha,beta", [(0, 1.0, 0.5), (0, 1.0, 0.0), (64, 0.0, -2.0),
                                          (64, 0.0, 0.0)])
def test_quick_returns_scale_c(K, alpha, beta):
    M, N = 37, 45
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=9)
    if alpha == 0.0:
        A = A.copy()
        A[0, 0] = np.inf       # A must not be read when alpha == 0
    ref, _ = oracle.sgemm(A, B, C, alpha, beta)
    got = run_gpu(A, B, C, alpha, beta).cpu().numpy()
    assert np.array_equal(got, ref)


def test_empty_sizes_are_no_ops():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    for (M, N, K) in [(0, 5, 3), (5, 0, 3), (0, 0, 0)]:
        A = torch.zeros((M, K), device="cuda")
        B = torch.zeros((K, N), device="cuda")
        C = torch.zeros((M, N), device="cuda")
        binding.sgemm_into(A, B, C, 1.0, 1.0)
    torch.cuda.synchronize()


def test_ones_times_twos_small_shapes_exact():
    for (M, N, K) in [(1, 1, 1), (7, 13, 29), (128, 128, 128), (129, 255, 511), (512, 512, 512)]:
        A = np.ones((M, K), np.float32)
        B = np.full((K, N), 2.0, np.float32)
        got = run_gpu(A, B, None, 1.0, 0.0).cpu().numpy()
        assert (got == 2 * K).all(), (M, N, K)


def test_bitwise_deterministic_run_to_run():
    """The race check of the tiling exercise (missing-barrier bug, exercise 5):
    a race shows up as results that change between runs."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 1031, 777, 1500
    A, B, C = make_inputs(M, N, K, "normal", "normal", "normal", seed=11)
    dA, dB = to_device(A), to_device(B)
    outs = []
    for _ in range(3):
        dC = to_device(C)
        binding.sgemm_into(dA, dB, dC, 1.0, 1.0)
        outs.append(dC.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_host_entry_point_matches_device_entry_point():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 321, 283, 259
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=13)
    dev = run_gpu(A, B, C, 0.5, 2.0).cpu()
    hA = torch.from_numpy(np.ascontiguousarray(A)).pin_memory()
    hB = torch.from_numpy(np.ascontiguousarray(B)).pin_memory()
    hC = torch.from_numpy(np.ascontiguousarray(C)).pin_memory()
    binding.sgemm_host(hA, hB, hC, 0.5, 2.0)
    assert torch.equal(hC, dev)
    # pageable memory with a row pitch
    A2, B2, C2 = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=13, lda=K + 3, ldb=N + 1,
                             ldc=N + 5)
    tA, tB = torch.from_numpy(A2.base)[:, :K], torch.from_numpy(B2.base)[:, :N]
    cbuf = torch.from_numpy(C2.base.copy())
    binding.sgemm_host(tA, tB, cbuf[:, :N], 0.5, 2.0)
    assert torch.equal(cbuf[:, :N], dev)
    assert torch.isnan(cbuf[:, N:]).all()


def test_runs_on_a_non_default_stream():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 260, 250, 240
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=17)
    ref, bound = oracle.sgemm(A, B, C, 1.0, 1.0)
    s = torch.cuda.Stream()
    dA, dB, dC = to_device(A), to_device(B), to_device(C)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        binding.sgemm_into(dA, dB, dC, 1.0, 1.0)
    s.synchronize()
    assert_within_bound(dC.cpu().numpy(), ref, bound, "side stream")


def test_bounded_wait_expiry_is_reported_and_context_survives():
    """Failure detection without a GPU fault: a barrier wait that nothing
    completes expires after 2 ms, the kernel reports it and returns; the
    context stays usable and the next GEMM is correct."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    assert binding.device_status() == binding.SGEMM_OK
    assert binding.selftest_wait_timeout(2_000_000) == binding.SGEMM_ERR_TIMEOUT
    assert binding.device_status() == binding.SGEMM_OK     # word was cleared
    M, N, K = 140, 150, 160
    A, B, _ = make_inputs(M, N, K, "upm1", "upm1", None, seed=19)
    ref, bound = oracle.sgemm(A, B, None, 1.0, 0.0)
    got = run_gpu(A, B, None, 1.0, 0.0).cpu().numpy()
    assert_within_bound(got, ref, bound, "after self test")
    assert binding.device_status() == binding.SGEMM_OK


def test_binding_rejects_bad_tensors():
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    A = torch.zeros((4, 4), device="cuda")
    with pytest.raises(TypeError):
        binding.sgemm_into(A.double(), A, A)
    with pytest.raises(ValueError):
        binding.sgemm_into(A, torch.zeros((3, 4), device="cuda"), A)
    with pytest.raises(ValueError):
        binding.sgemm_into(A, A, A.t())     # C columns not contiguous


def test_kernel_launches_are_counted():
    """A problem too small for the persistent kernel is one launch of the
    direct kernel; a larger one is the A transpose plus the main kernel."""
    from dense_fp32_gemm_02_gb300 import binding
    before = binding.kernel_launch_count()
    A, B, _ = make_inputs(64, 64, 64, seed=23)
    run_gpu(A, B, None, 1.0, 0.0)
    assert binding.kernel_launch_count() - before == 1     # small-problem kernel
    before = binding.kernel_launch_count()
    A, B, _ = make_inputs(1024, 1024, 1024, seed=24)
    run_gpu(A, B, None, 1.0, 0.0)
    assert binding.kernel_launch_count() - before == 2     # A transpose + main kernel


@pytest.mark.parametrize("M,N,K", [(600, 520, 300), (257, 1031, 95), (1, 300, 17)])
def test_every_kernel_variant_matches_oracle(M, N, K):
    """Each compiled tile configuration, forced in turn: integer inputs bit-exact
    and random inputs within the bound, on shapes that leave ragged tiles."""
    from dense_fp32_gemm_02_gb300 import binding
    try:
        for v in range(len(binding.variants())):
            binding.set_variant(v)
            A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=v + 100)
            ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
            got = run_gpu(A, B, C, 1.5, 0.5).cpu().numpy()
            assert np.array_equal(got, ref), (v, M, N, K)
            A, B, C = make_inputs(M, N, K, "normal", "upm1", "normal", seed=v + 200)
            ref, bound = oracle.sgemm(A, B, C, -1.25, 0.75)
            got = run_gpu(A, B, C, -1.25, 0.75).cpu().numpy()
            assert_within_bound(got, ref, bound, f"variant {v}")
    finally:
        binding.set_variant(-1)


@pytest.mark.parametrize("M,N,K", [
    (5120, 1152, 512),    # 180 tiles of 256x128: one whole-tile wave, 28 tiles split over all CTAs
    (512, 256, 64),       # 4 tiles, 2 slabs each: every tile split in two pieces
    (300, 4000, 16),      # one slab per tile: stream-K pieces are whole tiles, some CTAs idle
    (2048, 2048, 1056),   # 128 tiles, 33 slabs: the whole problem is stream-K
    (200, 100, 16384),    # one tile of 256 slabs: its pieces sit on every CTA
    (3, 5, 100003),       # one tile of 1563 slabs; rows of A, B and C not 16-byte aligned
])
def test_stream_k_split_matches_oracle(M, N, K, kernel):
    """Shapes whose leftover tiles are split along k between CTAs: integer
    inputs must stay bit-exact (any order of exact partial sums), random inputs
    within the bound, and two runs must agree bitwise (the partial sums are
    added in a fixed order whichever piece finishes last)."""
    import torch
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=M + K)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5, with_bound=False)
    got = run_gpu(A, B, C, 1.5, 0.5).cpu().numpy()
    assert np.array_equal(got, ref)
    A, B, C = make_inputs(M, N, K, "normal", "normal", "normal", seed=M + K + 1)
    ref, bound = oracle.sgemm(A, B, C, 0.5, -1.5)
    g1 = run_gpu(A, B, C, 0.5, -1.5).cpu()
    g2 = run_gpu(A, B, C, 0.5, -1.5).cpu()
    assert torch.equal(g1, g2)
    assert_within_bound(g1.numpy(), ref, bound, f"stream-K {M}x{N}x{K}")


@pytest.mark.parametrize("tensor_cores", [False, True])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_point_pipelined_over_row_blocks(tensor_cores, pinned):
    """M = 4100 splits into row blocks (copy in, multiply, copy back overlap):
    1024, 1280, 1284 and 512 rows on the FFMA path, four of 1025 on the 3xTF32
    path; padded leading dimensions and beta != 0; checked against the oracle
    on rows at every block boundary of both and on columns."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 4100, 777, 515
    A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=31, lda=K + 3, ldb=N + 1,
                          ldc=N + 5)
    tA = torch.from_numpy(A.base.copy())[:, :K]
    tB = torch.from_numpy(B.base.copy())[:, :N]
    cbuf = torch.from_numpy(C.base.copy())
    if pinned:
        tA = torch.from_numpy(A.base.copy()).pin_memory()[:, :K]
        tB = torch.from_numpy(B.base.copy()).pin_memory()[:, :N]
        cbuf = cbuf.pin_memory()
    binding.sgemm_host(tA, tB, cbuf[:, :N], 1.25, -0.5, tensor_cores=tensor_cores)
    rows = np.array([0, 1, 1023, 1024, 1025, 2049, 2050, 2303, 2304, 3075, 3076, 3587, 3588, 4099],
                    np.int64)
    cols = np.array([0, 5, 300, 776], np.int64)
    got = cbuf.numpy()
    ref, bound = oracle.sgemm_rows(A, B, C, 1.25, -0.5, rows)
    assert_within_bound(got[rows, :N], ref, bound, "host rows")
    ref, bound = oracle.sgemm_cols(A, B, C, 1.25, -0.5, cols)
    assert_within_bound(got[:, cols], ref, bound, "host cols")
    assert np.isnan(got[:, N:]).all(), "C padding written"
    assert binding.device_status() == binding.SGEMM_OK


@pytest.mark.parametrize("tensor_cores", [False, True])
def test_host_entry_point_first_block_in_k_chunks(tensor_cores):
    """K >= 4096: block 0 is multiplied in k-chunks of A and B as they
    arrive, accumulating into its rows of C.  FFMA path: chunks of 576, 896,
    1344 and 1284 (K/8 first, each next one half again as long, the last not a
    multiple of the tile depth), blocks of 1024 and 1076 rows, the first chunk
    with beta = 0 and beta * C_in added once C_in has arrived; 3xTF32 path:
    four chunks of 1088, 1088, 1088 and 836, two blocks of 1050 rows, C_in
    copied in front.  The other block takes the whole of K.  beta != 0 and
    padded leading dimensions; oracle on rows at both plans' boundaries and on
    columns."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 2100, 300, 4100
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=37, lda=K + 1, ldb=N + 3,
                          ldc=N + 2)
    tA = torch.from_numpy(A.base.copy()).pin_memory()[:, :K]
    tB = torch.from_numpy(B.base.copy()).pin_memory()[:, :N]
    cbuf = torch.from_numpy(C.base.copy()).pin_memory()
    binding.sgemm_host(tA, tB, cbuf[:, :N], 0.75, 1.5, tensor_cores=tensor_cores)
    rows = np.array([0, 1, 777, 1023, 1024, 1025, 1049, 1050, 2099], np.int64)
    cols = np.array([0, 150, 299], np.int64)
    got = cbuf.numpy()
    ref, bound = oracle.sgemm_rows(A, B, C, 0.75, 1.5, rows)
    assert_within_bound(got[rows, :N], ref, bound, "chunked host rows")
    ref, bound = oracle.sgemm_cols(A, B, C, 0.75, 1.5, cols)
    assert_within_bound(got[:, cols], ref, bound, "chunked host cols")
    assert np.isnan(got[:, N:]).all(), "C padding written"
    assert binding.device_status() == binding.SGEMM_OK


@pytest.mark.parametrize("tensor_cores", [False, True])
def test_host_entry_point_k_chunks_with_beta_zero_never_read_c(tensor_cores):
    """K >= 4096 and beta = 0: block 0's chunks start from beta = 0 with no
    C_in to add, and C_in (NaN here) is never copied in or read."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 2300, 260, 4096
    A, B, _ = make_inputs(M, N, K, "upm1", "upm1", None, seed=41)
    tA = torch.from_numpy(np.ascontiguousarray(A)).pin_memory()
    tB = torch.from_numpy(np.ascontiguousarray(B)).pin_memory()
    hC = torch.full((M, N), float("nan")).pin_memory()
    binding.sgemm_host(tA, tB, hC, -1.5, 0.0, tensor_cores=tensor_cores)
    rows = np.array([0, 1023, 1024, 1276, 2299], np.int64)
    ref, bound = oracle.sgemm_rows(A, B, None, -1.5, 0.0, rows)
    got = hC.numpy()
    assert not np.isnan(got).any()
    assert_within_bound(got[rows], ref, bound, "beta = 0 chunked host rows")


def test_last_kernel_names_the_kernel_each_call_ran():
    """sgemm_last_kernel reports the main kernel of the thread's last call: the
    small-problem kernel, the few-tiles tile, the default tile, the tall-batch
    and batched kernels of sgemm_ex, a 3xTF32 kernel, the scale-only kernel."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    dev = "cuda"

    def run(M, N, K, alpha=1.0):
        A = torch.ones((M, K), device=dev)
        B = torch.ones((K, N), device=dev)
        C = torch.zeros((M, N), device=dev)
        binding.sgemm_into(A, B, C, alpha, 0.0)
        torch.cuda.synchronize()
        return binding.last_kernel()

    assert run(256, 256, 256).startswith("direct small-problem kernel")
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert "tile=128x128x48" in run(1024, 1024, 1024)
    assert "tile=256x128x64" in run(4096, 4096, 256)
    assert run(300, 300, 300, alpha=0.0) == "scale only (C = beta * C)"
    A3 = torch.ones((4, 512, 128), device=dev)
    B3 = torch.ones((4, 128, 256), device=dev)
    C3 = torch.zeros((4, 512, 256), device=dev)
    binding.sgemm_ex_into(A3, B3, C3, 1.0, 0.0)
    assert "tall_batch" in binding.last_kernel()
    binding.sgemm_ex_into(A3, B3, C3, 1.0, 0.0, act="relu")
    assert "batched+epilogue" in binding.last_kernel()
    A = torch.ones((1024, 512), device=dev)
    B = torch.ones((512, 1024), device=dev)
    C = torch.zeros((1024, 1024), device=dev)
    binding.sgemm_3xtf32_into(A, B, C, 1.0, 0.0)
    torch.cuda.synchronize()
    assert binding.last_kernel().startswith("3xtf32")
    assert torch.all(C == 512.0)
    assert torch.all(C3 == 128.0)


# GEMMs of at most 32 rows (above the small-problem threshold) run the
# skinny-M kernel: B streamed once, the k range split over the grid and the
# partial sums added in order.  17 rows is just past the 16-row configuration;
# 33 rows is past the skinny range and runs the persistent kernel.
SKINNY_M = [1, 2, 3, 4, 5, 8, 9, 16, 17, 31, 32, 33]
SKINNY_NK = [(3001, 1023), (1000, 5000), (300, 4100)]


@pytest.mark.parametrize("N,K", SKINNY_NK)
def test_skinny_rows_bit_exact_on_integer_inputs(N, K):
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    for M in SKINNY_M:
        A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=41 + M + N)
        ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
        got = run_gpu(A, B, C, 1.5, 0.5).cpu().numpy()
        assert np.array_equal(got, ref), (M, N, K)
        assert ("skinny" in binding.last_kernel()) == (M <= 32), (M, binding.last_kernel())


@pytest.mark.parametrize("M", [1, 7, 16, 32])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.75, 1.25)])
def test_skinny_rows_random_parity(M, alpha, beta):
    N, K = 2500, 3000
    A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=42 + M)
    ref, bound = oracle.sgemm(A, B, C if beta != 0 else None, alpha, beta)
    got = run_gpu(A, B, C if beta != 0 else None, alpha, beta).cpu().numpy()
    assert_within_bound(got, ref, bound, f"skinny {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("offsets,ldc_pad", [((1, 3, 2), 0), ((0, 0, 0), 5), ((3, 1, 0), 3)])
def test_skinny_rows_misaligned_and_padded(offsets, ldc_pad):
    """Pointers off 16-byte boundaries, odd pitches and a padded C: the skinny
    kernel has no alignment rule, and C's padding columns stay untouched."""
    import torch
    from _helpers import to_device
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 6, 2049, 1537
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=43)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    dA = to_device(A, offset_elems=offsets[0])
    dB = to_device(B, offset_elems=offsets[1])
    full = torch.full((M, N + ldc_pad + offsets[2]), 777.0, device="cuda")
    full[:, offsets[2]:offsets[2] + N] = torch.from_numpy(C).cuda()
    dC = full[:, offsets[2]:offsets[2] + N]
    binding.sgemm_into(dA, dB, dC, 1.5, 0.5)
    torch.cuda.synchronize()
    assert "skinny" in binding.last_kernel()
    assert np.array_equal(dC.cpu().numpy(), ref)
    rest = torch.cat([full[:, :offsets[2]], full[:, offsets[2] + N:]], dim=1)
    assert bool((rest == 777.0).all()), "columns outside C written"


def test_skinny_rows_one_k_range_and_nan_c():
    """N wide enough that every SM gets column blocks without splitting K: the
    blocks write C themselves (no partial sums); beta 0 leaves NaN in C_in
    unread."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 4, 320000, 100
    A, B, _ = make_inputs(M, N, K, "int4", "int4", "int4", seed=44)
    ref, _ = oracle.sgemm(A, B, None, 2.0, 0.0)
    got = run_gpu(A, B, None, 2.0, 0.0).cpu().numpy()
    assert "skinny" in binding.last_kernel()
    assert np.array_equal(got, ref)


# GEMMs of at most 32 columns (above the small-problem threshold, more than 32
# rows) run the skinny-N kernel: A streamed once, 256 rows per block, the k
# range split over the grid and the partial sums added in order.  33 columns
# runs the persistent kernel.
SKINNY_N = [1, 2, 3, 4, 5, 8, 9, 16, 17, 31, 32, 33]
SKINNY_MK = [(3001, 1023), (5000, 1000), (600, 4100)]


@pytest.mark.parametrize("M,K", SKINNY_MK)
def test_skinny_columns_bit_exact_on_integer_inputs(M, K):
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    for N in SKINNY_N:
        A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=51 + M + N)
        ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
        got = run_gpu(A, B, C, 1.5, 0.5).cpu().numpy()
        assert np.array_equal(got, ref), (M, N, K)
        assert ("skinny-N" in binding.last_kernel()) == (N <= 32), (N, binding.last_kernel())


@pytest.mark.parametrize("N", [1, 7, 16, 32])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.75, 1.25)])
def test_skinny_columns_random_parity(N, alpha, beta):
    M, K = 2500, 3000
    A, B, C = make_inputs(M, N, K, "upm1", "normal", "normal", seed=52 + N)
    ref, bound = oracle.sgemm(A, B, C if beta != 0 else None, alpha, beta)
    got = run_gpu(A, B, C if beta != 0 else None, alpha, beta).cpu().numpy()
    assert_within_bound(got, ref, bound, f"skinny-N {M}x{N}x{K} a={alpha} b={beta}")


@pytest.mark.parametrize("offsets,ldc_pad", [((1, 3, 2), 0), ((0, 0, 0), 5), ((3, 1, 0), 3)])
def test_skinny_columns_misaligned_and_padded(offsets, ldc_pad):
    import torch
    from _helpers import to_device
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 2049, 6, 1537
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=53)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    dA = to_device(A, offset_elems=offsets[0])
    dB = to_device(B, offset_elems=offsets[1])
    full = torch.full((M, N + ldc_pad + offsets[2]), 777.0, device="cuda")
    full[:, offsets[2]:offsets[2] + N] = torch.from_numpy(C).cuda()
    dC = full[:, offsets[2]:offsets[2] + N]
    binding.sgemm_into(dA, dB, dC, 1.5, 0.5)
    torch.cuda.synchronize()
    assert "skinny-N" in binding.last_kernel()
    assert np.array_equal(dC.cpu().numpy(), ref)
    rest = torch.cat([full[:, :offsets[2]], full[:, offsets[2] + N:]], dim=1)
    assert bool((rest == 777.0).all()), "columns outside C written"


def test_skinny_columns_one_k_range_and_nan_c():
    """M tall enough that every SM gets row blocks without splitting K: the
    blocks write C themselves; beta 0 leaves NaN in C_in unread."""
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 160000, 4, 64
    A, B, _ = make_inputs(M, N, K, "int4", "int4", "int4", seed=54)
    ref, _ = oracle.sgemm(A, B, None, 2.0, 0.0)
    got = run_gpu(A, B, None, 2.0, 0.0).cpu().numpy()
    assert "skinny-N" in binding.last_kernel()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (64, 64, 200), (8, 3001, 1023), (3001, 8, 1023),
                                   (1024, 1024, 1024), (4096, 4096, 256), (4097, 3001, 1023),
                                   (16384, 16384, 64)])
def test_config_string_names_the_kernel_sgemm_runs(M, N, K):
    """With a device, sgemm_config_string makes the choice sgemm() makes: the
    text names the kernel that the call then records as launched.  (beta 0:
    the staged-epilogue form, which depends on C's alignment and beta, is
    outside what the shape alone decides.)"""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    binding.set_variant(-1)
    A = torch.ones((M, K), device="cuda")
    B = torch.ones((K, N), device="cuda")
    C = torch.full((M, N), float("nan"), device="cuda")
    binding.sgemm_into(A, B, C, 1.0, 0.0)
    torch.cuda.synchronize()
    assert binding.config_string(M, N, K).startswith(binding.last_kernel()), (
        binding.config_string(M, N, K), binding.last_kernel())
    assert bool((C == K).all())


@pytest.mark.parametrize("M,N,K", [(8, 3001, 1023), (2000, 8, 2048)])
def test_host_entry_point_on_skinny_shapes(M, N, K):
    """Host buffers on a skinny-M and a skinny-N shape of fewer than 2048 rows:
    the host path runs them as one row block on the same kernel as sgemm(),
    bitwise equal to the device entry point and bit-exact against the oracle
    on integer inputs."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=61 + M)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    dev = run_gpu(A, B, C, 1.5, 0.5).cpu()
    assert "skinny" in binding.last_kernel()
    hA = torch.from_numpy(np.ascontiguousarray(A)).pin_memory()
    hB = torch.from_numpy(np.ascontiguousarray(B)).pin_memory()
    hC = torch.from_numpy(np.ascontiguousarray(C)).pin_memory()
    binding.sgemm_host(hA, hB, hC, 1.5, 0.5)
    assert "skinny" in binding.last_kernel()
    assert torch.equal(hC, dev)
    assert np.array_equal(hC.numpy(), ref)
