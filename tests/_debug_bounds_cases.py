"""Cases run through the range-checked build of the library (started by
tests/test_debug_bounds_gpu.py in a subprocess with SGEMM_LIBRARY=debug_bounds).

Every kernel of that build checks the indices of its memory accesses and
reports an index out of range as SGEMM_ERR_BOUNDS.  Each case runs one entry
point, then requires SGEMM_OK from sgemm_device_status and a result within
the oracle's bound (bit-exact on integer inputs).  Prints "all cases in range"
at the end.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from dense_fp32_gemm_02_gb300 import binding  # noqa: E402
from dense_fp32_gemm_02_gb300.workloads import make_inputs  # noqa: E402
from _helpers import assert_within_bound, run_gpu, to_device  # noqa: E402


def status_ok(what):
    st = binding.device_status()
    if st != binding.SGEMM_OK:
        raise AssertionError(f"{what}: device status {binding.status_string(st)}")


def plain(M, N, K, alpha, beta, what, exact=False, offsets=(0, 0, 0), ldc_pad=0, entry=None):
    dist = "int4" if exact else "upm1"
    A, B, C = make_inputs(M, N, K, dist, dist, "int4" if exact else "normal",
                          seed=M + 3 * N + 7 * K, ldc=N + ldc_pad)
    c_in = C if beta != 0 else None
    ref, bound = oracle.sgemm(A, B, c_in, alpha, beta)
    if entry is None:
        got = run_gpu(A, B, c_in, alpha, beta, offsets=offsets).cpu().numpy()
    else:
        dA, dB = to_device(A, offset_elems=offsets[0]), to_device(B, offset_elems=offsets[1])
        dC = to_device(C if c_in is not None else np.full((M, N), np.nan, np.float32),
                       offset_elems=offsets[2])
        entry(dA, dB, dC, alpha, beta)
        torch.cuda.synchronize()
        got = dC.cpu().numpy()
    status_ok(what)
    if exact:
        assert np.array_equal(got, ref), what
    else:
        assert_within_bound(got, ref, bound, what)


def main():
    assert binding.lib.sgemm_debug_bounds_checks() == 1, "not the range-checked build"
    torch.cuda.set_device(0)
    # direct small-problem kernel and the default persistent kernel
    plain(7, 33, 5, 1.5, 0.5, "small 7x33x5", exact=True)
    plain(129, 257, 100, 1.5, 0.5, "small 129x257x100", exact=True)
    plain(640, 640, 640, 1.0, 0.0, "persistent 640^3")
    # every kernel variant, forced, on a ragged shape with beta (staged on 0 and 1)
    for v in range(binding.lib.sgemm_variant_count()):
        binding.set_variant(v)
        try:
            plain(300, 257, 129, 1.5, 0.5, f"variant {v}", exact=True)
            plain(300, 256, 129, -0.75, 1.0, f"variant {v}, aligned rows")
        finally:
            binding.set_variant(-1)
    # staged epilogue on both tiles: odd pitch, misaligned C; re-pitched B (fused pre-pass)
    for v in (0, 1):
        binding.set_variant(v)
        try:
            plain(515, 1003, 300, 1.5, 0.5, f"staged {v}", exact=True, offsets=(0, 1, 3), ldc_pad=2)
        finally:
            binding.set_variant(-1)
    plain(4097, 3001, 1023, 1.0, 1.0, "ragged 4097x3001x1023")
    # stream-K: one output tile split over every CTA
    plain(200, 100, 16384, 1.0, 0.5, "stream-K 200x100x16384", exact=True)
    # whole tiles only: 19 x 8 = 152 tiles of 256x128, one full wave, no stream-K
    plain(4864, 1024, 256, 1.0, 0.0, "whole tiles 4864x1024x256")
    # every tile by stream-K (64 slabs per tile): 128 tiles over all CTAs
    plain(2048, 2048, 4096, 1.5, 0.5, "all stream-K 2048x2048x4096", exact=True)
    # 3xTF32, both main kernels
    for pair in (False, True):
        binding.set_3xtf32_kernel(pair)
        try:
            plain(1024, 1024, 512, -0.75, 1.25, f"3xtf32 pair={pair}",
                  entry=binding.sgemm_3xtf32_into)
            plain(515, 1003, 300, 1.5, 0.5, f"3xtf32 ragged pair={pair}", exact=True,
                  entry=binding.sgemm_3xtf32_into)
        finally:
            binding.set_3xtf32_kernel(None)
    # the entry point without allocation
    plain(300, 257, 129, 1.5, 0.5, "noalloc", exact=True, offsets=(0, 1, 0),
          entry=binding.sgemm_noalloc_into)
    # batched with bias and GELU, odd batch strides; one GEMM with bias and ReLU
    batch, M, N, K = 3, 131, 97, 77
    As, Bs, Cs, bs = [], [], [], []
    for b in range(batch):
        A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=100 + b)
        As.append(A), Bs.append(B), Cs.append(C)
        bs.append(np.random.default_rng(200 + b).standard_normal(N).astype(np.float32))
    for act, nb in (("gelu", batch), ("relu", 1)):
        dA = torch.stack([torch.from_numpy(a) for a in As[:nb]]).cuda()
        dB = torch.stack([torch.from_numpy(b) for b in Bs[:nb]]).cuda()
        dC = torch.stack([torch.from_numpy(c) for c in Cs[:nb]]).cuda()
        dbias = torch.stack([torch.from_numpy(b) for b in bs[:nb]]).cuda()
        binding.sgemm_ex_into(dA, dB, dC, 1.25, 0.5, bias=dbias, act=act)
        torch.cuda.synchronize()
        status_ok(f"sgemm_ex {act} batch {nb}")
        ref, bound = oracle.sgemm_batched(As[:nb], Bs[:nb], Cs[:nb], 1.25, 0.5, bs[:nb], act)
        for b in range(nb):
            assert_within_bound(dC[b].cpu().numpy(), ref[b], bound[b], f"sgemm_ex {act} {b}")
    # skinny rows: k split over the grid (partial sums), and one k range per
    # block (N wide enough for every SM); odd pitches and misaligned pointers
    plain(5, 3001, 1023, 1.5, 0.5, "skinny 5x3001x1023", exact=True, offsets=(1, 3, 2))
    plain(32, 2049, 777, 1.5, 0.5, "skinny 32x2049x777", exact=True)
    plain(4, 320000, 64, 1.5, 0.5, "skinny one k range", exact=True)
    plain(3001, 5, 1023, 1.5, 0.5, "skinny-N 3001x5x1023", exact=True, offsets=(1, 3, 2))
    plain(2049, 32, 777, 1.5, 0.5, "skinny-N 2049x32x777", exact=True)
    plain(160000, 4, 64, 1.5, 0.5, "skinny-N one k range", exact=True)
    # batches run as one tall GEMM: contiguous B (48 tiles, all by stream-K),
    # and B re-pitched (rows of 203 floats) under a C with a padded pitch
    for batch, M, N, K, ldc in ((3, 512, 1000, 512, 1000), (2, 768, 203, 192, 207)):
        As, Bs, Cs = [], [], []
        for b in range(batch):
            A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=300 + b)
            As.append(A), Bs.append(B), Cs.append(C)
        dA = torch.stack([torch.from_numpy(a) for a in As]).cuda()
        dB = torch.stack([torch.from_numpy(b) for b in Bs]).cuda()
        full = torch.zeros((batch, M, ldc), device="cuda")
        full[:, :, :N] = torch.stack([torch.from_numpy(c) for c in Cs]).cuda()
        dC = full[:, :, :N]
        binding.sgemm_ex_into(dA, dB, dC, 1.5, 0.5)
        torch.cuda.synchronize()
        status_ok(f"tall batch {batch}x{M}x{N}x{K}")
        ref, _ = oracle.sgemm_batched(As, Bs, Cs, 1.5, 0.5, None, "none")
        for b in range(batch):
            assert np.array_equal(dC[b].cpu().numpy(), ref[b]), f"tall batch {b}"
    # host buffers (row blocks and k-chunks)
    A, B, C = make_inputs(2100, 300, 4100, "int4", "int4", "int4", seed=5)
    ref, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    hC = torch.from_numpy(C.copy())
    binding.sgemm_host(torch.from_numpy(A), torch.from_numpy(B), hC, 1.5, 0.5)
    status_ok("host buffers")
    assert np.array_equal(hC.numpy(), ref), "host buffers"
    # the abort path: an expiry, not an index out of range
    binding.set_wait_timeout_ns(2_000_000)
    binding.debug_drop_release(True)
    try:
        dA = torch.rand((4096, 512), device="cuda")
        dB = torch.rand((512, 1280), device="cuda")
        dC = torch.zeros((4096, 1280), device="cuda")
        binding.sgemm_into(dA, dB, dC, 1.0, 0.0)
        st = binding.device_status()
    finally:
        binding.debug_drop_release(False)
        binding.set_wait_timeout_ns(2_000_000_000)
    assert st == binding.SGEMM_ERR_TIMEOUT, binding.status_string(st)
    print("all cases in range", flush=True)


if __name__ == "__main__":
    main()
