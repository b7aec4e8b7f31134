"""Several host threads, each on its own CUDA stream, calling the library at the
same time: the FFMA path, the 3xTF32 path and the fused-epilogue entry point,
persistent, small-problem, skinny and tall-batch kernels mixed.  The calls share the library's
per-device state (pool, tensor-map encoder, launch counter) and the GPU, but no
workspace: every result must still match the oracle within its bound."""
import threading

import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs
from _helpers import assert_within_bound, to_device

pytestmark = pytest.mark.gpu

ALPHA, BETA = 1.25, -0.5
# (entry point, M, N, K, seed)
CASES = [
    ("ffma", 640, 520, 700, 301),
    ("tf32x3", 1030, 300, 257, 302),
    ("ffma", 257, 1100, 96, 303),      # small-problem kernel
    ("ex_relu", 300, 260, 130, 304),
    ("tf32x3", 900, 900, 900, 305),
    ("ffma", 900, 900, 900, 306),
    ("ex_relu", 1024, 768, 512, 307),
    ("ffma", 2048, 1024, 1056, 308),   # stream-K pieces
    ("ffma", 12, 3001, 1023, 309),     # skinny-M kernel (split K, partial sums)
    ("ffma", 3001, 6, 1023, 310),      # skinny-N kernel (split K, partial sums)
    ("tall4", 512, 256, 128, 311),     # 4 batches of 512 x 256 x 128 run as one tall GEMM
]
REPEATS = 4


def _expected(kind, A, B, C, bias):
    if kind == "ex_relu":
        return oracle.sgemm_ex_rows(A, B, C, ALPHA, BETA, bias, "relu")
    if kind == "tall4":
        return oracle.sgemm_batched(list(A), list(B), list(C), ALPHA, BETA, None, "none")
    return oracle.sgemm(A, B, C, ALPHA, BETA)


def test_concurrent_calls_from_host_threads_on_their_own_streams(cuda_device):
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    inputs = []
    for kind, M, N, K, seed in CASES:
        if kind == "tall4":
            parts = [make_inputs(M, N, K, "upm1", "upm1", "normal", seed=seed + 100 * b)
                     for b in range(4)]
            inputs.append(tuple(np.stack([p[x] for p in parts]) for x in range(3)) + (None,))
            continue
        A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed=seed)
        bias = (np.random.default_rng(seed).standard_normal(N).astype(np.float32)
                if kind == "ex_relu" else None)
        inputs.append((A, B, C, bias))
    results, errors = {}, {}
    start = threading.Barrier(len(CASES))

    def worker(i):
        try:
            kind = CASES[i][0]
            A, B, C, bias = inputs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                if kind == "tall4":
                    dA, dB, dC0 = (torch.from_numpy(x).cuda() for x in (A, B, C))
                else:
                    dA, dB, dC0 = to_device(A), to_device(B), to_device(C)
                dbias = torch.from_numpy(bias).cuda() if bias is not None else None
                start.wait(timeout=60)
                for _ in range(REPEATS):
                    dC = dC0.clone()
                    if kind == "ffma":
                        binding.sgemm_into(dA, dB, dC, ALPHA, BETA)
                    elif kind == "tf32x3":
                        binding.sgemm_3xtf32_into(dA, dB, dC, ALPHA, BETA)
                    elif kind == "tall4":
                        binding.sgemm_ex_into(dA, dB, dC, ALPHA, BETA)
                    else:
                        binding.sgemm_ex_into(dA, dB, dC, ALPHA, BETA, bias=dbias, act="relu")
            s.synchronize()
            results[i] = dC.cpu().numpy()
        except Exception as e:   # reported below, on the test's own thread
            errors[i] = e

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    assert binding.device_status() == 0
    for i, (kind, M, N, K, _) in enumerate(CASES):
        A, B, C, bias = inputs[i]
        ref, bound = _expected(kind, A, B, C, bias)
        if kind == "tall4":
            for b in range(4):
                assert_within_bound(results[i][b], ref[b], bound[b],
                                    f"{kind} batch {b} (thread {i})")
            continue
        assert_within_bound(results[i], ref, bound, f"{kind} {M}x{N}x{K} (thread {i})")
