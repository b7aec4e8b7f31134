"""Maximum sizes: element counts past 2^31 in C (FFMA and 3xTF32 paths) and in A
(the A transpose and its workspace), so every offset computation has to be
64-bit.  The inputs are closed-form integer patterns v[i][j] = ((a*i + b*j) mod 9)
- 4, built in chunks on the device and row by row on the host for the oracle:
every partial sum is an exact small integer, so the sampled outputs must match
the oracle bit for bit."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


def _host_pattern(rows, cols, a, b):
    """The pattern's rows `rows` (an index array) as float32."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(cols, dtype=np.int64)[None, :]
    return (((a * i + b * j) % 9) - 4).astype(np.float32)


def _device_pattern(rows, cols, a, b, chunk_rows):
    import torch
    out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    j = torch.arange(cols, dtype=torch.int64, device="cuda")[None, :]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        i = torch.arange(r0, r1, dtype=torch.int64, device="cuda")[:, None]
        out[r0:r1] = (((a * i + b * j) % 9) - 4).to(torch.float32)
    return out


@pytest.mark.parametrize("path", ["ffma", "3xtf32"])
def test_output_past_2_to_the_31_elements(cuda_device, path):
    """C of 49152 x 49152 (2.42e9 elements, 9.7 GB): rows before and after
    element 2^31 (row 43690) and the last row, bit-exact."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M = N = 49152
    K = 64
    assert M * N > 2 ** 31
    dA = _device_pattern(M, K, 7, 3, 8192)
    dB = _device_pattern(K, N, 5, 11, K)
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fn = binding.sgemm_into if path == "ffma" else binding.sgemm_3xtf32_into
    fn(dA, dB, dC, 1.5, 0.0)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    rows = np.array([0, 1, 43689, 43690, 43691, 49150, 49151], np.int64)
    A = _host_pattern(np.arange(M), K, 7, 3)
    B = _host_pattern(np.arange(K), N, 5, 11)
    ref, _ = oracle.sgemm_rows(A, B, None, 1.5, 0.0, rows)
    got = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(got, ref), f"{path}: sampled rows differ from the oracle"
    cols = np.array([0, 12345, 49151], np.int64)
    refc, _ = oracle.sgemm_cols(A, B, None, 1.5, 0.0, cols)
    gotc = dC[:, torch.from_numpy(cols).cuda()].cpu().numpy()
    assert np.array_equal(gotc, refc), f"{path}: sampled columns differ from the oracle"
    del dC


def test_a_past_2_to_the_31_elements(cuda_device):
    """A of 4096 x 589824 (2.42e9 elements, 9.7 GB) and its transposed copy in the
    workspace: sampled rows bit-exact, including one past element 2^31 of A
    (row 3641) and the last row."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    M, N, K = 4096, 128, 589824
    assert M * K > 2 ** 31
    dA = _device_pattern(M, K, 7, 3, 256)
    dB = _device_pattern(K, N, 5, 11, 65536)
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    # alpha 1: sums reach 16 * K = 9.4e6 < 2^24, exact; 1.5 times that would not be
    binding.sgemm_into(dA, dB, dC, 1.0, 0.0)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    del dA
    rows = np.array([0, 3640, 3641, 4095], np.int64)
    A_rows = _host_pattern(rows, K, 7, 3)
    B = _host_pattern(np.arange(K), N, 5, 11)
    ref, _ = oracle.sgemm(A_rows, B, None, 1.0, 0.0)
    got = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(got, ref), "sampled rows differ from the oracle"


@pytest.mark.parametrize("kind", ["tall", "batched"])
def test_batched_output_past_2_to_the_31_elements(cuda_device, kind):
    """12 batches of 4096 x 49152 (C 2.42e9 elements, 9.7 GB in all; element
    2^31 lies in row 2730 of batch 10, and batch 11 starts past it).  Without an
    activation the batch runs as one tall GEMM of 49152 rows; with ReLU it runs
    the batched kernel.  Sampled rows (row 2730 among them) of the first, the
    tenth and the last batch, bit-exact."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    batch, M, N, K = 12, 4096, 49152, 64
    assert batch * M * N > 2 ** 31
    dA = torch.stack([_device_pattern(M, K, 7 + b, 3, M) for b in range(batch)])
    dB = torch.stack([_device_pattern(K, N, 5, 11 + b, K) for b in range(batch)])
    dC = torch.full((batch, M, N), float("nan"), dtype=torch.float32, device="cuda")
    act = "none" if kind == "tall" else "relu"
    binding.sgemm_ex_into(dA, dB, dC, 1.5, 0.0, act=act)
    torch.cuda.synchronize()
    assert binding.device_status() == binding.SGEMM_OK
    assert ("tall_batch" in binding.last_kernel()) == (kind == "tall")
    rows = np.array([0, 1, 2730, 4095], np.int64)
    for b in (0, 10, batch - 1):
        A = _host_pattern(np.arange(M), K, 7 + b, 3)
        B = _host_pattern(np.arange(K), N, 5, 11 + b)
        ref, _ = oracle.sgemm_ex_rows(A, B, None, 1.5, 0.0, None, act, rows)
        got = dC[b][torch.from_numpy(rows).cuda()].cpu().numpy()
        assert np.array_equal(got, ref), f"{kind}: batch {b} sampled rows differ from the oracle"
    del dC
