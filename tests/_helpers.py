"""Shared helpers of the GPU parity tests: move numpy inputs (with their row
pitch and NaN padding) to the device, run the library, compare with the oracle."""
import numpy as np


def storage_of(x: np.ndarray) -> np.ndarray:
    """The rows x ld buffer behind a row-major view x (padding included)."""
    ld = x.strides[0] // 4 if x.shape[0] > 1 else x.shape[1]
    ld = max(ld, x.shape[1], 1)
    if ld == x.shape[1] or x.shape[0] == 0:
        return np.ascontiguousarray(x)
    return np.lib.stride_tricks.as_strided(x, shape=(x.shape[0], ld), strides=(ld * 4, 4))


def to_device(x: np.ndarray, device="cuda", offset_elems: int = 0):
    """CUDA float32 view with the same shape and row pitch as x.  offset_elems
    shifts the first element inside a larger allocation (to test addresses that
    are 4-byte but not 16-byte aligned)."""
    import torch
    if x is None:
        return None
    st = storage_of(x)
    rows, ld = st.shape
    flat = torch.full((rows * ld + offset_elems + 4,), float("nan"), dtype=torch.float32,
                      device=device)
    flat[offset_elems:offset_elems + rows * ld] = torch.from_numpy(
        np.ascontiguousarray(st).reshape(-1)).to(device)
    return flat[offset_elems:offset_elems + rows * ld].view(rows, ld)[:, :x.shape[1]]


def run_gpu(A, B, C, alpha, beta, offsets=(0, 0, 0)):
    """alpha*A@B + beta*C through the C ABI; returns the device C view."""
    import torch
    from dense_fp32_gemm_02_gb300 import binding
    dA = to_device(A, offset_elems=offsets[0])
    dB = to_device(B, offset_elems=offsets[1])
    M, N = A.shape[0], B.shape[1]
    if C is None:
        C = np.full((M, N), np.nan, dtype=np.float32)
    dC = to_device(C, offset_elems=offsets[2])
    binding.sgemm_into(dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    return dC


def assert_within_bound(got: np.ndarray, ref: np.ndarray, bound: np.ndarray, what=""):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    both_nan = np.isnan(got) & np.isnan(ref)
    err = np.abs(got - ref)
    ok = (err <= bound) | both_nan
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        detail = ", ".join(f"{tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} "
                           f"bound {bound[tuple(i)]:.3e}" for i in idx)
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside the bound; {detail}")
    # report the worst ratio for the log
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, 0.0)
    return float(np.nanmax(ratio)) if ratio.size else 0.0
