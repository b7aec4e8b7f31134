"""The seeded input generators (CPU only): distributions and ranges, NaN padding
beyond a row, determinism per seed, the batch and bias recipes and the oracle's
sampled rows and columns.  They feed both the oracle and the GPU path, so a
mistake here would hide in both."""
import numpy as np
import pytest

from dense_fp32_gemm_02_gb300.workloads import (WORKLOADS, Workload, make_inputs, sample_indices,
                                                workload_bias, workload_inputs)


@pytest.mark.parametrize("dist,lo,hi", [("u01", 0.0, 1.0), ("upm1", -1.0, 1.0), ("int4", -4, 4)])
def test_distributions_stay_in_their_ranges(dist, lo, hi):
    A, B, _ = make_inputs(64, 48, 32, dist, dist, None, seed=5)
    for x in (A, B):
        assert x.dtype == np.float32
        assert x.min() >= lo and x.max() <= hi
    if dist == "int4":
        assert np.array_equal(A, np.round(A)) and set(np.unique(A)) <= set(range(-4, 5))
    else:
        assert A.max() < hi and B.max() < hi   # U[0,1) never reaches 1


def test_padding_beyond_a_row_is_nan_and_views_keep_the_pitch():
    A, B, C = make_inputs(7, 5, 3, "upm1", "normal", "normal", seed=1, lda=8, ldb=9, ldc=6)
    for x, width, ld in ((A, 3, 8), (B, 5, 9), (C, 5, 6)):
        assert x.shape[1] == width and x.strides == (ld * 4, 4)
        base = np.lib.stride_tricks.as_strided(x, shape=(x.shape[0], ld), strides=(ld * 4, 4))
        assert np.isnan(base[:, width:]).all() and np.isfinite(x).all()


def test_same_seed_same_inputs_other_seed_other_inputs():
    a1 = make_inputs(40, 30, 20, "upm1", "upm1", "normal", seed=9)
    a2 = make_inputs(40, 30, 20, "upm1", "upm1", "normal", seed=9)
    a3 = make_inputs(40, 30, 20, "upm1", "upm1", "normal", seed=10)
    for x, y, z in zip(a1, a2, a3):
        assert np.array_equal(x, y) and not np.array_equal(x, z)


def test_batched_workload_draws_each_batch_from_its_own_seed():
    w = Workload("tiny_batched", M=3, N=4, K=5, alpha=1.0, beta=0.0, dist_a="upm1",
                 dist_b="upm1", dist_c=None, seed=77, batch=3)
    A, B, C = workload_inputs(w)
    assert A.shape == (3, 3, 5) and B.shape == (3, 5, 4) and C is None
    for b in range(3):
        a, bb, _ = make_inputs(3, 4, 5, "upm1", "upm1", None, seed=77 + 7919 * b)
        assert np.array_equal(A[b], a) and np.array_equal(B[b], bb)


def test_bias_recipe():
    w = WORKLOADS["sgemm_8192_bias_gelu"]
    bias = workload_bias(w)
    assert bias.shape == (w.batch, w.N) and bias.dtype == np.float32
    assert np.array_equal(bias, np.random.default_rng(w.seed + 17).standard_normal(
        (w.batch, w.N), dtype=np.float32))
    assert workload_bias(WORKLOADS["sgemm_8192_ab"]) is None


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_sampled_rows_and_columns_are_sorted_unique_and_in_range(name):
    w = WORKLOADS[name]
    rows, cols = sample_indices(w)
    if w.check == "full":
        assert rows is None and cols is None
        return
    for idx, n in ((rows, w.M), (cols, w.N)):
        if idx is None:
            continue
        assert idx.dtype == np.int64 and np.all(np.diff(idx) > 0)
        assert idx.min() >= 0 and idx.max() < n
    assert sample_indices(w)[0] is None or np.array_equal(sample_indices(w)[0], rows)
