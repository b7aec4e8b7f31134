"""Pins for the CPU oracle (no GPU).

The oracle is checked against facts that do not come from the oracle itself:
  * the closed form printed by the exercise page "3.3 Shared memory and tiling -
    exercises" (all-ones A times all-twos B gives 2K everywhere), read from
    tests/golden/ones_twos.txt;
  * brute force in exact rational arithmetic (Python ``fractions``) on tiny
    shapes whose exact results are representable in float32;
  * numpy's float64 matmul (a library routine) for the alpha/beta formula;
  * invariants of the definition: (A B)^T = B^T A^T, alpha scaling, the
    alpha/beta identities, leading-dimension padding that must never be read;
  * closed forms with K up to 8192 that tell rows from columns.
The last test plants mistakes in copies of the oracle's C source and checks
that at least one pin catches each one.
"""
import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ones_twos.txt")


def _golden_rows():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                M, N, K, v = line.split()
                out.append((int(M), int(N), int(K), float(v)))
    return out


# --------------------------------------------------------------------------- pins
# Each pin takes an optional ``lib`` (an oracle build) so the mutation test can
# run the same checks against planted-mistake builds.  A pin raises
# AssertionError when the oracle disagrees with the fact it encodes.

def pin_ones_twos(lib=None):
    for M, N, K, expected in _golden_rows():
        assert expected == 2 * K
        A = np.ones((M, K), np.float32)
        B = np.full((K, N), 2.0, np.float32)
        rows = np.array(sorted({0, M // 3, M - 1}), np.int64)
        out, bound = oracle.sgemm_rows(A, B, None, 1.0, 0.0, rows, lib=lib)
        assert np.all(out == np.float32(expected)), (M, N, K)
        # Sum_k |1|*|2| = 2K, so the bound is 1e-6 * K * 2K.
        assert np.allclose(bound, 1e-6 * K * 2 * K, rtol=1e-12, atol=0)
    # non-square, non-tile sizes
    for (M, N, K) in [(7, 13, 29), (1, 5, 1), (33, 2, 17)]:
        out, _ = oracle.sgemm(np.ones((M, K), np.float32), np.full((K, N), 2.0, np.float32),
                              None, 1.0, 0.0, lib=lib)
        assert out.shape == (M, N) and np.all(out == 2 * K)


def _exact(A, B, C, alpha, beta):
    """Exact rational alpha*A@B + beta*C and the exact tolerance bound."""
    M, K = A.shape
    N = B.shape[1]
    al, be = Fraction(float(alpha)), Fraction(float(beta))
    res = np.empty((M, N), np.float64)
    bnd = np.empty((M, N), np.float64)
    for i in range(M):
        for j in range(N):
            s = sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)),
                    Fraction(0))
            sa = sum((abs(Fraction(float(A[i, k])) * Fraction(float(B[k, j])))
                      for k in range(K)), Fraction(0))
            c = Fraction(float(C[i, j])) if (C is not None and be != 0) else Fraction(0)
            res[i, j] = float(al * s + be * c)
            bnd[i, j] = float(Fraction(1, 10**6) * K * abs(al) * sa
                              + Fraction(1, 10**6) * abs(be * c))
    return res, bnd


TINY_CASES = [
    # (M, N, K, alpha, beta, seed)
    (1, 1, 1, 1.0, 0.0, 1),
    (2, 3, 4, 1.0, 0.0, 2),
    (5, 7, 3, -0.5, 0.25, 3),
    (4, 1, 9, 2.0, -1.0, 4),
    (3, 5, 0, 1.0, 0.5, 5),
    (6, 4, 11, 0.0, 1.0, 6),
    (3, 6, 5, 0.75, 1.0, 7),
]


def pin_bruteforce_exact(lib=None):
    for (M, N, K, alpha, beta, seed) in TINY_CASES:
        rng = np.random.default_rng(seed)
        # quarter-integers in [-2, 2]: every product and sum is exact in float32
        A = (rng.integers(-8, 9, size=(M, K)) / 4).astype(np.float32)
        B = (rng.integers(-8, 9, size=(K, N)) / 4).astype(np.float32)
        C = (rng.integers(-8, 9, size=(M, N)) / 4).astype(np.float32)
        ref, ref_bound = _exact(A, B, C, alpha, beta)
        assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
        out, bound = oracle.sgemm(A, B, C if beta != 0 else None, alpha, beta, lib=lib)
        assert np.array_equal(out.astype(np.float64), ref), (M, N, K, alpha, beta)
        assert np.allclose(bound, ref_bound, rtol=1e-12, atol=1e-300), (M, N, K)


def pin_numpy_float64(lib=None):
    for (M, N, K, alpha, beta, seed) in [(33, 47, 65, 1.5, 0.5, 11), (64, 64, 64, 1.0, 0.0, 12),
                                         (17, 129, 31, -2.0, 3.0, 13)]:
        A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", seed)
        ref = (alpha * (A.astype(np.float64) @ B.astype(np.float64))
               + beta * C.astype(np.float64)).astype(np.float32)
        out, bound = oracle.sgemm(A, B, C, alpha, beta, lib=lib)
        ulp = np.spacing(np.maximum(np.abs(ref), np.abs(out)))
        diff = np.abs(out.astype(np.float64) - ref.astype(np.float64))
        # the two double sums differ only in summation order; after the single
        # rounding to float they agree except on rare rounding-boundary ties
        assert np.all(diff <= ulp), (M, N, K)
        assert np.mean(diff == 0) > 0.99, (M, N, K)
        sabs = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
        exp_bound = 1e-6 * K * abs(alpha) * sabs + 1e-6 * np.abs(beta * C.astype(np.float64))
        assert np.allclose(bound, exp_bound, rtol=1e-9), (M, N, K)


def pin_transpose(lib=None):
    # (A B)^T = B^T A^T: each element is the same products in the same k order.
    A, B, C = make_inputs(19, 23, 37, "normal", "normal", "normal", 21)
    out, bnd = oracle.sgemm(A, B, C, 1.25, -0.5, lib=lib)
    outT, bndT = oracle.sgemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T),
                              np.ascontiguousarray(C.T), 1.25, -0.5, lib=lib)
    assert np.array_equal(out, outT.T)
    assert np.allclose(bnd, bndT.T, rtol=1e-12)


def pin_alpha_beta_identities(lib=None):
    A, B, C = make_inputs(21, 18, 27, "upm1", "upm1", "upm1", 31)
    base, _ = oracle.sgemm(A, B, None, 1.0, 0.0, lib=lib)
    two, _ = oracle.sgemm(A, B, None, 2.0, 0.0, lib=lib)
    neg, _ = oracle.sgemm(A, B, None, -1.0, 0.0, lib=lib)
    assert np.array_equal(two, 2 * base)          # scaling by 2 commutes with rounding
    assert np.array_equal(neg, -base)
    # alpha = 0, beta = 1 leaves C unchanged, even with Inf/NaN in A and B
    An = A.copy(); An[0, 0] = np.inf; An[1, 1] = np.nan
    keep, _ = oracle.sgemm(An, B, C, 0.0, 1.0, lib=lib)
    assert np.array_equal(keep, C)
    # beta = 0: C_in is never read (NaN does not propagate)
    nanC = np.full_like(C, np.nan)
    z, _ = oracle.sgemm(A, B, nanC, 1.0, 0.0, lib=lib)
    assert np.array_equal(z, base)
    # K = 0: the empty sum, so C = beta * C
    A0 = np.zeros((21, 0), np.float32)
    B0 = np.zeros((0, 18), np.float32)
    k0, b0 = oracle.sgemm(A0, B0, C, 3.0, 0.5, lib=lib)
    assert np.array_equal(k0, 0.5 * C)
    assert np.allclose(b0, 1e-6 * np.abs(0.5 * C.astype(np.float64)), rtol=1e-12)
    # beta term on its own: alpha = 0, beta = -3
    b3, bb3 = oracle.sgemm(A, B, C, 0.0, -3.0, lib=lib)
    assert np.array_equal(b3, (-3.0 * C.astype(np.float64)).astype(np.float32))
    assert np.allclose(bb3, 1e-6 * np.abs(3.0 * C.astype(np.float64)), rtol=1e-12)


def pin_leading_dimensions(lib=None):
    # NaN in the padding beyond each row must never reach the result.
    M, N, K = 13, 11, 9
    A, B, C = make_inputs(M, N, K, "upm1", "upm1", "normal", 41, lda=K + 3, ldb=N + 5,
                          ldc=N + 2)
    assert np.isnan(A.base[:, K:]).all() and np.isnan(B.base[:, N:]).all()
    out, bnd = oracle.sgemm(A, B, C, 1.0, 1.0, lib=lib)
    outc, bndc = oracle.sgemm(np.ascontiguousarray(A), np.ascontiguousarray(B),
                              np.ascontiguousarray(C), 1.0, 1.0, lib=lib)
    assert np.isfinite(out).all()
    assert np.array_equal(out, outc) and np.array_equal(bnd, bndc)


def pin_rows_cols_subsets(lib=None):
    A, B, C = make_inputs(40, 36, 25, "normal", "normal", "normal", 51)
    full, fb = oracle.sgemm(A, B, C, 0.5, 2.0, lib=lib)
    rows = np.array([0, 7, 39, 13], np.int64)
    cols = np.array([35, 0, 18], np.int64)
    r, rb = oracle.sgemm_rows(A, B, C, 0.5, 2.0, rows, lib=lib)
    c, cb = oracle.sgemm_cols(A, B, C, 0.5, 2.0, cols, lib=lib)
    assert np.array_equal(r, full[rows]) and np.array_equal(rb, fb[rows])
    assert np.array_equal(c, full[:, cols]) and np.array_equal(cb, fb[:, cols])


def pin_closed_forms_long_k(lib=None):
    # A[i][k] = (i mod 3) + 1, B[k][j] = (j mod 5) - 2: C[i][j] = K ((i mod 3)+1)((j mod 5)-2)
    for (M, N, K) in [(6, 10, 8192), (5, 7, 1023)]:
        A = np.tile(((np.arange(M) % 3) + 1).astype(np.float32)[:, None], (1, K))
        B = np.tile(((np.arange(N) % 5) - 2).astype(np.float32)[None, :], (K, 1))
        out, _ = oracle.sgemm(A, B, None, 1.0, 0.0, lib=lib)
        exp = K * np.outer((np.arange(M) % 3) + 1, (np.arange(N) % 5) - 2)
        assert np.array_equal(out, exp.astype(np.float32))
        c, _ = oracle.sgemm_cols(A, B, None, 1.0, 0.0, np.array([N - 1, 1]), lib=lib)
        assert np.array_equal(c, exp[:, [N - 1, 1]].astype(np.float32))


PINS = [pin_ones_twos, pin_bruteforce_exact, pin_numpy_float64, pin_transpose,
        pin_alpha_beta_identities, pin_leading_dimensions, pin_rows_cols_subsets,
        pin_closed_forms_long_k]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin()


def test_argument_errors():
    A, B, C = make_inputs(4, 4, 4, dist_c="normal", seed=1)
    with pytest.raises(ValueError):
        oracle.sgemm(A, B[:3], None, 1.0, 0.0)
    with pytest.raises(TypeError):
        oracle.sgemm(A.astype(np.float64), B, None, 1.0, 0.0)
    with pytest.raises(ValueError):
        oracle.sgemm(A, B, C[:3], 1.0, 1.0)


# ----------------------------------------------------------------- planted mistakes
MUTANTS = {
    "sign_of_product": ("acc[j] += a * b;", "acc[j] -= a * b;"),
    "dropped_beta_term": ("cterm = beta * (double)(*c_in_elem);", "cterm = 0.0;"),
    "alpha_on_c_term": ("double prod = (alpha == 0.0) ? 0.0 : alpha * sum;",
                        "double prod = sum;"),
    "k_starts_at_one": ("for (long long k = 0; k < K; ++k) {\n                double a = (double)A[i * lda + k];\n                double abs_a = fabs(a);\n                const float *brow = B + k * ldb;",
                        "for (long long k = 1; k < K; ++k) {\n                double a = (double)A[i * lda + k];\n                double abs_a = fabs(a);\n                const float *brow = B + k * ldb;"),
    "reversed_rows_of_A": ("double a = (double)A[i * lda + k];\n                double abs_a = fabs(a);\n                const float *brow = B + k * ldb;",
                           "double a = (double)A[(M - 1 - i) * lda + k];\n                double abs_a = fabs(a);\n                const float *brow = B + k * ldb;"),
    "reversed_cols_of_B": ("bcols[k * ncols + c] = B[k * ldb + cols[c]];",
                           "bcols[k * ncols + c] = B[k * ldb + (N - 1 - cols[c])];"),
    "signed_bound": ("abs_acc[j] += abs_a * fabs(b);", "abs_acc[j] += a * b;"),
    "beta_twice": ("return (float)(prod + cterm);", "return (float)(prod + 2.0 * cterm);"),
}


def _mutant_source(src, old, new):
    assert src.count(old) >= 1, f"mutation anchor not found: {old[:40]!r}"
    return src.replace(old, new, 1)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    msrc = tmp_path / f"mutant_{name}.c"
    msrc.write_text(_mutant_source(src, old, new))
    lib = oracle.load_library(oracle.compile_source(str(msrc), str(tmp_path / f"{name}.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"


def test_pins_catch_single_precision_accumulation(tmp_path):
    # Accumulating in float instead of double is the classic CPU-reference mistake
    # (the exercise page's own host check accumulates in float).
    src = open(oracle._SRC).read()
    msrc = src.replace("acc[j] += a * b;", "acc[j] = (double)(float)(acc[j] + a * b);", 1)
    assert msrc != src
    p = tmp_path / "mutant_float_acc.c"
    p.write_text(msrc)
    lib = oracle.load_library(oracle.compile_source(str(p), str(tmp_path / "fa.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught
