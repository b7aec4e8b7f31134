"""Pins for the oracle's fused epilogue and batched form (no GPU).

The fused GEMM is act(alpha*A@B + beta*C_in + bias) with a per-column bias and
act in {identity, ReLU, GELU}; a batched GEMM is that, once per batch.  The
pins check it against facts the oracle does not produce itself:
  * exact integer arithmetic (numpy int64) on integer-valued inputs, where every
    intermediate is exactly representable, for bias and ReLU;
  * printed values of the standard normal distribution function Phi (GELU is
    z * Phi(z)) and the identity GELU(z) - GELU(-z) = z;
  * numpy's float64 matmul per batch, for the batch loop and strided views;
  * the reduction to the plain GEMM when there is neither bias nor activation.
The last tests plant mistakes in copies of the oracle's C source and check that
a pin catches each one.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_gemm_02_gb300.workloads import make_inputs

# Phi(z) at integer z, as printed in standard normal tables (to 16 digits).
PHI = {0: 0.5, 1: 0.8413447460685429, 2: 0.9772498680518208, 3: 0.9986501019683699}


def pin_ex_plain_reduction(lib=None):
    A, B, C = make_inputs(37, 29, 53, "upm1", "upm1", "normal", seed=71)
    for beta, Cin in ((0.0, None), (0.75, C)):
        plain, pb = oracle.sgemm(A, B, Cin, 1.25, beta)
        ex, eb = oracle.sgemm_ex_rows(A, B, Cin, 1.25, beta, None, "none", lib=lib)
        assert np.array_equal(plain, ex)
        assert np.allclose(pb, eb, rtol=1e-12, atol=0)


def pin_ex_integer_bias_relu(lib=None):
    # integers in [-4, 4]: |sum| <= 16K, so every partial sum is exact; with
    # alpha = 1.5, beta = 0.5 and integer C and bias the result is a multiple of
    # 1/2 below 2^22 and therefore exact in float32.
    M, N, K = 23, 31, 40          # M != N: a bias applied per row would show
    A, B, C = make_inputs(M, N, K, "int4", "int4", "int4", seed=72)
    bias = np.random.default_rng(73).integers(-50, 51, size=N).astype(np.float32)
    z2 = (3 * (A.astype(np.int64) @ B.astype(np.int64)) + C.astype(np.int64)
          + 2 * bias.astype(np.int64)[None, :])           # 2 * Z, exact
    for act, ref2 in (("none", z2), ("relu", np.maximum(z2, 0))):
        out, bound = oracle.sgemm_ex_rows(A, B, C, 1.5, 0.5, bias, act, lib=lib)
        assert np.array_equal(out, (ref2 / 2).astype(np.float32)), act
        assert np.all(bound >= 1e-6 * np.abs(bias)[None, :])


def pin_ex_gelu_table(lib=None):
    # K = 1, B = [[1]]: Z = A[i][0] exactly, so the output is GELU(z) = z * Phi(z)
    zs = np.array([0, 1, 2, 3, -1, -2, -3], np.float32)
    out, bound = oracle.sgemm_ex_rows(zs[:, None].copy(), np.ones((1, 1), np.float32), None,
                                      1.0, 0.0, None, "gelu", lib=lib)
    for z, got in zip(zs, out[:, 0]):
        phi = PHI[abs(int(z))] if z >= 0 else 1.0 - PHI[abs(int(z))]
        want = np.float32(float(z) * phi)
        assert abs(float(got) - float(want)) <= 1e-7 * max(1.0, abs(float(want))), (z, got, want)
    # odd part: GELU(z) - GELU(-z) = z
    zr = np.random.default_rng(74).uniform(-6, 6, 64).astype(np.float32)
    pos, _ = oracle.sgemm_ex_rows(zr[:, None].copy(), np.ones((1, 1), np.float32), None, 1.0,
                                  0.0, None, "gelu", lib=lib)
    neg, _ = oracle.sgemm_ex_rows((-zr)[:, None].copy(), np.ones((1, 1), np.float32), None,
                                  1.0, 0.0, None, "gelu", lib=lib)
    assert np.allclose(pos[:, 0] - neg[:, 0], zr, rtol=0, atol=2e-6)
    # bound: Sum|a||b| = |z|, so 1.129 * 1e-6|z| + 1e-6|z|
    assert np.allclose(bound[:, 0], 2.129e-6 * np.abs(zs.astype(np.float64)), rtol=1e-9, atol=0)


def pin_ex_batched_vs_numpy(lib=None):
    batch, M, N, K = 3, 19, 27, 33
    rng = np.random.default_rng(75)
    store_a = rng.uniform(-1, 1, (batch, M, K + 5)).astype(np.float32)   # padded rows
    store_b = rng.uniform(-1, 1, (batch, K, N)).astype(np.float32)
    Cs = rng.standard_normal((batch, M, N)).astype(np.float32)
    biases = rng.standard_normal((batch, N)).astype(np.float32)
    As = [store_a[b, :, :K] for b in range(batch)]
    out, bound = oracle.sgemm_batched(As, list(store_b), list(Cs), 0.5, -1.0, list(biases),
                                      "relu", lib=lib)
    for b in range(batch):
        z = (0.5 * (store_a[b, :, :K].astype(np.float64) @ store_b[b].astype(np.float64))
             - Cs[b].astype(np.float64) + biases[b].astype(np.float64)[None, :])
        ref = np.maximum(z, 0).astype(np.float32)
        assert np.allclose(out[b], ref, rtol=1e-6, atol=1e-6), b
        assert np.all(np.abs(out[b].astype(np.float64) - np.maximum(z, 0)) <= bound[b] + 1e-30)


PINS = [pin_ex_plain_reduction, pin_ex_integer_bias_relu, pin_ex_gelu_table,
        pin_ex_batched_vs_numpy]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_ex_pin(pin):
    pin()


def test_ex_rejects_bad_arguments():
    A, B, _ = make_inputs(4, 5, 6, seed=76)
    with pytest.raises(KeyError):
        oracle.sgemm_ex_rows(A, B, None, 1.0, 0.0, None, "tanh")
    with pytest.raises(TypeError):
        oracle.sgemm_ex_rows(A, B, None, 1.0, 0.0, np.zeros(4, np.float32), "none")
    with pytest.raises(ValueError):
        oracle.sgemm_batched([A, A], [B], None, 1.0, 0.0)


# ----------------------------------------------------------------- planted mistakes
MUTANTS = {
    "bias_per_row": ("z += (double)bias[j];", "z += (double)bias[i % N];"),
    "bias_scaled_by_alpha": ("z += (double)bias[j];", "z += (double)alpha * (double)bias[j];"),
    "relu_is_abs": ("return z > 0.0 ? z : 0.0;", "return fabs(z);"),
    "gelu_without_half": ("return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
                          "return z * (1.0 + erf(z / sqrt(2.0)));"),
    "gelu_wrong_scale": ("return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
                         "return 0.5 * z * (1.0 + erf(z / 2.0));"),
    "beta_dropped": ("z += cterm;", "z += 0.0 * cterm;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_ex_pins_catch_planted_mistake(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    msrc = tmp_path / f"mutant_{name}.c"
    msrc.write_text(src.replace(old, new, 1))
    lib = oracle.load_library(oracle.compile_source(str(msrc), str(tmp_path / f"{name}.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
