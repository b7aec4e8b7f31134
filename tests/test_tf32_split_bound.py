"""The error of the 3xTF32 split, in exact arithmetic on the CPU.

Every fp32 x is written x = hi + lo with hi = tf32(x) rounded to nearest (ties
away from zero) and lo = tf32(x - hi); a product a*b is taken as
hi_a*hi_b + hi_a*lo_b + lo_a*hi_b.  The terms below are exact in float64 (tf32
values carry 11 significant bits), so the error measured here is the split's own
and the bound is checked directly:
  * hi rounded to nearest: |error| <= 3 * 2^-22 * |a||b| (slightly more: the
    second-order terms), inside the FP32 tolerance 1e-6 * K * |alpha| * sum|A||B|
    for every K >= 1;
  * hi truncated (what the tensor core makes of a raw fp32 operand): up to
    2^-19 * |a||b|, which is why the library rounds hi itself.
No GPU and no library code is involved; the split is restated from its
definition with integer operations on the float bits."""
import numpy as np
import pytest


def tf32_rna(x):
    """Round fp32 to tf32 (10 stored mantissa bits), ties away from zero."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x1000) & ~np.uint64(0x1FFF)
    return u.astype(np.uint32).view(np.float32)


def tf32_trunc(x):
    u = np.asarray(x, np.float32).view(np.uint32)
    return (u & np.uint32(~0x1FFF & 0xFFFFFFFF)).view(np.float32)


def three_term_product(a, b, hi_fn):
    ha, hb = hi_fn(a), hi_fn(b)
    la = tf32_rna((a.astype(np.float64) - ha).astype(np.float32))
    lb = tf32_rna((b.astype(np.float64) - hb).astype(np.float32))
    h = [t.astype(np.float64) for t in (ha, hb, la, lb)]
    return h[0] * h[1] + h[0] * h[3] + h[2] * h[1]


def _operands(seed, n=200_000):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(n).astype(np.float32)
    b = rng.standard_normal(n).astype(np.float32)
    # spread the exponents (no denormal products)
    a *= np.exp2(rng.integers(-20, 21, n)).astype(np.float32)
    b *= np.exp2(rng.integers(-20, 21, n)).astype(np.float32)
    return a, b


def test_tf32_rounding_restated_from_the_bits():
    one = np.float32(1.0)
    cases = {0x3F801400: 0x3F802000,    # above the midpoint: up
             0x3F801000: 0x3F802000,    # midpoint: away from zero
             0x3F800FFF: 0x3F800000,    # below it: down
             0xBF801000: 0xBF802000,    # negative midpoint: away from zero
             0x3F803000: 0x3F804000}    # midpoint with an odd kept bit: away from zero
    for x, want in cases.items():
        got = tf32_rna(np.array([x], np.uint32).view(np.float32)).view(np.uint32)[0]
        assert got == want, hex(x)
    assert tf32_rna(np.array([one]))[0] == one
    assert tf32_trunc(np.array([0x3F801FFF], np.uint32).view(np.float32)).view(np.uint32)[0] \
        == 0x3F800000


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_rounded_split_error_within_three_times_two_to_the_minus_22(seed):
    a, b = _operands(seed)
    exact = a.astype(np.float64) * b.astype(np.float64)      # exact: 24 x 24 bits
    err = np.abs(three_term_product(a, b, tf32_rna) - exact) / np.abs(exact)
    assert err.max() <= 3.01 * 2.0 ** -22
    assert err.max() > 2.0 ** -23      # the bound is nearly reached, not vacuous
    assert err.max() < 1e-6            # inside the per-product share of the FP32 tolerance


@pytest.mark.parametrize("seed", [4, 5])
def test_truncated_hi_error_reaches_past_the_tolerance_for_short_k(seed):
    a, b = _operands(seed)
    exact = a.astype(np.float64) * b.astype(np.float64)
    err = np.abs(three_term_product(a, b, tf32_trunc) - exact) / np.abs(exact)
    assert err.max() <= 2.0 ** -19
    assert err.max() > 1e-6            # above the tolerance's share at K = 1
