"""Seeded synthetic inputs for the FP32 GEMM workloads.

This module only draws numbers: it holds none of the GEMM arithmetic, imports
neither the CUDA binding nor the CPU oracle, and is the one piece both sides
share.  Every array is numpy float32, row-major, produced by numpy's PCG64
generator from a fixed seed, so the oracle and the CUDA path see the same bits.

Workloads (shapes, distributions, alpha/beta and seeds) follow the five
measured cases of the FP32 SGEMM study: a 256^3 case with the all-ones x
all-twos sanity check of the exercise page ("3.3 Shared memory and tiling -
exercises", skeleton: every element of C equals 2N), the 4096^3 square shape
the pages benchmark, an 8192^3 case with alpha/beta, a ragged case whose sizes
are not tile multiples, and a short-K 16384x16384x512 case.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dist_a: str
    dist_b: str
    dist_c: str | None          # None: C_in unused (beta == 0)
    seed: int
    lda: int = 0                # 0: compact (= K)
    ldb: int = 0                # 0: compact (= N)
    ldc: int = 0                # 0: compact (= N)
    check: str = "full"         # full | rows:<n> | rows:<n>+cols:<n>
    note: str = ""
    extra: dict = field(default_factory=dict)
    batch: int = 1              # independent GEMMs of this shape (sgemm_ex)
    bias: bool = False          # a per-column bias vector per batch (sgemm_ex)
    act: str = "none"           # none | relu | gelu (sgemm_ex)
    bound: str = "alu"          # the roofline of its main kernel: alu (FFMA) or hbm

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K * self.batch

    @property
    def extended(self) -> bool:
        """True when the workload needs sgemm_ex (batches, bias or activation)."""
        return self.batch > 1 or self.bias or self.act != "none"

    def lds(self):
        return (self.lda or self.K, self.ldb or self.N, self.ldc or self.N)


WORKLOADS = {
    "sgemm_256": Workload("sgemm_256", 256, 256, 256, 1.0, 0.0, "u01", "u01", None, 1001,
                          note="plus the A=1, B=2 sanity run (every C equals 512)"),
    "sgemm_4096": Workload("sgemm_4096", 4096, 4096, 4096, 1.0, 0.0, "upm1", "upm1", None,
                           1002, check="full",
                           note="the pages' main square benchmark shape"),
    "sgemm_8192_ab": Workload("sgemm_8192_ab", 8192, 8192, 8192, 1.5, 0.5, "upm1", "upm1",
                              "upm1", 1003, check="rows:64+cols:64"),
    "sgemm_ragged_4097x3001x1023": Workload("sgemm_ragged_4097x3001x1023", 4097, 3001, 1023,
                                            1.0, 1.0, "upm1", "upm1", "normal", 1004,
                                            lda=1023, ldb=3001, ldc=3001, check="full"),
    "sgemm_16384x16384x512": Workload("sgemm_16384x16384x512", 16384, 16384, 512, 1.0, 0.0,
                                      "normal", "normal", None, 1005, check="rows:128",
                                      note="short K, epilogue heavy"),
    # the adjacent uses of the same main loop: many independent GEMMs in one
    # call, and the GEMM of a neural-network layer with its bias and activation
    "sgemm_batched_64x1024": Workload("sgemm_batched_64x1024", 1024, 1024, 1024, 1.0, 0.0,
                                      "upm1", "upm1", None, 1006, check="rows:16", batch=64,
                                      note="64 independent 1024^3 GEMMs in one call"),
    "sgemm_8192_bias_gelu": Workload("sgemm_8192_bias_gelu", 8192, 8192, 8192, 1.0, 0.0,
                                     "upm1", "upm1", None, 1007, check="rows:64",
                                     bias=True, act="gelu",
                                     note="layer form: bias per output column, then GELU"),
    # a degenerate shape of the same operation: one column (a matrix-vector
    # product), bound by reading A once from HBM
    "sgemv_16384x1x16384": Workload("sgemv_16384x1x16384", 16384, 1, 16384, 1.0, 0.0, "upm1",
                                    "upm1", None, 1008, check="full", bound="hbm",
                                    note="N = 1: the skinny-N kernel streams A (1.07 GB) once"),
    "sgemv_1x16384x16384": Workload("sgemv_1x16384x16384", 1, 16384, 16384, 1.0, 0.0, "upm1",
                                    "upm1", None, 1009, check="full", bound="hbm",
                                    note="M = 1: the skinny-M kernel streams B (1.07 GB) once"),
}

# The timed workload of the benchmark.
BENCH_WORKLOAD = "sgemm_8192_ab"


def _draw(rng: np.random.Generator, dist: str, shape) -> np.ndarray:
    if dist == "u01":
        return rng.random(shape, dtype=np.float32)
    if dist == "upm1":
        x = rng.random(shape, dtype=np.float32)
        x *= 2.0
        x -= 1.0
        return x
    if dist == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if dist == "ones":
        return np.ones(shape, dtype=np.float32)
    if dist == "twos":
        return np.full(shape, 2.0, dtype=np.float32)
    if dist.startswith("int"):
        # "int4": integers uniform in [-4, 4]
        r = int(dist[3:])
        return rng.integers(-r, r + 1, size=shape).astype(np.float32)
    if dist == "nan":
        return np.full(shape, np.nan, dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def _with_ld(rng, dist, rows, cols, ld, pad_value=np.nan):
    """rows x cols logical matrix inside a rows x ld buffer; padding holds pad_value."""
    if ld == cols:
        return _draw(rng, dist, (rows, cols))
    buf = np.full((rows, ld), pad_value, dtype=np.float32)
    buf[:, :cols] = _draw(rng, dist, (rows, cols))
    return buf[:, :cols]


def make_inputs(M, N, K, dist_a="upm1", dist_b="upm1", dist_c=None, seed=0,
                lda=0, ldb=0, ldc=0):
    """(A, B, C_in) as float32 views with the requested leading dimensions.
    C_in is None when dist_c is None.  Padding beyond the logical width is NaN
    so that a read outside the matrix shows up in the result."""
    rng = np.random.default_rng(seed)
    lda, ldb, ldc = lda or K, ldb or N, ldc or N
    A = _with_ld(rng, dist_a, M, K, lda)
    B = _with_ld(rng, dist_b, K, N, ldb)
    C = _with_ld(rng, dist_c, M, N, ldc) if dist_c is not None else None
    return A, B, C


def workload_inputs(w: Workload):
    """(A, B, C_in) of a workload; for batch > 1, arrays (batch, rows, cols) with
    batch b drawn from seed + 7919 * b (compact leading dimensions)."""
    lda, ldb, ldc = w.lds()
    if w.batch == 1:
        return make_inputs(w.M, w.N, w.K, w.dist_a, w.dist_b, w.dist_c, w.seed, lda, ldb, ldc)
    parts = [make_inputs(w.M, w.N, w.K, w.dist_a, w.dist_b, w.dist_c, w.seed + 7919 * b)
             for b in range(w.batch)]
    A = np.stack([p[0] for p in parts])
    B = np.stack([p[1] for p in parts])
    C = np.stack([p[2] for p in parts]) if w.dist_c is not None else None
    return A, B, C


def workload_bias(w: Workload):
    """The bias of a workload: float32 (batch, N) drawn N(0, 1) from seed + 17,
    or None."""
    if not w.bias:
        return None
    rng = np.random.default_rng(w.seed + 17)
    return rng.standard_normal((w.batch, w.N), dtype=np.float32)


def sample_indices(w: Workload):
    """(rows, cols) the oracle checks for a workload: None means "all"."""
    rng = np.random.default_rng(w.seed + 1)
    rows = cols = None
    if w.check == "full":
        return None, None
    for part in w.check.split("+"):
        kind, n = part.split(":")
        n = int(n)
        if kind == "rows":
            rows = np.sort(rng.choice(w.M, size=min(n, w.M), replace=False)).astype(np.int64)
        elif kind == "cols":
            cols = np.sort(rng.choice(w.N, size=min(n, w.N), replace=False)).astype(np.int64)
    return rows, cols
