"""Seeded synthetic inputs and counting conventions for the FP32 GEMM.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the product's arithmetic: only random draws (numpy PCG64,
one fresh generator per problem; A is drawn before B), the problem shapes,
and the FLOP / byte counts used to turn times into throughput.

Problem shapes (M, K, N), value laws and seeds:
  c1      100 x 37 x 70      uniform[-1, 1)          seed 0
  c1int   100 x 37 x 70      integers in [-8, 8]     seed 0  (bit-exact case)
  c2      1024 x 512 x 1024  uniform[-1, 1)          seed 1  (the regular size
          timed on "LeetGPU problem 2", section "benchmark summary")
  c3      1001 x 513 x 777   uniform[-1, 1)          seed 2  (the ragged size
          timed on the same page)
  c4      4096^3             standard normal         seed 3
  c5a     8192^3             standard normal         seed 4
  c5b     65536 x 1024 x 64  standard normal         seed 4  (tall-skinny)
  c5c     64 x 4096 x 65536  standard normal         seed 4  (short-wide)
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Problem:
    name: str
    M: int
    K: int
    N: int
    law: str        # "uniform", "normal" or "int8"
    seed: int
    note: str = ""


CONFIGS = {
    "c1": Problem("c1", 100, 37, 70, "uniform", 0, "tiny ragged, misaligned strides"),
    "c1int": Problem("c1int", 100, 37, 70, "int8", 0, "integers in [-8, 8]: exact in fp32"),
    "c2": Problem("c2", 1024, 512, 1024, "uniform", 1, "regular, tile aligned"),
    "c3": Problem("c3", 1001, 513, 777, "uniform", 2, "ragged on every edge"),
    "c4": Problem("c4", 4096, 4096, 4096, "normal", 3, "compute-bound square"),
    "c5a": Problem("c5a", 8192, 8192, 8192, "normal", 4, "large compute-bound square"),
    "c5b": Problem("c5b", 65536, 1024, 64, "normal", 4, "tall-skinny, bandwidth bound"),
    "c5c": Problem("c5c", 64, 4096, 65536, "normal", 4, "short-wide, bandwidth bound"),
}


def draw(rng: np.random.Generator, shape, law: str) -> np.ndarray:
    """One float32 array of the given law from ``rng``."""
    if law == "uniform":
        return rng.random(shape, dtype=np.float32) * np.float32(2) - np.float32(1)
    if law == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if law == "int8":
        return rng.integers(-8, 9, size=shape, dtype=np.int8).astype(np.float32)
    raise ValueError("unknown law %r" % law)


def make_inputs(M: int, K: int, N: int, law: str, seed: int):
    """(A [M,K], B [K,N]) float32, C-contiguous, A drawn first."""
    rng = np.random.default_rng(seed)
    A = draw(rng, (M, K), law)
    B = draw(rng, (K, N), law)
    return A, B


def problem_inputs(name: str):
    p = CONFIGS[name]
    return make_inputs(p.M, p.K, p.N, p.law, p.seed)


def gemm_flops(M: int, N: int, K: int) -> int:
    """FP32 work of one product: one multiply and one add per (i, j, k)."""
    return 2 * M * N * K


def algorithmic_bytes(M: int, N: int, K: int, elem: int = 4) -> int:
    """Least HBM traffic: each operand read once, C written once."""
    return elem * (M * K + K * N + M * N)


def naive_read_bytes(M: int, N: int, K: int, elem: int = 4) -> int:
    """Reads of a kernel that fetches a row of A and a column of B per output."""
    return elem * M * N * 2 * K


def tiled_read_bytes(M: int, N: int, K: int, T: int, elem: int = 4) -> int:
    """Reads of a T x T shared-memory tiled kernel: one A tile and one B tile
    per output tile and per K phase (sizes that are multiples of T)."""
    tiles = (M // T) * (N // T)
    phases = K // T
    return elem * tiles * phases * 2 * T * T
