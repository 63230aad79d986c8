"""Seeded synthetic inputs and counting conventions for the FP32 GEMM.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the product's arithmetic: only random draws (numpy PCG64,
one fresh generator per problem; A is drawn before B), the problem shapes,
and the FLOP / byte counts used to turn times into throughput.

Problems, named by their shape M x K x N, with value laws and seeds:
  100x37x70        uniform[-1, 1)          seed 0  (tiny, misaligned strides)
  100x37x70-int    integers in [-8, 8]     seed 0  (bit-exact case)
  1024x512x1024    uniform[-1, 1)          seed 1  (the regular size timed on
                   "LeetGPU problem 2", section "benchmark summary")
  1001x513x777     uniform[-1, 1)          seed 2  (the ragged size timed on
                   the same page)
  4096x4096x4096   standard normal         seed 3
  8192x8192x8192   standard normal         seed 4
  65536x1024x64    standard normal         seed 4  (tall-skinny)
  64x4096x65536    standard normal         seed 4  (short-wide)
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


PROBLEMS = {
    "100x37x70": Problem("100x37x70", 100, 37, 70, "uniform", 0, "tiny ragged, misaligned strides"),
    "100x37x70-int": Problem("100x37x70-int", 100, 37, 70, "int8", 0, "integers in [-8, 8]: exact in fp32"),
    "1024x512x1024": Problem("1024x512x1024", 1024, 512, 1024, "uniform", 1, "regular, tile aligned"),
    "1001x513x777": Problem("1001x513x777", 1001, 513, 777, "uniform", 2, "ragged on every edge"),
    "4096x4096x4096": Problem("4096x4096x4096", 4096, 4096, 4096, "normal", 3, "compute-bound square"),
    "8192x8192x8192": Problem("8192x8192x8192", 8192, 8192, 8192, "normal", 4, "large compute-bound square"),
    "65536x1024x64": Problem("65536x1024x64", 65536, 1024, 64, "normal", 4, "tall-skinny, bandwidth bound"),
    "64x4096x65536": Problem("64x4096x65536", 64, 4096, 65536, "normal", 4, "short-wide, bandwidth bound"),
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
    p = PROBLEMS[name]
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
