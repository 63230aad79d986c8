"""Pins of the oracle's general form C = alpha op(A) op(B) + beta C.

The scaled, strided and transposed interface is the cuBLAS call on
"LeetGPU problem 2: matrix multiplication" (yekq.top, section "cuBLAS
reference"), restated for row-major storage; its meaning is fixed by
ordinary linear algebra, so these checks hold the oracle to it without
reusing its formula:
  * with alpha = 1, beta = 0 and unit storage it is the plain product, which
    test_oracle_pins.py pins on its own (bitwise);
  * a transposed operand stored transposed gives the same product as the
    plain one on the untransposed matrix (bitwise: same k order);
  * padding beyond the leading dimension's window is never read, and C
    outside its window is never written;
  * power-of-two alpha and beta scale exactly; beta = 0 never reads C;
  * small integers give the exact integer result (Python int arithmetic);
  * random floats lie within half an ulp (plus the double-sum bound) of the
    exact rational alpha * sum + beta * c.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests._exact import exact_dot, round_f32


def _rand(rng, shape):
    return (rng.random(shape, dtype=np.float32) * 2 - 1).astype(np.float32)


def test_unit_form_is_the_plain_product():
    rng = np.random.default_rng(1)
    A, B = _rand(rng, (13, 7)), _rand(rng, (7, 11))
    C0 = np.full((13, 11), np.nan, np.float32)   # beta = 0: never read
    C, absC = oracle.gemm_general(A, B, C0, 13, 11, 7)
    Cp, absp = oracle.gemm(A, B)
    assert np.array_equal(C.view(np.uint32), Cp.view(np.uint32))
    assert np.array_equal(absC, absp)


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
def test_transposed_storage_gives_the_same_product(ta, tb):
    rng = np.random.default_rng(2 + 2 * ta + tb)
    M, K, N = 9, 14, 6
    A, B = _rand(rng, (M, K)), _rand(rng, (K, N))
    As = np.ascontiguousarray(A.T) if ta else A
    Bs = np.ascontiguousarray(B.T) if tb else B
    C, _ = oracle.gemm_general(As, Bs, np.zeros((M, N), np.float32), M, N, K, trans_a=ta, trans_b=tb)
    Cp, _ = oracle.gemm(A, B)
    assert np.array_equal(C.view(np.uint32), Cp.view(np.uint32))


def test_padding_is_never_read_and_outside_of_c_never_written():
    rng = np.random.default_rng(5)
    M, K, N = 5, 6, 7
    A, B = _rand(rng, (M, K)), _rand(rng, (K, N))
    As = np.full((M, K + 3), np.nan, np.float32)
    As[:, :K] = A
    Bs = np.full((K + 2, N + 5), np.nan, np.float32)   # extra rows too: never reached
    Bs[:K, :N] = B
    Cs = np.full((M + 1, N + 4), -7.0, np.float32)
    C, _ = oracle.gemm_general(As, Bs, Cs, M, N, K)
    Cp, _ = oracle.gemm(A, B)
    assert np.array_equal(C[:M, :N], Cp)
    assert np.all(C[:M, N:] == -7.0) and np.all(C[M:, :] == -7.0)


@pytest.mark.parametrize("alpha,beta", [(2.0, 0.0), (-0.5, 0.0), (0.25, 4.0), (1.0, -1.0)])
def test_power_of_two_scalings_are_exact(alpha, beta):
    # the product of a float by a power of two is exact, so alpha * sum rounds
    # like sum; with A = 0 the result is beta * C_old exactly
    rng = np.random.default_rng(7)
    M, K, N = 8, 5, 9
    A, B, C0 = _rand(rng, (M, K)), _rand(rng, (K, N)), _rand(rng, (M, N))
    C, _ = oracle.gemm_general(A, B, np.zeros((M, N), np.float32), M, N, K, alpha=alpha)
    Cp, _ = oracle.gemm(A, B)
    assert np.array_equal(C, (Cp * np.float32(alpha)).astype(np.float32))
    Cz, _ = oracle.gemm_general(np.zeros((M, K), np.float32), B, C0, M, N, K, alpha=alpha, beta=beta)
    assert np.array_equal(Cz, (C0 * np.float32(beta)).astype(np.float32) + np.float32(0))


def test_small_integers_are_exact():
    rng = np.random.default_rng(11)
    M, K, N = 6, 9, 5
    A = rng.integers(-8, 9, (K, M)).astype(np.float32)      # stored transposed
    B = rng.integers(-8, 9, (N, K)).astype(np.float32)      # stored transposed
    C0 = rng.integers(-100, 101, (M, N)).astype(np.float32)
    alpha, beta = 3.0, -2.0
    C, _ = oracle.gemm_general(A, B, C0, M, N, K, alpha=alpha, beta=beta, trans_a=True, trans_b=True)
    Ai, Bi, Ci = A.astype(np.int64), B.astype(np.int64), C0.astype(np.int64)
    want = 3 * (Ai.T @ Bi.T) - 2 * Ci
    assert np.array_equal(C.astype(np.int64), want)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_floats_within_the_exact_bound(seed):
    rng = np.random.default_rng(100 + seed)
    M, K, N = 4, 17, 3
    A, B, C0 = _rand(rng, (M, K)), _rand(rng, (K, N)), _rand(rng, (M, N))
    alpha, beta = np.float32(rng.random() * 3 - 1.5), np.float32(rng.random() * 3 - 1.5)
    C, _ = oracle.gemm_general(A, B, C0, M, N, K, alpha=float(alpha), beta=float(beta))
    for i in range(M):
        for j in range(N):
            s = exact_dot(A[i, :], B[:, j])
            q = Fraction(float(alpha)) * s + Fraction(float(beta)) * Fraction(float(C0[i, j]))
            want = round_f32(q)
            # the double evaluation rounds the K-term sum, alpha * sum and the
            # final add, each within 2^-53 relative of the magnitudes involved;
            # the float result is the rounding of that, so it is the correctly
            # rounded value unless q sits that close to a rounding boundary
            if C[i, j] != want:
                r_abs = abs(Fraction(float(alpha))) * exact_dot(np.abs(A[i, :]), np.abs(B[:, j])) \
                    + abs(Fraction(float(beta)) * Fraction(float(C0[i, j])))
                slack = abs(q) * Fraction(1, 1 << 24) + (K + 3) * r_abs * Fraction(1, 1 << 52)
                assert abs(Fraction(float(C[i, j])) - q) <= slack


def test_planted_transpose_mistake_fails():
    # a wrongly indexed transpose (reading A as if untransposed) breaks the
    # transposed-storage pin: the check above is not vacuous
    rng = np.random.default_rng(13)
    M = K = N = 6
    A, B = _rand(rng, (M, K)), _rand(rng, (K, N))
    C_bad, _ = oracle.gemm_general(A, B, np.zeros((M, N), np.float32), M, N, K, trans_a=True)
    Cp, _ = oracle.gemm(A, B)
    assert not np.array_equal(C_bad, Cp)


def test_bad_arguments_are_refused():
    A = np.zeros((4, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.gemm_general(A, A, A, 5, 4, 4)          # window larger than C
    with pytest.raises(ValueError):
        oracle.gemm_general(A[:, :3], A, A, 4, 4, 4)    # lda < K
