"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself or with the CUDA library.
Sources of truth:
  * the pages' printed timings (FLOP convention) and worked traffic example,
    kept as cited text fixtures under tests/golden/;
  * closed forms with exactly representable results (ones, identity, zeros,
    K = 0, K = 1, power-of-two scaling);
  * invariants of the product ((AB)^T = B^T A^T, row/column permutations,
    zero padding of K as in the tile simulator of "Lesson 10");
  * brute force over every small {-1, 0, 1} matrix against Python integers,
    and exact rational arithmetic (tests/_exact.py) with correct rounding;
  * a planted-mistake check: plausible wrong versions of the formula fail
    these same pins.
"""
import os

import numpy as np
import pytest

import oracle
import workloads
from tests._exact import exact_abs_dot, exact_dot, round_f32, ulp_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- counting
def test_flop_convention_matches_printed_tables():
    """GFLOPS * ms on both printed tables equals 2MNK to the ms rounding."""
    rows = _read_golden("p1_benchmark_tables.txt")
    assert len(rows) == 12
    for M, K, N, kernel, ms, gflops, _pct in rows:
        M, K, N, ms, gflops = int(M), int(K), int(N), float(ms), float(gflops)
        t_pred_ms = workloads.gemm_flops(M, N, K) / (gflops * 1e9) * 1e3
        assert abs(t_pred_ms - ms) <= 0.0005 + 1e-9, (kernel, M, K, N, t_pred_ms, ms)
        # a different convention (MNK, or 2MNK counted with M and K swapped
        # in the ragged case) misses the printed ms
        assert abs(M * N * K / (gflops * 1e9) * 1e3 - ms) > 0.0005


def test_traffic_worked_example():
    kv = {k: float(v) for k, v in _read_golden("p3_traffic_example.txt")}
    M, N, K, T = int(kv["M"]), int(kv["N"]), int(kv["K"]), int(kv["T"])
    flop = workloads.gemm_flops(M, N, K)
    assert abs(flop / kv["flop"] - 1) < 1e-3
    naive = workloads.naive_read_bytes(M, N, K)
    assert abs(naive / kv["naive_bytes"] - 1) < 1e-3
    assert abs(flop / naive - kv["naive_intensity"]) < 1e-3
    assert (M // T) * (N // T) == kv["tiles"]
    assert K // T == kv["phases"]
    assert 2 * T * T == kv["floats_per_phase"]
    tiled = workloads.tiled_read_bytes(M, N, K, T)
    assert tiled // 4 == kv["tiles"] * kv["phases"] * kv["floats_per_phase"]
    assert abs(tiled / kv["tiled_bytes"] - 1) < 1e-4
    assert abs(tiled // 4 / kv["tiled_reads"] - 1) < 1e-2
    assert naive // tiled == kv["ratio"]
    assert abs(flop / tiled - kv["tiled_intensity"]) < 1e-3


def test_algorithmic_bytes_closed_form():
    # 1024^3: each operand once (4 MiB each) plus C once
    assert workloads.algorithmic_bytes(1024, 1024, 1024) == 3 * 4 * 1024 * 1024
    assert workloads.algorithmic_bytes(100, 70, 37) == 4 * (100 * 37 + 37 * 70 + 100 * 70)


# ----------------------------------------------------------------- closed forms
def _rand(shape, seed, law="uniform"):
    return workloads.draw(np.random.default_rng(seed), shape, law)


@pytest.mark.parametrize("M,K,N", [(7, 9, 5), (33, 70, 17), (1, 1, 1), (64, 300, 3)])
def test_ones_gives_column_sums(M, K, N):
    # dyadic B with few bits: every partial sum is exact in double and in float
    B = (np.random.default_rng(M * 1000 + K).integers(-64, 65, size=(K, N)) / 16.0).astype(np.float32)
    A = np.ones((M, K), np.float32)
    C, absAB = oracle.gemm(A, B)
    colsum = np.array([sum(int(v) for v in (B[:, j] * 16).astype(np.int64)) / 16.0 for j in range(N)])
    abssum = np.array([sum(abs(int(v)) for v in (B[:, j] * 16).astype(np.int64)) / 16.0 for j in range(N)])
    assert np.array_equal(C, np.broadcast_to(colsum.astype(np.float32), (M, N)))
    assert np.array_equal(absAB, np.broadcast_to(abssum, (M, N)))


@pytest.mark.parametrize("n,m", [(1, 3), (17, 5), (64, 64), (130, 33)])
def test_identity(n, m):
    X = _rand((n, m), n + m, "normal")
    C, _ = oracle.gemm(np.eye(n, dtype=np.float32), X)
    assert np.array_equal(C.view(np.uint32), (X + 0).view(np.uint32))
    Y = _rand((m, n), n * m, "normal")
    C, _ = oracle.gemm(Y, np.eye(n, dtype=np.float32))
    assert np.array_equal(C.view(np.uint32), (Y + 0).view(np.uint32))


def test_zeros_and_empty_k():
    A = _rand((6, 4), 1)
    C, absAB = oracle.gemm(A, np.zeros((4, 9), np.float32))
    assert not C.any() and not absAB.any()
    assert not np.signbit(C).any()           # +0.0, never -0.0
    C, absAB = oracle.gemm(np.zeros((6, 0), np.float32), np.zeros((0, 9), np.float32))
    assert C.shape == (6, 9) and not C.any() and not absAB.any()
    C, _ = oracle.gemm(np.zeros((0, 3), np.float32), np.zeros((3, 5), np.float32))
    assert C.shape == (0, 5)


def test_k1_outer_product_is_correctly_rounded():
    a = _rand((40, 1), 11, "normal")
    b = _rand((1, 30), 12, "normal")
    C, absAB = oracle.gemm(a, b)
    for i in range(0, 40, 3):
        for j in range(0, 30, 4):
            q = exact_dot(a[i, :], b[:, j])
            assert C[i, j] == round_f32(q)
            assert absAB[i, j] == float(abs(q))


@pytest.mark.parametrize("p", [-20, -3, 1, 7, 30])
def test_power_of_two_scaling(p):
    A = _rand((19, 23), 5, "normal")
    B = _rand((23, 11), 6, "normal")
    C, absAB = oracle.gemm(A, B)
    s = np.float32(2.0 ** p)
    C2, absAB2 = oracle.gemm(A * s, B)
    assert np.array_equal(C2, C * s)
    assert np.array_equal(absAB2, absAB * (2.0 ** p))


# ----------------------------------------------------------------- invariants
def test_transpose_identity_bitwise():
    # (AB)^T = B^T A^T: each entry keeps its k order, so equality is bitwise
    A = _rand((37, 29), 21, "normal")
    B = _rand((29, 41), 22, "normal")
    C, absAB = oracle.gemm(A, B)
    Ct, absABt = oracle.gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))
    assert np.array_equal(Ct.T, C)
    assert np.array_equal(absABt.T, absAB)


def test_row_and_column_permutations():
    rng = np.random.default_rng(3)
    A = _rand((31, 20), 31)
    B = _rand((20, 27), 32)
    C, _ = oracle.gemm(A, B)
    P = rng.permutation(31)
    Q = rng.permutation(27)
    assert np.array_equal(oracle.gemm(A[P], B)[0], C[P])
    assert np.array_equal(oracle.gemm(A, np.ascontiguousarray(B[:, Q]))[0], C[:, Q])


def test_zero_padding_is_invisible():
    # the tile simulator of "Lesson 10" pads every tile with zeros; padding K
    # (and M, N) with zeros must leave the product unchanged, bitwise
    A = _rand((35, 45), 42, "normal")
    B = _rand((45, 25), 43, "normal")
    C, absAB = oracle.gemm(A, B)
    T = 16
    Mp, Kp, Np = 48, 48, 32
    Ap = np.zeros((Mp, Kp), np.float32)
    Ap[:35, :45] = A
    Bp = np.zeros((Kp, Np), np.float32)
    Bp[:45, :25] = B
    Cp, absABp = oracle.gemm(Ap, Bp)
    assert np.array_equal(Cp[:35, :25], C)
    assert np.array_equal(absABp[:35, :25], absAB)
    assert not Cp[35:, :].any() and not Cp[:, 25:].any()
    assert Kp % T == 0


def test_lesson10_simulator_shape_against_library_matmul():
    # the unit-test shape of "Lesson 10" (35x45 times 45x25, normal inputs,
    # absolute tolerance 1e-5); here compared with numpy's float64 matmul,
    # an independent library routine, rounded to float
    A = _rand((35, 45), 42, "normal")
    B = _rand((45, 25), 7, "normal")
    C, _ = oracle.gemm(A, B)
    ref = (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)
    assert np.allclose(C, ref, rtol=0, atol=1e-5)
    # and a tile-by-tile simulation with T = 16 zero-padded tiles
    T = 16
    acc = np.zeros((48, 32), np.float64)
    Ap = np.zeros((48, 48)); Ap[:35, :45] = A
    Bp = np.zeros((48, 32)); Bp[:45, :25] = B
    for k0 in range(0, 48, T):
        acc += Ap[:, k0:k0 + T] @ Bp[k0:k0 + T, :]
    assert np.allclose(C, acc[:35, :25].astype(np.float32), rtol=0, atol=1e-5)


# ----------------------------------------------------------------- brute force
def _all_ternary(rows, cols):
    n = rows * cols
    for code in range(3 ** n):
        vals = []
        c = code
        for _ in range(n):
            vals.append(c % 3 - 1)
            c //= 3
        yield np.array(vals, np.float32).reshape(rows, cols)


def test_brute_force_ternary_2x2x2():
    As = list(_all_ternary(2, 2))
    Bs = list(_all_ternary(2, 2))
    for A in As[::7]:
        for B in Bs:
            C, absAB = oracle.gemm(A, B)
            Ai = A.astype(np.int64)
            Bi = B.astype(np.int64)
            want = [[sum(int(Ai[i, k]) * int(Bi[k, j]) for k in range(2)) for j in range(2)] for i in range(2)]
            want_abs = [[sum(abs(int(Ai[i, k]) * int(Bi[k, j])) for k in range(2)) for j in range(2)] for i in range(2)]
            assert C.tolist() == want
            assert absAB.tolist() == want_abs


def test_brute_force_ternary_1x3x2():
    for A in _all_ternary(1, 3):
        for B in list(_all_ternary(3, 2))[::3]:
            C, _ = oracle.gemm(A, B)
            want = [[int(sum(A[0, k] * B[k, j] for k in range(3))) for j in range(2)]]
            assert C.tolist() == want


@pytest.mark.parametrize("seed", range(12))
def test_random_tiny_against_exact_rationals(seed):
    rng = np.random.default_rng(100 + seed)
    M, K, N = (int(x) for x in rng.integers(1, [5, 6, 4]))
    law = ["uniform", "normal"][seed % 2]
    A = workloads.draw(rng, (M, K), law)
    B = workloads.draw(rng, (K, N), law)
    C, absAB = oracle.gemm(A, B)
    Cpy, absABpy = oracle.gemm_py(A, B)
    assert np.array_equal(C, Cpy) and np.array_equal(absAB, absABpy)
    for i in range(M):
        for j in range(N):
            q = exact_dot(A[i, :], B[:, j])
            qa = exact_abs_dot(A[i, :], B[:, j])
            r = round_f32(q)
            bound = 0.5 * ulp_f32(r) + K * 2.0 ** -53 * float(qa)
            assert abs(float(C[i, j]) - float(q)) <= bound + 1e-300
            if C[i, j] != r:    # only a double rounding may move it, by one ulp
                assert abs(float(C[i, j]) - float(r)) <= ulp_f32(r)
            assert abs(absAB[i, j] - float(qa)) <= K * 2.0 ** -52 * float(qa)


@pytest.mark.parametrize("name", ["1001x513x777", "4096x4096x4096"])
def test_sampled_entries_within_exact_bound(name):
    """P-R: 100 random entries lie within 0.5 ulp + K*2^-53*absAB of exact."""
    A, B = workloads.problem_inputs(name)
    M, K = A.shape
    N = B.shape[1]
    rng = np.random.default_rng(7)
    rows = rng.integers(0, M, 100)
    cols = rng.integers(0, N, 100)
    vals, absv = oracle.gemm_entries(A, B, rows, cols)
    hits = 0
    for t in range(100):
        i, j = int(rows[t]), int(cols[t])
        q = exact_dot(A[i, :], B[:, j])
        qa = float(exact_abs_dot(A[i, :], B[:, j]))
        r = round_f32(q)
        assert abs(float(vals[t]) - float(q)) <= 0.5 * ulp_f32(r) + K * 2.0 ** -53 * qa
        assert abs(absv[t] - qa) <= K * 2.0 ** -52 * qa
        hits += vals[t] == r
    assert hits >= 95      # double rounding is rare


def test_entries_equal_full_product_bitwise():
    A, B = workloads.problem_inputs("1001x513x777")
    C, absAB = oracle.gemm(A, B)
    rng = np.random.default_rng(9)
    rows = rng.integers(0, A.shape[0], 500)
    cols = rng.integers(0, B.shape[1], 500)
    vals, absv = oracle.gemm_entries(A, B, rows, cols)
    assert np.array_equal(vals, C[rows, cols])
    assert np.array_equal(absv, absAB[rows, cols])


# ----------------------------------------------------------------- integers
def test_integer_problem_exact():
    A, B = workloads.problem_inputs("100x37x70-int")
    assert A.min() >= -8 and A.max() <= 8 and B.min() >= -8 and B.max() <= 8
    C, absAB = oracle.gemm(A, B)
    Ci = A.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(C, Ci.astype(np.float32))
    assert np.array_equal(absAB, (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)).astype(np.float64))


def test_integer_k512_exact():
    A, B = workloads.make_inputs(96, 512, 80, "int8", 5)
    C, _ = oracle.gemm(A, B)
    Ci = A.astype(np.int64) @ B.astype(np.int64)
    assert np.abs(Ci).max() < 2 ** 24
    assert np.array_equal(C, Ci.astype(np.float32))


# ----------------------------------------------------------------- planted mistakes
def _pins_pass(fn):
    """Run a subset of the pins above against a candidate implementation."""
    try:
        A = _rand((5, 4), 1, "normal")
        B = _rand((4, 3), 2, "normal")
        C = fn(A, B)
        if C.shape != (5, 3):
            return False
        for i in range(5):
            for j in range(3):
                q = exact_dot(A[i, :], B[:, j])
                if abs(float(C[i, j]) - float(q)) > ulp_f32(round_f32(q)) + 1e-30:
                    return False
        # identity pins
        if not np.array_equal(fn(np.eye(4, dtype=np.float32), B), B):
            return False
        return True
    except Exception:
        return False


def test_planted_mistakes_fail_the_pins():
    def good(A, B):
        return oracle.gemm_py(A, B)[0]

    def transposed_b(A, B):       # indexes B's buffer as if it held B^T (j*K + k)
        M, K = A.shape
        N = B.shape[1]
        return np.array([[sum(float(A[i, k]) * float(B.flat[j * K + k]) for k in range(K))
                          for j in range(N)] for i in range(M)], np.float32)

    def dropped_last_term(A, B):
        return oracle.gemm_py(A[:, :-1], B[:-1, :])[0]

    def wrong_sign(A, B):
        C = oracle.gemm_py(A, B)[0].copy()
        C[-1, -1] = -C[-1, -1]
        return C

    def float64_library(A, B):        # a correct product by another route: control
        return (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)

    assert _pins_pass(good)
    assert not _pins_pass(transposed_b)
    assert not _pins_pass(dropped_last_term)
    assert not _pins_pass(wrong_sign)
    assert _pins_pass(float64_library)
