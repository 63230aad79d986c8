"""CPU oracle for row-major FP32 GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
CUDA library never calls it, and it imports nothing from the CUDA side.

It computes the plain definition C[i][j] = sum_k A[i][k] * B[k][j]
("LeetGPU problem 2: matrix multiplication", yekq.top, section "problem
statement"; "Lesson 10: shared-memory tiled GEMM", hpc.payai.win, section
1), with every product formed exactly in double, the sum taken in double in
ascending k, and one round-to-nearest-even conversion to float.  In the
same pass it forms absAB[i][j] = sum_k |A[i][k]| * |B[k][j]|, which scales
the tolerance of every parity check.

Two implementations of the same formula live here:
  * ``gemm`` / ``gemm_entries``: plain C (``gemm_oracle.c``), OpenMP over
    rows, compiled with ``-ffp-contract=off``; ``gemm_general`` adds the
    scaled, strided and transposed form C = alpha op(A) op(B) + beta C;
  * ``gemm_py``: pure-Python loops, for tiny cases only.
Both are pinned by the ``-m "not gpu"`` tests against closed forms, brute
force with exact rational arithmetic, invariants and the pages' printed
numbers.  Nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle.so`` next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, ptr = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_gemm_f64acc.argtypes = [ptr, ptr, ptr, ptr, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_f64acc.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [ptr, ptr, i64, i64, i64, ptr, ptr, i64,
                                                ptr, ptr, ctypes.c_int]
            lib.oracle_gemm_entries.restype = ctypes.c_int
            f32 = ctypes.c_float
            lib.oracle_gemm_general.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, f32, ptr, i64,
                                                ptr, i64, f32, ptr, i64, ptr, ctypes.c_int]
            lib.oracle_gemm_general.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle inputs must be float32, got %s" % x.dtype)
    return x


def max_threads() -> int:
    """Threads an OpenMP region of the oracle uses by default."""
    return int(_load().oracle_max_threads())


def gemm(A, B, threads: int = 0):
    """Full product.  Returns (C float32 [M,N], absAB float64 [M,N])."""
    A = _as_f32(A)
    B = _as_f32(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shapes %s x %s do not chain" % (A.shape, B.shape))
    M, K = A.shape
    N = B.shape[1]
    C = np.empty((M, N), np.float32)
    absAB = np.empty((M, N), np.float64)
    rc = _load().oracle_gemm_f64acc(A.ctypes.data, B.ctypes.data, C.ctypes.data,
                                    absAB.ctypes.data, M, N, K, int(threads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_f64acc failed (%d)" % rc)
    return C, absAB


def gemm_entries(A, B, rows, cols, threads: int = 0):
    """Entries (rows[t], cols[t]) of the product, bitwise equal to ``gemm``'s.

    Returns (values float32 [n], absAB float64 [n])."""
    A = _as_f32(A)
    B = _as_f32(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shapes %s x %s do not chain" % (A.shape, B.shape))
    M, K = A.shape
    N = B.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and equally long")
    out = np.empty(rows.shape, np.float32)
    out_abs = np.empty(rows.shape, np.float64)
    rc = _load().oracle_gemm_entries(A.ctypes.data, B.ctypes.data, M, N, K,
                                     rows.ctypes.data, cols.ctypes.data, rows.size,
                                     out.ctypes.data, out_abs.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_entries failed (%d)" % rc)
    return out, out_abs


def gemm_general(A, B, C, M: int, N: int, K: int, alpha: float = 1.0, beta: float = 0.0,
                 trans_a: bool = False, trans_b: bool = False, threads: int = 0):
    """C = alpha * op(A) * op(B) + beta * C on row-major storage arrays.

    A, B, C are 2-D float32 arrays holding the stored matrices; each one's
    row stride is its width (so a wider array is a padded leading
    dimension).  With trans_a, A stores op(A)^T (K x M window); with
    trans_b, B stores op(B)^T (N x K window).  Only C[:M, :N] changes.
    Returns (new C, a copy; absC float64 [M, N] = |alpha| |op(A)||op(B)| +
    |beta| |C_old|)."""
    A = _as_f32(A)
    B = _as_f32(B)
    C = _as_f32(C).copy()
    for name, x in (("A", A), ("B", B), ("C", C)):
        if x.ndim != 2:
            raise ValueError("%s must be 2-D" % name)
    ra, ca = (K, M) if trans_a else (M, K)
    rb, cb = (N, K) if trans_b else (K, N)
    if A.shape[0] < ra or A.shape[1] < ca or B.shape[0] < rb or B.shape[1] < cb \
            or C.shape[0] < M or C.shape[1] < N:
        raise ValueError("stored arrays smaller than the windows")
    absC = np.empty((M, N), np.float64)
    rc = _load().oracle_gemm_general(int(bool(trans_a)), int(bool(trans_b)), M, N, K, float(alpha),
                                     A.ctypes.data, A.shape[1], B.ctypes.data, B.shape[1],
                                     float(beta), C.ctypes.data, C.shape[1], absC.ctypes.data,
                                     int(threads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_general failed (%d)" % rc)
    return C, absC


def gemm_py(A, B):
    """Pure-Python loops (tiny inputs only): same definition and order."""
    A = _as_f32(A)
    B = _as_f32(B)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("shapes do not chain")
    a = A.tolist()
    b = B.tolist()
    C = np.empty((M, N), np.float32)
    absAB = np.empty((M, N), np.float64)
    for i in range(M):
        for j in range(N):
            s = 0.0
            s_abs = 0.0
            for k in range(K):
                s += a[i][k] * b[k][j]      # Python float = IEEE double
                s_abs += abs(a[i][k]) * abs(b[k][j])
            C[i, j] = np.float32(s)
            absAB[i, j] = s_abs
    return C, absAB
