"""Helpers for the GPU parity tests: run the C ABI with guard bands and
compare with the oracle element by element."""
from __future__ import annotations

import numpy as np

import oracle

GUARD = 1024                       # floats of sentinel on each side of C
SENTINEL = np.uint32(0x7FC0DEAD)   # a NaN payload no kernel writes

TOL = {"tc3x": 1e-5, "ffma": 1e-5, "tc1x": 2e-3}


def lib():
    from accelerator_row_major_gb300 import build as build_mod
    build_mod.build()
    import accelerator_row_major_gb300 as g
    return g


def run_abi(A: np.ndarray, B: np.ndarray, mode="tc3x", flags=0, offset_a=0, offset_b=0,
            offset_c=0, repeats=1, stream=None, ladder_step=None):
    """C = A @ B through gemm_f32_ex on cuda:0 (through gemm_f32_ladder with
    that step when ladder_step is given).

    offset_*: extra floats before each operand (4 bytes each), to move the
    base pointers off 16-byte alignment.  C sits inside a sentinel-filled
    buffer; returns (C, results of every repeat)."""
    import torch

    g = lib()
    M, K = A.shape
    N = B.shape[1]
    dev = torch.device("cuda:0")
    a_buf = torch.empty(offset_a + M * K + 1, dtype=torch.float32, device=dev)
    b_buf = torch.empty(offset_b + K * N + 1, dtype=torch.float32, device=dev)
    a_buf[offset_a:offset_a + M * K].copy_(torch.from_numpy(A.reshape(-1)))
    b_buf[offset_b:offset_b + K * N].copy_(torch.from_numpy(B.reshape(-1)))
    c_host = np.full(GUARD + offset_c + M * N + GUARD, SENTINEL, dtype=np.uint32)
    c_buf = torch.from_numpy(c_host.view(np.float32)).to(dev)
    a_ptr = a_buf.data_ptr() + 4 * offset_a
    b_ptr = b_buf.data_ptr() + 4 * offset_b
    c_ptr = c_buf.data_ptr() + 4 * (GUARD + offset_c)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    outs = []
    for _ in range(repeats):
        if ladder_step is None:
            rc = g.gemm_f32_ex(a_ptr, b_ptr, c_ptr, M, N, K, mode, flags, s)
        else:
            rc = g.gemm_f32_ladder(a_ptr, b_ptr, c_ptr, M, N, K, ladder_step, s)
        assert rc == g.GEMM_F32_OK, "the call returned %d" % rc
        # the product, plus up to two launches copying operands for TMA
        expect = (0,) if (M == 0 or N == 0) else (1, 2, 3)
        assert g.gemm_f32_last_launches() in expect
        st, site = g.gemm_f32_status(s)
        assert st == g.GEMM_F32_OK, "device error word: site %d" % site
        host = c_buf.cpu().numpy().view(np.uint32)
        outs.append(host[GUARD + offset_c:GUARD + offset_c + M * N].view(np.float32).reshape(M, N).copy())
        guards = np.concatenate([host[:GUARD + offset_c], host[GUARD + offset_c + M * N:]])
        assert np.all(guards == SENTINEL), "a write landed outside C"
    return outs[-1], outs


def assert_close(C: np.ndarray, Co: np.ndarray, absAB: np.ndarray, tol: float, what=""):
    """|C - C_oracle| <= tol * (|A||B|)_ij for every element; no NaN."""
    assert not np.isnan(C).any(), "NaN in C " + what
    err = np.abs(C.astype(np.float64) - Co.astype(np.float64))
    bound = tol * absAB
    bad = err > bound
    if bad.any():
        i, j = np.argwhere(bad)[0]
        ratio = (err / np.where(absAB > 0, absAB, 1)).max()
        raise AssertionError("%s: %d elements out of bound; first (%d,%d): got %r want %r absAB %r; "
                             "max err/absAB %.3e" % (what, bad.sum(), i, j, C[i, j], Co[i, j],
                                                     absAB[i, j], ratio))


# (what, max err / (|A||B|), bound) of the full-size comparisons, printed in
# the terminal summary (tests/conftest.py)
ERROR_REPORT = []


def max_rel_err(C, Co, absAB):
    err = np.abs(C.astype(np.float64) - Co.astype(np.float64))
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(absAB > 0, err / absAB, np.where(err > 0, np.inf, 0.0))
    return float(r.max()) if r.size else 0.0


def assert_bit_exact(C: np.ndarray, Co: np.ndarray, what=""):
    """Equality after mapping -0.0 to +0.0 (float ==), NaN forbidden."""
    assert not np.isnan(C).any(), "NaN in C " + what
    bad = C != Co
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError("%s: %d elements differ; first (%d,%d): got %r want %r"
                             % (what, bad.sum(), i, j, C[i, j], Co[i, j]))


def sample_indices(M, N, count, seed):
    """Random entries plus the four corners and the ragged last row/column."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, count))
    cols = list(rng.integers(0, N, count))
    for i in (0, M - 1):
        for j in (0, N - 1):
            rows.append(i)
            cols.append(j)
    for j in rng.integers(0, N, 64):      # last row
        rows.append(M - 1)
        cols.append(int(j))
    for i in rng.integers(0, M, 64):      # last column
        rows.append(int(i))
        cols.append(N - 1)
    return np.array(rows, np.int64), np.array(cols, np.int64)


def oracle_full(A, B):
    return oracle.gemm(A, B)


def run_general(A_store, B_store, C_store, M, N, K, alpha, beta, trans_a=0, trans_b=0, mode="tc3x"):
    """gemm_f32_general on cuda:0 with the stored arrays as given (row strides
    = their widths).  C_store sits inside a sentinel guard band; checks that
    nothing outside the M x N window of C changed and returns the new C_store."""
    import torch

    g = lib()
    dev = torch.device("cuda:0")
    a = torch.from_numpy(np.ascontiguousarray(A_store)).to(dev)
    b = torch.from_numpy(np.ascontiguousarray(B_store)).to(dev)
    C_store = np.ascontiguousarray(C_store, dtype=np.float32)
    flat = np.concatenate([np.full(GUARD, SENTINEL, np.uint32), C_store.reshape(-1).view(np.uint32),
                           np.full(GUARD, SENTINEL, np.uint32)])
    c = torch.from_numpy(flat.view(np.float32).copy()).to(dev)
    s = torch.cuda.current_stream(dev)
    rc = g.gemm_f32_general(trans_a, trans_b, M, N, K, alpha, a.data_ptr(), A_store.shape[1],
                            b.data_ptr(), B_store.shape[1], beta, c.data_ptr() + 4 * GUARD,
                            C_store.shape[1], mode, s)
    assert rc == g.GEMM_F32_OK, "gemm_f32_general returned %d" % rc
    st, site = g.gemm_f32_status(s)
    assert st == g.GEMM_F32_OK, "device error word: site %d" % site
    host = c.cpu().numpy().view(np.uint32)
    assert np.all(host[:GUARD] == SENTINEL) and np.all(host[-GUARD:] == SENTINEL), "write outside C"
    out = host[GUARD:-GUARD].view(np.float32).reshape(C_store.shape).copy()
    outside = np.ones(C_store.shape, bool)
    outside[:M, :N] = False
    assert np.array_equal(out.view(np.uint32)[outside], C_store.view(np.uint32)[outside]), \
        "a write landed in C's padding"
    return out
