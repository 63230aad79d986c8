"""gemm_f32_host: C = A * B with host buffers (copies in, product, copy out,
pipelined across calls through two device slots).  Parity with the oracle
as gemm_f32_ex's, and the reuse of the device slots is checked by queueing
several calls with different operands, sizes and outputs before reading any
result (a slot overwritten too early would corrupt an earlier result)."""
import numpy as np
import pytest

import workloads
from tests._gpu import TOL, assert_bit_exact, assert_close, lib, oracle_full

pytestmark = pytest.mark.gpu


def pinned(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def host_call(A, B, mode="tc3x", use_pinned=True):
    import torch
    g = lib()
    M, K = A.shape
    N = B.shape[1]
    if use_pinned:
        a, b = pinned(A), pinned(B)
        c = torch.full((M, N), float("nan")).pin_memory()
    else:
        a, b = np.ascontiguousarray(A), np.ascontiguousarray(B)
        c = np.full((M, N), np.nan, np.float32)
    s = torch.cuda.current_stream()
    g.check(g.gemm_f32_host(a, b, c, M, N, K, mode, s))
    rc, site = g.gemm_f32_status(s)
    assert rc == 0, site
    return c.numpy() if use_pinned else c


@pytest.mark.parametrize("mode", ["tc3x", "ffma", "tc1x"])
@pytest.mark.parametrize("name", ["100x37x70", "1024x512x1024", "1001x513x777"])
def test_host_buffers_within_tolerance(name, mode):
    A, B = workloads.problem_inputs(name)
    Co, absAB = oracle_full(A, B)
    C = host_call(A, B, mode)
    assert_close(C, Co, absAB, TOL[mode], "host %s/%s" % (name, mode))


def test_host_buffers_pageable_memory():
    A, B = workloads.problem_inputs("1001x513x777")
    Co, absAB = oracle_full(A, B)
    C = host_call(A, B, "tc3x", use_pinned=False)
    assert_close(C, Co, absAB, TOL["tc3x"], "pageable")


def test_host_buffers_integers_exact():
    A, B = workloads.problem_inputs("100x37x70-int")
    Co, _ = oracle_full(A, B)
    assert_bit_exact(host_call(A, B, "tc3x"), Co, "host 100x37x70-int")


def test_host_k_zero_writes_zeros():
    C = host_call(np.zeros((7, 0), np.float32), np.zeros((0, 9), np.float32))
    assert np.all(C == 0)


def test_queued_calls_keep_their_own_operands():
    # eight calls queued back to back on alternating slots, sizes growing and
    # shrinking (a slot reallocates mid-sequence), results read only at the end
    import torch
    g = lib()
    shapes = [(300, 200, 250), (513, 129, 777), (64, 64, 64), (1024, 512, 1024),
              (300, 200, 250), (1500, 300, 900), (17, 1000, 33), (1024, 512, 1024)]
    s = torch.cuda.current_stream()
    jobs = []
    for t, (M, K, N) in enumerate(shapes):
        A, B = workloads.make_inputs(M, K, N, "uniform", 500 + t)
        a, b = pinned(A), pinned(B)
        c = torch.full((M, N), float("nan")).pin_memory()
        g.check(g.gemm_f32_host(a, b, c, M, N, K, "tc3x", s))
        jobs.append((A, B, a, b, c))
    rc, site = g.gemm_f32_status(s)
    assert rc == 0, site
    for t, (A, B, _, _, c) in enumerate(jobs):
        Co, absAB = oracle_full(A, B)
        assert_close(c.numpy(), Co, absAB, TOL["tc3x"], "queued call %d" % t)


def test_release_frees_the_slots_and_calls_still_work():
    g = lib()
    A, B = workloads.problem_inputs("1024x512x1024")
    host_call(A, B)
    assert g.gemm_f32_release() == 0
    Co, absAB = oracle_full(A, B)
    assert_close(host_call(A, B), Co, absAB, TOL["tc3x"], "after release")
