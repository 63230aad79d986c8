"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The test flag makes CTA 0's producer skip its first operand copy, so the
waits that depend on it give up after their 2 s budget.  The call must
return, gemm_f32_status() must report GEMM_F32_ETIMEOUT with a site code,
and the context must stay usable for the next call.
"""
import time

import numpy as np
import pytest

import workloads
from tests._gpu import TOL, assert_close, lib, oracle_full, run_abi

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,extra", [("tc3x", 0), ("tc1x", 0), ("tc3x", 0x400), ("ffma", 0)])
def test_lost_copy_reports_timeout_and_context_survives(mode, extra):
    import torch

    g = lib()
    A, B = workloads.make_inputs(256, 64, 256, "uniform", 8)
    dev = torch.device("cuda:0")
    At = torch.from_numpy(A).to(dev)
    Bt = torch.from_numpy(B).to(dev)
    C = torch.empty((256, 256), dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream(dev)
    t0 = time.time()
    rc = g.gemm_f32_ex(At, Bt, C, 256, 256, 64, mode, g.FLAG_TEST_DROP_COPY | extra, s)
    assert rc == g.GEMM_F32_OK
    st, site = g.gemm_f32_status(s)
    elapsed = time.time() - t0
    assert st == g.GEMM_F32_ETIMEOUT
    assert site in (1, 2, 3, 4, 5, 6, 7, 8)
    assert 1.5 < elapsed < 30.0
    # the error word was cleared by the read, and the context still works
    assert g.gemm_f32_status(s) == (g.GEMM_F32_OK, 0)
    Co, absAB = oracle_full(A, B)
    C2, _ = run_abi(A, B, mode)
    assert_close(C2, Co, absAB, TOL[mode], "after timeout/%s" % mode)


def test_per_thread_copies_ignore_the_test_flag():
    # an odd K keeps FFMA on its per-thread copies, which have no waits
    g = lib()
    A, B = workloads.make_inputs(200, 63, 136, "uniform", 9)
    Co, absAB = oracle_full(A, B)
    C, _ = run_abi(A, B, "ffma", g.FLAG_TEST_DROP_COPY)
    assert_close(C, Co, absAB, TOL["ffma"], "ffma with test flag")


@pytest.mark.parametrize("mode,flags", [("tc3x", 0), ("tc3x", 0x800), ("tc1x", 0), ("ffma", 0)])
def test_split_tail_after_a_timeout_needs_no_status_call(mode, flags):
    """A split-tail call whose bounded waits run out leaves some tile
    counters of its workspace half counted (CTA 0 never publishes its
    partials).  The next split-tail call on the same stream, made without
    gemm_f32_status() in between, must still pick the right CTA to sum each
    tile: its whole C is compared with the oracle.  3000 x 4096 x 2000
    splits its last wave along K on the CTA-pair kernel (default), on the
    single-CTA kernel (0x800) and on the FFMA kernel's TMA path."""
    import torch

    g = lib()
    M, K, N = 3000, 4096, 2000
    A, B = workloads.make_inputs(M, K, N, "normal", 41)
    Co, absAB = oracle_full(A, B)
    dev = torch.device("cuda:0")
    At = torch.from_numpy(A).to(dev)
    Bt = torch.from_numpy(B).to(dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream(dev)
    assert g.gemm_f32_ex(At, Bt, C, M, N, K, mode, flags, s) == g.GEMM_F32_OK
    assert g.gemm_f32_status(s) == (g.GEMM_F32_OK, 0)
    assert g.gemm_f32_ex(At, Bt, C, M, N, K, mode, flags | g.FLAG_TEST_DROP_COPY, s) == g.GEMM_F32_OK
    for call in range(2):
        C.fill_(float("nan"))
        assert g.gemm_f32_ex(At, Bt, C, M, N, K, mode, flags, s) == g.GEMM_F32_OK
        st, site = g.gemm_f32_status(s)
        if call == 0:
            assert st == g.GEMM_F32_ETIMEOUT and site in range(1, 9)
        else:
            assert (st, site) == (g.GEMM_F32_OK, 0)
        assert_close(C.cpu().numpy(), Co, absAB, TOL[mode], "call %d after a timeout/%s/%#x" % (call, mode, flags))
