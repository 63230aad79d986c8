"""Dependent products queued back to back on one stream: each reads the C
the previous one wrote, with no synchronisation in between.  The tensor
and FFMA kernels are launched so that a kernel may begin as the previous one
finishes (programmatic dependent launch) and wait on the device before its
first global access; a read of a stale operand would show here.  Integer
inputs keep every intermediate exact (below 2^24, and split exactly by the
3xTF32 parts), so the last result must equal the oracle's chain bit for bit.
"""
import numpy as np
import pytest

import workloads
from tests._gpu import assert_bit_exact, lib, oracle_full

pytestmark = pytest.mark.gpu

FLAG_PAIR, FLAG_SINGLE = 0x400, 0x800


def _ints(rng, shape, lo, hi):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


def test_chain_of_dependent_products_on_one_stream():
    import torch

    g = lib()
    rng = np.random.default_rng(2027)
    A = _ints(rng, (512, 64), -2, 2)
    B = _ints(rng, (64, 384), -2, 2)      # C1 = A B    on CTA pairs
    D = _ints(rng, (384, 256), -1, 1)     # C2 = C1 D   FFMA, TMA loads
    E = _ints(rng, (256, 4096), -1, 1)    # C3 = C2 E   single-CTA tensor kernel
    F = _ints(rng, (4096, 64), 0, 1)      # C4 = C3 F   narrow tiles, K split across CTAs
    F[64:] = 0.0
    # the oracle's chain (asserted below) stays below 2^22 up to C3 and 2^24
    # for C4, so every product and sum is exact in every kernel
    dev = torch.device("cuda:0")
    s = torch.cuda.current_stream(dev)
    t = {k: torch.from_numpy(v).to(dev) for k, v in dict(A=A, B=B, D=D, E=E, F=F).items()}
    C1 = torch.full((512, 384), float("nan"), device=dev)
    C2 = torch.full((512, 256), float("nan"), device=dev)
    C3 = torch.full((512, 4096), float("nan"), device=dev)
    C4 = torch.full((512, 64), float("nan"), device=dev)
    for _ in range(3):   # the chain three times, still without synchronising
        assert g.gemm_f32_ex(t["A"], t["B"], C1, 512, 384, 64, "tc3x", FLAG_PAIR, s) == 0
        assert g.gemm_f32_ex(C1, t["D"], C2, 512, 256, 384, "ffma", 0, s) == 0
        assert g.gemm_f32_ex(C2, t["E"], C3, 512, 4096, 256, "tc3x", FLAG_SINGLE, s) == 0
        assert g.gemm_f32_ex(C3, t["F"], C4, 512, 64, 4096, "tc3x", 0, s) == 0
    assert g.gemm_f32_status(s) == (g.GEMM_F32_OK, 0)
    o1, _ = oracle_full(A, B)
    o2, _ = oracle_full(o1, D)
    o3, _ = oracle_full(o2, E)
    o4, _ = oracle_full(o3, F)
    assert np.abs(o4).max() < 2 ** 24 and np.abs(o3).max() < 2 ** 22
    assert_bit_exact(C1.cpu().numpy(), o1, "chain step 1")
    assert_bit_exact(C2.cpu().numpy(), o2, "chain step 2")
    assert_bit_exact(C3.cpu().numpy(), o3, "chain step 3")
    assert_bit_exact(C4.cpu().numpy(), o4, "chain step 4")
