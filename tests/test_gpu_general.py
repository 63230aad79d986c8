"""Parity of gemm_f32_general (C = alpha op(A) op(B) + beta C on row-major
storage with row strides and stored transposes: the cuBLAS call on "LeetGPU
problem 2: matrix multiplication", yekq.top, section "cuBLAS reference",
restated for row-major matrices) with the oracle's general form.

Bound: |C - C_oracle| <= tol * (|alpha| |op(A)||op(B)| + |beta| |C_old|),
tol as gemm_f32_ex's for the mode; integers exact; nothing written outside
the C window (padding and guard bands checked on every call)."""
import numpy as np
import pytest

import oracle
import workloads
from tests._gpu import TOL, assert_bit_exact, assert_close, lib, run_general

pytestmark = pytest.mark.gpu

MODES = ["tc3x", "ffma", "tc1x"]


def stored(rng, rows, cols, pad, law="uniform"):
    """A row-major array of rows x cols values with `pad` NaN columns after
    each row (a leading dimension of cols + pad that must never be read)."""
    x = np.full((rows, cols + pad), np.nan, np.float32)
    x[:, :cols] = workloads.draw(rng, (rows, cols), law)
    return x


def case(seed, M, N, K, ta, tb, pads=(3, 5, 2), law="uniform"):
    rng = np.random.default_rng(seed)
    A = stored(rng, K, M, pads[0], law) if ta else stored(rng, M, K, pads[0], law)
    B = stored(rng, N, K, pads[1], law) if tb else stored(rng, K, N, pads[1], law)
    C = stored(rng, M + 2, N, pads[2], law)    # two extra rows below the window
    return A, B, C


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_general_ragged_with_padding(mode, ta, tb):
    M, N, K = 301, 259, 203
    A, B, C0 = case(10 + 2 * ta + tb, M, N, K, ta, tb)
    Co, absC = oracle.gemm_general(A, B, C0, M, N, K, alpha=1.5, beta=-0.75, trans_a=ta, trans_b=tb)
    C = run_general(A, B, C0, M, N, K, 1.5, -0.75, ta, tb, mode)
    assert_close(C[:M, :N], Co[:M, :N], absC, TOL[mode], "general %d%d/%s" % (ta, tb, mode))


@pytest.mark.parametrize("mode", MODES)
def test_general_aligned_strides_take_the_tma_path(mode):
    # strides padded by 4 floats keep 16-byte rows: the TMA path with strides
    M, N, K = 1024, 768, 512
    A, B, C0 = case(20, M, N, K, 0, 0, pads=(4, 8, 4))
    Co, absC = oracle.gemm_general(A, B, C0, M, N, K, alpha=-2.0, beta=0.5)
    C = run_general(A, B, C0, M, N, K, -2.0, 0.5, 0, 0, mode)
    assert_close(C[:M, :N], Co[:M, :N], absC, TOL[mode], "aligned strides/%s" % mode)


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("ta,tb,pads", [(0, 0, (4, 4, 4)), (1, 1, (3, 1, 2))])
def test_general_on_the_pair_kernel(mode, ta, tb, pads):
    # 90 tiles of 256 x 256 and a K deep enough for the pair kernel on the
    # TMA path (the operands are copied to TMA-readable form first)
    M, N, K = 2304, 2560, (3072 if mode == "tc3x" else 6144)
    A, B, C0 = case(30 + ta, M, N, K, ta, tb, pads=pads)
    Co, absC = oracle.gemm_general(A, B, C0, M, N, K, alpha=0.75, beta=1.25, trans_a=ta, trans_b=tb)
    C = run_general(A, B, C0, M, N, K, 0.75, 1.25, ta, tb, mode)
    assert lib().gemm_f32_last_kernel() == "tc_pair_kernel"
    assert_close(C[:M, :N], Co[:M, :N], absC, TOL[mode], "pair %d%d/%s" % (ta, tb, mode))


@pytest.mark.parametrize("mode", MODES)
def test_general_split_tail_applies_alpha_beta_once(mode):
    # few tiles, long K: the K range is split across CTAs and the partial
    # tiles are reduced at the end, where alpha and beta must be applied once
    M, N, K = 512, 384, 8192
    A, B, C0 = case(40, M, N, K, 0, 0, pads=(4, 4, 0))
    Co, absC = oracle.gemm_general(A, B, C0, M, N, K, alpha=3.0, beta=-1.0)
    C = run_general(A, B, C0, M, N, K, 3.0, -1.0, 0, 0, mode)
    assert_close(C[:M, :N], Co[:M, :N], absC, TOL[mode], "split/%s" % mode)


@pytest.mark.parametrize("mode", MODES)
def test_general_beta_zero_never_reads_c(mode):
    M, N, K = 130, 140, 70
    A, B, C0 = case(50, M, N, K, 1, 0)
    C0[:M, :N] = np.nan
    Co, absC = oracle.gemm_general(A, B, C0, M, N, K, alpha=2.0, beta=0.0, trans_a=1)
    C = run_general(A, B, C0, M, N, K, 2.0, 0.0, 1, 0, mode)
    assert not np.isnan(C[:M, :N]).any()
    assert_close(C[:M, :N], Co[:M, :N], absC, TOL[mode], "beta 0/%s" % mode)


@pytest.mark.parametrize("alpha,K", [(0.0, 50), (1.0, 0)])
def test_general_empty_product_scales_c(alpha, K):
    M, N = 70, 90
    A, B, C0 = case(60, M, N, max(K, 1), 0, 0)
    C = run_general(A, B, C0, M, N, K, alpha, -0.5, 0, 0, "tc3x")
    assert lib().gemm_f32_last_kernel() == "scale_window_kernel"
    assert np.array_equal(C[:M, :N], (C0[:M, :N] * np.float32(-0.5)).astype(np.float32))
    C = run_general(A, B, C0, M, N, K, alpha, 0.0, 0, 0, "tc3x")
    assert np.all(C[:M, :N] == 0)


@pytest.mark.parametrize("mode", MODES)
def test_general_integers_exact(mode):
    M, N, K = 200, 136, 96
    A, B, C0 = case(70, M, N, K, 1, 1, law="int8")
    C0[:M, :N] = np.round(C0[:M, :N] * 10)
    Co, _ = oracle.gemm_general(A, B, C0, M, N, K, alpha=2.0, beta=-1.0, trans_a=1, trans_b=1)
    C = run_general(A, B, C0, M, N, K, 2.0, -1.0, 1, 1, mode)
    assert_bit_exact(C[:M, :N], Co[:M, :N], "int general/%s" % mode)


def test_plain_form_equals_gemm_f32_ex():
    # alpha = 1, beta = 0 and unit strides: the same kernels as gemm_f32_ex,
    # bitwise
    import torch

    g = lib()
    A, B = workloads.make_inputs(700, 300, 500, "uniform", 80)
    dev = torch.device("cuda:0")
    a, b = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    c1 = torch.empty(700, 500, device=dev)
    c2 = torch.full((700, 500), float("nan"), device=dev)
    for mode in MODES:
        g.check(g.gemm_f32_ex(a, b, c1, 700, 500, 300, mode))
        g.check(g.gemm_f32_general(0, 0, 700, 500, 300, 1.0, a, 300, b, 500, 0.0, c2, 500, mode))
        torch.cuda.synchronize()
        assert torch.equal(c1.view(torch.int32), c2.view(torch.int32)), mode


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
@pytest.mark.parametrize("shape", [(3000, 60, 700), (60, 3000, 700), (5000, 64, 2048)])
def test_general_ffma_skinny_tiles(shape, ta, tb):
    """FFMA's tiles for N <= 64 (256 x 64) and M <= 64 (64 x 256) in the
    general form: strides, stored transposes, alpha / beta, split tails."""
    M, N, K = shape
    A, B, C0 = case(50 + M + ta, M, N, K, ta, tb)
    Co, absC = oracle.gemm_general(A, B, C0, M, N, K, alpha=-1.25, beta=0.5, trans_a=ta, trans_b=tb)
    C = run_general(A, B, C0, M, N, K, -1.25, 0.5, ta, tb, "ffma")
    assert lib().gemm_f32_last_kernel() == "ffma_gemm_kernel"
    assert_close(C[:M, :N], Co[:M, :N], absC, TOL["ffma"], "ffma skinny %s %d%d" % (shape, ta, tb))
