"""Parity of the CUDA library (through the C ABI) with the CPU oracle.

Bars: |C - C_oracle| <= tol * (|A||B|)_ij with tol 1e-5 for tc3x and ffma
and 2e-3 for tc1x; integer inputs in [-8, 8] with K <= 512 bit-exact in
every mode; nothing written outside C; no NaN.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests._gpu import (ERROR_REPORT, TOL, assert_bit_exact, assert_close, lib, max_rel_err,
                        oracle_full, run_abi, sample_indices)

pytestmark = pytest.mark.gpu

MODES = ["tc3x", "ffma", "tc1x"]
FLAG_STAGED = 0x1
FLAG_TILE = {64: 0x10, 128: 0x20, 224: 0x80, 256: 0x40}
FLAG_ONE_TILE = 0x100
FLAG_NO_SPLIT = 0x200
FLAG_PAIR = 0x400
FLAG_SINGLE = 0x800


@pytest.fixture(scope="module")
def small_problems():
    out = {}
    for name in ("100x37x70", "100x37x70-int", "1024x512x1024", "1001x513x777"):
        A, B = workloads.problem_inputs(name)
        C, absAB = oracle_full(A, B)
        out[name] = (A, B, C, absAB)
    return out


# Without flags, products below the small-problem size (100x37x70, the edge sweep,
# most degenerate shapes) run on the small CUDA-core kernel; FLAG_SINGLE
# keeps them on the mode's own kernels (the tensor-core single-CTA kernel,
# or the FFMA kernel), so both are checked.
SMALL_OR_OWN = [0, FLAG_SINGLE]


@pytest.mark.parametrize("flags", SMALL_OR_OWN)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["100x37x70", "1024x512x1024", "1001x513x777"])
def test_small_configs_within_tolerance(small_problems, name, mode, flags):
    A, B, Co, absAB = small_problems[name]
    C, _ = run_abi(A, B, mode, flags)
    assert_close(C, Co, absAB, TOL[mode], "%s/%s/%#x" % (name, mode, flags))


@pytest.mark.parametrize("flags", SMALL_OR_OWN)
@pytest.mark.parametrize("mode", MODES)
def test_integer_config_bit_exact(small_problems, mode, flags):
    A, B, Co, _ = small_problems["100x37x70-int"]
    C, _ = run_abi(A, B, mode, flags)
    assert_bit_exact(C, Co, "100x37x70-int/%s/%#x" % (mode, flags))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("flags", [0, FLAG_STAGED])
def test_integer_k512_bit_exact(mode, flags):
    # the regular size with integer values: every partial sum is exact
    A, B = workloads.make_inputs(1024, 512, 1024, "int8", 11)
    Co, _ = oracle_full(A, B)
    C, _ = run_abi(A, B, mode, flags)
    assert_bit_exact(C, Co, "int 1024x512x1024/%s/%d" % (mode, flags))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("tm", [64, 128, 256])
@pytest.mark.parametrize("staged", [False, True])
def test_every_tensor_variant_on_ragged_and_regular(small_problems, mode, tm, staged):
    for name in ("1001x513x777", "1024x512x1024"):
        A, B, Co, absAB = small_problems[name]
        flags = FLAG_TILE[tm] | (FLAG_STAGED if staged else 0)
        C, _ = run_abi(A, B, mode, flags)
        assert_close(C, Co, absAB, TOL[mode], "%s/%s/tm%d/staged%d" % (name, mode, tm, staged))


@pytest.mark.parametrize("mode", MODES)
def test_one_tile_per_cta_grid(small_problems, mode):
    A, B, Co, absAB = small_problems["1001x513x777"]
    C, _ = run_abi(A, B, mode, FLAG_ONE_TILE)
    assert_close(C, Co, absAB, TOL[mode], "1001x513x777/one-tile/%s" % mode)


@pytest.mark.parametrize("mode", MODES)
def test_deterministic(small_problems, mode):
    A, B, _, _ = small_problems["1001x513x777"]
    _, outs = run_abi(A, B, mode, repeats=2)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


# sizes around tile and swizzle edges: 1, the vector width, 8, 16, 32,
# 64, 128, 256 and their neighbours
EDGE = [1, 2, 3, 4, 5, 7, 8, 15, 17, 31, 33, 63, 65, 127, 129, 255, 257]


def _edge_cases(seed, count):
    rng = np.random.default_rng(seed)
    cases = set()
    while len(cases) < count:
        cases.add(tuple(int(x) for x in rng.choice(EDGE, 3)))
    return sorted(cases)


@pytest.mark.parametrize("flags", SMALL_OR_OWN)
@pytest.mark.parametrize("mode", MODES)
def test_edge_sweep(mode, flags):
    for (M, K, N) in _edge_cases(5 + MODES.index(mode), 40):
        A, B = workloads.make_inputs(M, K, N, "uniform", M * 7 + K * 3 + N)
        Co, absAB = oracle_full(A, B)
        C, _ = run_abi(A, B, mode, flags)
        assert_close(C, Co, absAB, TOL[mode], "edge %dx%dx%d/%s/%#x" % (M, K, N, mode, flags))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_base_pointers(mode, offsets):
    A, B = workloads.make_inputs(300, 264, 200, "uniform", 77)
    Co, absAB = oracle_full(A, B)
    oa, ob, oc = offsets
    C, _ = run_abi(A, B, mode, offset_a=oa, offset_b=ob, offset_c=oc)
    assert_close(C, Co, absAB, TOL[mode], "misaligned %s/%s" % (offsets, mode))


@pytest.mark.parametrize("mode", MODES)
def test_k_zero_writes_zeros(mode):
    A = np.zeros((70, 0), np.float32)
    B = np.zeros((0, 90), np.float32)
    C, _ = run_abi(A, B, mode)
    assert C.shape == (70, 90) and not C.any()


@pytest.mark.parametrize("flags", SMALL_OR_OWN)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 513, 300), (300, 513, 1), (1, 1, 4096),
                                   (129, 1, 257), (2, 3000, 2)])
def test_degenerate_shapes(mode, shape, flags):
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "normal", sum(shape))
    Co, absAB = oracle_full(A, B)
    C, _ = run_abi(A, B, mode, flags)
    assert_close(C, Co, absAB, TOL[mode], "degenerate %s/%s/%#x" % (shape, mode, flags))


@pytest.mark.parametrize("flags", SMALL_OR_OWN)
def test_closed_forms_on_gpu(flags):
    # A = I gives B exactly in every mode for TF32-exact values; ones give
    # column sums of small integers exactly
    n = 200
    B = workloads.make_inputs(1, n, 150, "int8", 3)[1]
    for mode in MODES:
        C, _ = run_abi(np.eye(n, dtype=np.float32), B, mode, flags)
        assert_bit_exact(C, B, "identity/%s" % mode)
        C, _ = run_abi(np.ones((33, n), np.float32), B, mode, flags)
        assert_bit_exact(C, np.broadcast_to(B.sum(axis=0, dtype=np.float64).astype(np.float32), (33, 150)),
                         "ones/%s" % mode)


# The full-size problems in the default launch configuration, every element
# of C against the oracle in every mode.  The oracle runs once per problem
# (about 34 s for 8192^3 on 16 host cores) and is kept while that problem's
# modes run: the cases are ordered problem by problem.
FULL_SIZE = [(name, mode) for name in ("4096x4096x4096", "65536x1024x64", "64x4096x65536",
                                       "8192x8192x8192") for mode in MODES]
_full_cache = {}


def _full_oracle(name):
    if name not in _full_cache:
        _full_cache.clear()          # one problem's inputs and oracle at a time
        A, B = workloads.problem_inputs(name)
        C, absAB = oracle_full(A, B)
        _full_cache[name] = (A, B, C, absAB)
    return _full_cache[name]


@pytest.mark.parametrize("name,mode", FULL_SIZE)
def test_full_size_every_element(name, mode):
    A, B, Co, absAB = _full_oracle(name)
    C, _ = run_abi(A, B, mode)
    assert_close(C, Co, absAB, TOL[mode], "%s/%s" % (name, mode))
    ratio = max_rel_err(C, Co, absAB)
    ERROR_REPORT.append(("%s/%s (%s)" % (name, mode, lib().gemm_f32_last_kernel()), ratio, TOL[mode]))
    print("%s/%s max err/absAB %.3e" % (name, mode, ratio))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x", "ffma"])
@pytest.mark.parametrize("shape", [(700, 2000, 900), (700, 2001, 900), (256, 4096, 384),
                                   (512, 16384, 512), (3000, 2048, 2000), (1024, 512, 1024)])
def test_split_tail_matches_whole_tiles(mode, shape):
    """Tiles split along K (workspace, fixed-order sum) against whole tiles."""
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "normal", M + K + N)
    Co, absAB = oracle_full(A, B)
    C_split, outs = run_abi(A, B, mode, 0, repeats=2)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    C_whole, _ = run_abi(A, B, mode, FLAG_NO_SPLIT)
    assert_close(C_split, Co, absAB, TOL[mode], "split %s/%s" % (shape, mode))
    assert_close(C_whole, Co, absAB, TOL[mode], "whole %s/%s" % (shape, mode))


def test_split_tail_on_two_streams_and_after_release():
    import torch
    from tests._gpu import lib
    g = lib()
    A, B = workloads.make_inputs(1001, 513, 777, "uniform", 31)
    Co, absAB = oracle_full(A, B)
    s2 = torch.cuda.Stream(torch.device("cuda:0"))
    C, _ = run_abi(A, B, "tc3x", stream=s2)
    assert_close(C, Co, absAB, TOL["tc3x"], "second stream")
    assert g.gemm_f32_release() == g.GEMM_F32_OK
    C, _ = run_abi(A, B, "tc3x")
    assert_close(C, Co, absAB, TOL["tc3x"], "after release")


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("shape", [(1024, 512, 1024), (1001, 513, 777), (300, 264, 200),
                                   (700, 2000, 900), (3000, 2048, 2000), (129, 33, 257)])
def test_cta_pair_path(mode, staged, shape):
    """256 x 256 tiles on CTA pairs (cta_group::2), forced on any shape."""
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "uniform", 3 * M + K)
    Co, absAB = oracle_full(A, B)
    flags = FLAG_PAIR | (FLAG_STAGED if staged else 0)
    C, outs = run_abi(A, B, mode, flags, repeats=2)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert_close(C, Co, absAB, TOL[mode], "pair %s/%s/staged%d" % (shape, mode, staged))
    C, _ = run_abi(A, B, mode, flags | FLAG_NO_SPLIT)
    assert_close(C, Co, absAB, TOL[mode], "pair whole tiles %s/%s/staged%d" % (shape, mode, staged))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
def test_cta_pair_integer_bit_exact(mode):
    A, B = workloads.make_inputs(1024, 512, 1024, "int8", 12)
    Co, _ = oracle_full(A, B)
    C, _ = run_abi(A, B, mode, FLAG_PAIR)
    assert_bit_exact(C, Co, "pair int/%s" % mode)


def test_single_and_pair_agree_on_a_large_problem():
    A, B = workloads.make_inputs(2048, 1024, 2048, "normal", 21)
    C_pair, _ = run_abi(A, B, "tc3x", FLAG_PAIR)
    C_single, _ = run_abi(A, B, "tc3x", FLAG_SINGLE)
    rows, cols = sample_indices(2048, 2048, 3000, 5)
    vals, absv = oracle.gemm_entries(A, B, rows, cols)
    for C in (C_pair, C_single):
        assert_close(C[rows, cols][None, :], vals[None, :], absv[None, :], TOL["tc3x"], "pair/single")


def test_last_kernel_names_the_path():
    import torch
    from tests._gpu import lib
    g = lib()
    dev = torch.device("cuda:0")
    # 4096 x 4096 gives 256 tiles of 256 x 256: the pair path by default
    # once K is deep enough (3072 with three products, 6144 with one), the
    # single-SM path below that
    A = torch.zeros((4096, 6144), device=dev)
    B = torch.zeros((6144, 4096), device=dev)
    C = torch.empty((4096, 4096), device=dev)
    s = torch.cuda.current_stream(dev)
    for mode, K, flags, want in (("tc3x", 4096, 0, "tc_pair_kernel"),
                                 ("tc3x", 4096, FLAG_SINGLE, "tc_gemm_kernel"),
                                 ("tc3x", 1024, 0, "tc_gemm_kernel"),
                                 ("tc3x", 1024, FLAG_PAIR, "tc_pair_kernel"),
                                 ("tc3x", 3068, 0, "tc_gemm_kernel"),    # just below the K bound
                                 ("tc3x", 3072, 0, "tc_pair_kernel"),    # at it
                                 ("tc1x", 6144, 0, "tc_pair_kernel"),
                                 ("tc1x", 6140, 0, "tc_gemm_kernel"),
                                 ("tc1x", 4096, 0, "tc_gemm_kernel"),
                                 ("ffma", 64, 0, "ffma_gemm_kernel")):
        assert g.gemm_f32_ex(A, B, C, 4096, 4096, K, mode, flags, s) == 0
        assert g.gemm_f32_last_kernel() == want, (mode, K, flags)
    assert g.gemm_f32_ex(A, B, C, 4096, 4096, 0, "tc3x", 0, s) == 0
    assert g.gemm_f32_last_kernel() == "memset"
    # small products take the small CUDA-core kernel in every mode, unless a
    # flag asks for the mode's own kernels
    for mode in MODES:
        assert g.gemm_f32_ex(A, B, C, 100, 70, 37, mode, 0, s) == 0
        assert g.gemm_f32_last_kernel() == "small_gemm_kernel", mode
    assert g.gemm_f32_ex(A, B, C, 100, 70, 37, "tc3x", FLAG_SINGLE, s) == 0
    assert g.gemm_f32_last_kernel() == "tc_gemm_kernel"
    assert g.gemm_f32_ex(A, B, C, 1000, 1000, 100, "tc3x", 0, s) == 0
    assert g.gemm_f32_last_kernel() == "tc_gemm_kernel"
    assert g.gemm_f32_status(s) == (0, 0)
    assert not C.any()


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("shape", [(1000, 300, 64), (517, 129, 60), (64, 64, 4), (3000, 2048, 32),
                                   (256, 4096, 64), (1, 40, 8)])
def test_narrow_tiles(mode, shape):
    # N <= 64 on the TMA path: 64-column tiles with an M = 64 MMA (rows in
    # lanes 0-15 of each TMEM lane quarter); includes split tails (long K,
    # few tiles) and N below the tile width
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "uniform", 700 + M + N)
    Co, absAB = oracle_full(A, B)
    C, _ = run_abi(A, B, mode)
    assert_close(C, Co, absAB, TOL[mode], "narrow %s/%s" % (shape, mode))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("shape,flags", [((64, 65536, 64), 0), ((50, 20000, 40), 0),
                                         ((517, 129, 60), FLAG_SINGLE), ((64, 64, 4), FLAG_SINGLE),
                                         ((1, 40, 8), FLAG_SINGLE), ((1000, 300, 64), FLAG_TILE[64]),
                                         ((1000, 300, 64), FLAG_TILE[128]), ((3000, 700, 20), FLAG_TILE[256])])
def test_narrow_tiles_of_64_rows(mode, shape, flags):
    # 64-column tiles of every height, 64 rows mostly: with three products
    # B^T hi and lo stacked by lanes into an M = 128 operand (the
    # accumulator's lane halves summed through shared memory); the small
    # shapes are kept off the small-product kernel
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "normal", 710 + M + N)
    Co, absAB = oracle_full(A, B)
    C, outs = run_abi(A, B, mode, flags, repeats=2)
    assert lib().gemm_f32_last_kernel() == "tc_gemm_kernel"
    assert_close(C, Co, absAB, TOL[mode], "narrow 64-row %s/%s" % (shape, mode))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
def test_narrow_tiles_integers_exact(mode):
    A, B = workloads.make_inputs(777, 512, 64, "int8", 31)
    Co, _ = oracle_full(A, B)
    C, _ = run_abi(A, B, mode)
    assert_bit_exact(C, Co, "narrow int/%s" % mode)


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("shape,offsets", [((1027, 1029, 1031), (0, 0, 0)),
                                           ((1024, 1024, 1024), (1, 0, 0)),
                                           ((2049, 511, 1536), (0, 0, 0))])
def test_large_operands_tma_cannot_read_are_packed(mode, shape, offsets):
    # odd strides or unaligned bases in a product of at least 2^27
    # multiply-adds: the operands are copied into aligned buffers and the TMA
    # path runs (the copies, then the product)
    from tests._gpu import lib
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "uniform", 900 + M)
    Co, absAB = oracle_full(A, B)
    oa, ob, oc = offsets
    C, _ = run_abi(A, B, mode, offset_a=oa, offset_b=ob, offset_c=oc)
    assert_close(C, Co, absAB, TOL[mode], "packed %s/%s" % (shape, mode))
    assert lib().gemm_f32_last_launches() >= 2


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
def test_forced_staged_large_misaligned(mode):
    # the staged loads stay available for large products (FORCE_STAGED)
    M, K, N = 1027, 1029, 1031
    A, B = workloads.make_inputs(M, K, N, "uniform", 910)
    Co, absAB = oracle_full(A, B)
    C, _ = run_abi(A, B, mode, FLAG_STAGED)
    assert_close(C, Co, absAB, TOL[mode], "staged large/%s" % mode)


@pytest.mark.parametrize("mode,flags", [("tc3x", 0), ("tc3x", FLAG_SINGLE), ("ffma", 0), ("tc1x", 0)])
def test_output_beyond_two_to_the_31_elements(mode, flags):
    # C with 49152^2 = 2.4e9 elements (9.7 GB): every kernel's index
    # arithmetic must stay 64-bit where it addresses C; sampled entries,
    # including the last rows and columns, against the oracle
    import torch
    from tests._gpu import lib
    g = lib()
    M = N = 49152
    K = 32
    A_h, B_h = workloads.make_inputs(M, K, N, "uniform", 1234)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    C = torch.full((M, N), float("nan"), device=dev)
    s = torch.cuda.current_stream(dev)
    g.check(g.gemm_f32_ex(A, B, C, M, N, K, mode, flags, s))
    rc, site = g.gemm_f32_status(s)
    assert rc == 0, site
    rng = np.random.default_rng(5)
    rows = np.concatenate([rng.integers(0, M, 2000), [0, M - 1, M - 1, M - 2, 43690, 43691]])
    cols = np.concatenate([rng.integers(0, N, 2000), [0, N - 1, 0, N - 1, 43690, 5]])
    got = C[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)].cpu().numpy()
    want, absAB = oracle.gemm_entries(A_h, B_h, rows, cols)
    err = np.abs(got.astype(np.float64) - want)
    assert not np.isnan(got).any()
    assert (err <= TOL[mode] * absAB).all(), float((err / absAB).max())
    del C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["tc3x", "tc1x", "ffma"])
@pytest.mark.parametrize("shape", [(16384, 8192, 128), (128, 131072, 128), (512, 65536, 512)])
def test_split_tail_repeats_with_other_work_between(mode, shape):
    """Shapes whose every tile is split along K (up to 64 CTAs on one tile):
    twelve calls, each after a different split product on the same stream
    has overwritten the shared partial-tile workspace, give bitwise the same
    C, and sampled entries lie within the mode's bound of the oracle.  A
    partial read before its writer published it, or a tile counter left
    non-zero by an earlier call, would change some of them."""
    import torch
    from tests._gpu import lib
    g = lib()
    M, K, N = shape
    dev = torch.device("cuda:0")
    s = torch.cuda.current_stream(dev)
    A, B = workloads.make_inputs(M, K, N, "normal", 7 + M + N)
    dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    dC = torch.empty(M, N, dtype=torch.float32, device=dev)
    others = []
    for (m, k, n), seed in (((1024, 8192, 512), 3), ((128, 65536, 256), 4)):
        oA, oB = workloads.make_inputs(m, k, n, "uniform", seed)
        others.append((torch.from_numpy(oA).to(dev), torch.from_numpy(oB).to(dev),
                       torch.empty(m, n, dtype=torch.float32, device=dev), m, n, k))
    code = {"tc3x": g.MODE_TC3X, "tc1x": g.MODE_TC1X, "ffma": g.MODE_FFMA}[mode]
    first = None
    for it in range(12):
        oA, oB, oC, m, n, k = others[it % 2]
        assert g.gemm_f32_ex(oA, oB, oC, m, n, k, code, 0, s) == g.GEMM_F32_OK
        assert g.gemm_f32_ex(dA, dB, dC, M, N, K, code, 0, s) == g.GEMM_F32_OK
        got = dC.cpu().numpy()
        if first is None:
            first = got.copy()
        else:
            assert np.array_equal(got.view(np.uint32), first.view(np.uint32)), "call %d differs" % it
    st, site = g.gemm_f32_status(s)
    assert st == g.GEMM_F32_OK, "device error word: site %d" % site
    rows, cols = sample_indices(M, N, 600, 99)
    vals, absv = oracle.gemm_entries(A, B, rows, cols)
    assert_close(first[rows, cols][None, :], vals[None, :], absv[None, :], TOL[mode],
                 "split repeats %s/%s" % (shape, mode))


FFMA_SKINNY = [(1000, 300, 64), (517, 129, 60), (64, 4096, 3000), (33, 1000, 5000),
               (20000, 1024, 64), (64, 20000, 512), (65, 777, 63), (300, 2048, 1)]


@pytest.mark.parametrize("shape", FFMA_SKINNY)
def test_ffma_skinny_tiles(shape):
    """FFMA block tiles of 256 x 64 (N <= 64) and 64 x 256 (M <= 64), two
    CTAs per SM: ragged edges, split tails (long K, few tiles) and whole
    tiles, deterministic, against the oracle on every element."""
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "normal", 880 + M + N)
    Co, absAB = oracle_full(A, B)
    C, outs = run_abi(A, B, "ffma", FLAG_SINGLE, repeats=2)
    assert lib().gemm_f32_last_kernel() == "ffma_gemm_kernel"
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert_close(C, Co, absAB, TOL["ffma"], "ffma skinny %s" % (shape,))
    for flags in (FLAG_NO_SPLIT, FLAG_ONE_TILE):
        C, _ = run_abi(A, B, "ffma", flags)
        assert_close(C, Co, absAB, TOL["ffma"], "ffma skinny %s/%#x" % (shape, flags))
    C, _ = run_abi(A, B, "ffma", FLAG_SINGLE, offset_a=1, offset_b=3)
    assert_close(C, Co, absAB, TOL["ffma"], "ffma skinny %s/misaligned" % (shape,))


def test_ffma_skinny_integers_exact():
    for (M, K, N) in ((700, 512, 64), (64, 512, 900)):
        A, B = workloads.make_inputs(M, K, N, "int8", 5 + M)
        Co, _ = oracle_full(A, B)
        C, _ = run_abi(A, B, "ffma", FLAG_SINGLE)
        assert_bit_exact(C, Co, "ffma skinny int %dx%dx%d" % (M, K, N))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
@pytest.mark.parametrize("shape,flags", [
    ((1024, 512, 1024), FLAG_TILE[224]),      # 5 tile rows, the last one 128 rows
    ((1000, 300, 64), FLAG_TILE[224]),        # narrow tiles
    ((2000, 8192, 64), FLAG_TILE[224]),       # split tail: partials of 224 x 64 (odd float4 count per thread)
    ((2000, 8192, 300), FLAG_TILE[224]),      # split tail, 128-column tiles
    ((60000, 1024, 100), 0),                  # chosen by the wave model: 268 tiles, two waves
    ((60000, 512, 64), 0),                    # chosen, narrow
])
def test_tiles_of_224_rows(mode, shape, flags):
    """224-row tiles (TMA path): ragged last tile rows, split tails and the
    heights the wave model picks, against the oracle on every element."""
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "normal", 224 + M + N)
    Co, absAB = oracle_full(A, B)
    C, outs = run_abi(A, B, mode, flags, repeats=2)
    assert lib().gemm_f32_last_kernel() == "tc_gemm_kernel"
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert_close(C, Co, absAB, TOL[mode], "224 rows %s/%s/%#x" % (shape, mode, flags))


@pytest.mark.parametrize("mode", ["tc3x", "tc1x"])
def test_tiles_of_224_rows_integers_exact(mode):
    A, B = workloads.make_inputs(1000, 512, 200, "int8", 224)
    Co, _ = oracle_full(A, B)
    C, _ = run_abi(A, B, mode, FLAG_TILE[224])
    assert_bit_exact(C, Co, "224 rows int/%s" % mode)
