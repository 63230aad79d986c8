"""Parity of the pages' teaching kernels v0 .. v4 (gemm_f32_ladder) with the
CPU oracle ("LeetGPU problem 2: matrix multiplication", yekq.top, sections
v0 .. v4): fp32 fused multiply-adds, so the FFMA bound 1e-5 * (|A||B|)_ij;
integers in [-8, 8] bit-exact; nothing written outside C.  The ragged
configuration and the edge shapes exercise each step's zero-filled loads
and guarded stores (the pages' point about boundary checks)."""
import numpy as np
import pytest

import workloads
from tests._gpu import TOL, assert_bit_exact, assert_close, lib, oracle_full, run_abi

pytestmark = pytest.mark.gpu

STEPS = [0, 1, 2, 3, 4]


@pytest.fixture(scope="module")
def problems():
    out = {}
    for name in ("100x37x70", "100x37x70-int", "1024x512x1024", "1001x513x777"):
        A, B = workloads.problem_inputs(name)
        out[name] = (A, B) + oracle_full(A, B)
    return out


@pytest.mark.parametrize("step", STEPS)
@pytest.mark.parametrize("name", ["100x37x70", "1024x512x1024", "1001x513x777"])
def test_ladder_configs_within_tolerance(problems, name, step):
    A, B, Co, absAB = problems[name]
    C, _ = run_abi(A, B, ladder_step=step)
    assert_close(C, Co, absAB, TOL["ffma"], "%s/v%d" % (name, step))
    assert lib().gemm_f32_last_kernel() == "ladder_v%d" % step


@pytest.mark.parametrize("step", STEPS)
def test_ladder_integers_bit_exact(problems, step):
    A, B, Co, _ = problems["100x37x70-int"]
    C, _ = run_abi(A, B, ladder_step=step)
    assert_bit_exact(C, Co, "100x37x70-int/v%d" % step)


@pytest.mark.parametrize("step", STEPS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (17, 33, 65), (64, 16, 64), (65, 17, 65),
                                   (63, 15, 129), (1, 300, 1), (300, 1, 7), (129, 64, 3)])
def test_ladder_edge_shapes(step, shape):
    M, K, N = shape
    A, B = workloads.make_inputs(M, K, N, "uniform", 100 + M + K + N)
    Co, absAB = oracle_full(A, B)
    C, _ = run_abi(A, B, ladder_step=step)
    assert_close(C, Co, absAB, TOL["ffma"], "%s/v%d" % (shape, step))


@pytest.mark.parametrize("step", STEPS)
def test_ladder_k_zero_writes_zeros(step):
    A = np.zeros((5, 0), np.float32)
    B = np.zeros((0, 7), np.float32)
    C, _ = run_abi(A, B, ladder_step=step)
    assert np.all(C == 0)
    assert lib().gemm_f32_last_kernel() == "memset"


@pytest.mark.parametrize("step", STEPS)
def test_ladder_is_deterministic(problems, step):
    A, B, _, _ = problems["1001x513x777"]
    _, outs = run_abi(A, B, ladder_step=step, repeats=2)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
