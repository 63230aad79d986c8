"""The bounds-checked debug build (libgemm_f32_checked.so, -DGEMM_BOUNDS_CHECK).

In it every hand-indexed global load and store -- per-thread operand loads,
FFMA copies, C stores, split-tail partials, operand packing, the small and
teaching kernels -- is checked against its array's extent; an index outside
is skipped and recorded in the error word, which every parity helper reads
through gemm_f32_status() after each call.  This test builds that library
and runs the parity tests that reach those paths (tiny and ragged shapes,
misaligned bases, forced per-thread loads, packed operands, split tails,
CTA pairs, the general form with transposes and strides, the ladder, the
FFMA skinny tiles) on it, in a child pytest process: any out-of-extent
index fails them with site 16-20, any wrong value with the usual bound.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELECTION = " or ".join([
    "test_small_configs_within_tolerance", "test_integer_config_bit_exact",
    "test_every_tensor_variant_on_ragged_and_regular", "test_one_tile_per_cta_grid",
    "test_edge_sweep", "test_misaligned_base_pointers", "test_degenerate_shapes",
    "test_split_tail_matches_whole_tiles", "test_cta_pair_path", "test_narrow_tiles",
    "test_large_operands_tma_cannot_read_are_packed", "test_forced_staged_large_misaligned",
    "test_ffma_skinny_tiles", "test_general", "test_ladder",
])


def test_checked_build_reports_no_out_of_extent_access():
    from accelerator_row_major_gb300 import build as build_mod
    lib = build_mod.build(checked=True)
    env = dict(os.environ, GEMM_F32_LIBRARY=lib)
    probe = subprocess.run(
        [sys.executable, "-c", "import accelerator_row_major_gb300 as g; print(g.gemm_f32_version())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr
    assert probe.stdout.strip().endswith("bounds-checked"), probe.stdout
    run = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
         "tests/test_gpu_parity.py", "tests/test_gpu_general.py", "tests/test_gpu_ladder.py",
         "-k", SELECTION],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((run.stdout + run.stderr).splitlines()[-30:])
    assert run.returncode == 0, tail
    assert " passed" in run.stdout and "failed" not in run.stdout, tail
