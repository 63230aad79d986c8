"""Host-side checks of the C-ABI library that need no GPU.

The library must build with nvcc here, load without a GPU, export every
function include/gemm_f32.h declares, and reject malformed requests on the
host before it makes any CUDA call.
"""
import ctypes
import subprocess

import pytest

from accelerator_row_major_gb300 import build as build_mod


@pytest.fixture(scope="module")
def g():
    build_mod.build()
    import accelerator_row_major_gb300 as pkg
    return pkg


def test_header_declares_the_entry_points(g):
    names = g.declared_symbols()
    assert names == sorted(["gemm_f32", "gemm_f32_ex", "gemm_f32_status", "gemm_f32_ladder",
                            "gemm_f32_general", "gemm_f32_host",
                            "gemm_f32_last_kernel", "gemm_f32_last_launches", "gemm_f32_noalloc",
                            "gemm_f32_release", "gemm_f32_unit_rates",
                            "gemm_f32_clock_record", "gemm_f32_version"])


def test_library_exports_every_declared_symbol(g):
    lib = ctypes.CDLL(g.LIB_PATH)
    for name in g.declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in g.declared_symbols():
        assert name in exported, name


def test_version(g):
    assert g.gemm_f32_version().startswith("gemm_f32 ")
    assert "sm_103a" in g.gemm_f32_version()
    assert not g.gemm_f32_version().endswith("bounds-checked")   # the default build


def test_unit_rates_rejects_a_null_record(g):
    from accelerator_row_major_gb300 import _binding
    assert _binding.lib().gemm_f32_unit_rates(None) == g.GEMM_F32_EINVAL


def test_clock_record_rejects_null_outputs(g):
    # checked before the device is touched, so this runs without a GPU
    from accelerator_row_major_gb300 import _binding
    c = ctypes.c_ulonglong(7)
    assert _binding.lib().gemm_f32_clock_record(None, None, ctypes.byref(c)) == g.GEMM_F32_EINVAL
    assert c.value == 0
    assert _binding.lib().gemm_f32_clock_record(None, ctypes.byref(c), None) == g.GEMM_F32_EINVAL


def test_tile224_flag_is_known_and_exclusive(g):
    # 224-row tiles are a tile-height flag like the others: accepted alone
    # (the call then stops at the device check), refused with another height
    args = (FAKE_A, FAKE_B, FAKE_C, 4, 4, 4)
    assert g.gemm_f32_ex(*args, mode=0, flags=0x80) != g.GEMM_F32_EINVAL
    assert g.gemm_f32_ex(*args, mode=0, flags=0x80 | 0x40) == g.GEMM_F32_EINVAL


FAKE_A, FAKE_B, FAKE_C = 0x100000, 0x200000, 0x300000


@pytest.mark.parametrize("args,mode,flags", [
    ((FAKE_A, FAKE_B, FAKE_C, -1, 4, 4), 0, 0),          # negative M
    ((FAKE_A, FAKE_B, FAKE_C, 4, -1, 4), 0, 0),          # negative N
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, -3), 0, 0),          # negative K
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, 4), 7, 0),           # unknown mode
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, 4), 0, 0x8000),      # unknown flag
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, 4), 0, 0x30),        # two tile widths
    ((FAKE_A, FAKE_B, 0, 4, 4, 4), 0, 0),                # null C
    ((0, FAKE_B, FAKE_C, 4, 4, 4), 0, 0),                # null A with K > 0
    ((FAKE_A, FAKE_B, FAKE_A + 8, 4, 4, 4), 1, 0),       # C overlaps A
    ((FAKE_A, FAKE_B, FAKE_B - 16, 4, 4, 4), 2, 0),      # C overlaps B
    ((FAKE_A + 2, FAKE_B, FAKE_C, 4, 4, 4), 0, 0),       # A not 4-byte aligned
])
def test_malformed_requests_are_rejected_on_the_host(g, args, mode, flags):
    assert g.gemm_f32_ex(*args, mode=mode, flags=flags) == g.GEMM_F32_EINVAL
    assert g.gemm_f32_last_launches() == 0


@pytest.mark.parametrize("args,step", [
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, 4), -1),             # step below 0
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, 4), 5),              # step above 4
    ((FAKE_A, FAKE_B, FAKE_C, -1, 4, 4), 0),             # negative M
    ((FAKE_A, FAKE_B, 0, 4, 4, 4), 3),                   # null C
    ((FAKE_A, FAKE_B, FAKE_A + 8, 4, 4, 4), 4),          # C overlaps A
])
def test_ladder_rejects_malformed_requests_on_the_host(g, args, step):
    assert g.gemm_f32_ladder(*args, step=step) == g.GEMM_F32_EINVAL
    assert g.gemm_f32_last_launches() == 0


# (trans_a, trans_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode)
GOOD = (0, 0, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 0.0, FAKE_C, 4, 0)


def _with(**kw):
    names = ["ta", "tb", "M", "N", "K", "alpha", "A", "lda", "B", "ldb", "beta", "C", "ldc", "mode"]
    args = dict(zip(names, GOOD))
    args.update(kw)
    return tuple(args[n] for n in names)


@pytest.mark.parametrize("args", [
    _with(ta=2),                              # trans flag not 0/1
    _with(tb=-1),
    _with(M=-1),
    _with(lda=3),                             # lda < K
    _with(ta=1, M=6, lda=5),                  # stored K x M needs lda >= M
    _with(ldb=3),                             # ldb < N
    _with(tb=1, K=6, ldb=5),                  # stored N x K needs ldb >= K
    _with(ldc=3),                             # ldc < N
    _with(alpha=float("nan")),
    _with(beta=float("inf")),
    _with(mode=9),
    _with(C=0),
    _with(A=0),
    _with(B=FAKE_B + 2),                      # misaligned
    _with(C=FAKE_A + 4 * 4 * 3),              # C window starts inside A's last row
    _with(ldc=64, C=FAKE_B - 64 * 4 * 3),     # strided C window reaches into B
])
def test_general_rejects_malformed_requests_on_the_host(g, args):
    assert g.gemm_f32_general(*args) == g.GEMM_F32_EINVAL
    assert g.gemm_f32_last_launches() == 0


@pytest.mark.parametrize("args,mode", [
    ((FAKE_A, FAKE_B, FAKE_C, 4, 4, 4), 5),              # unknown mode
    ((FAKE_A, FAKE_B, FAKE_C, 4, -4, 4), 0),             # negative N
    ((FAKE_A, FAKE_B, 0, 4, 4, 4), 0),                   # null C
    ((FAKE_A, FAKE_B, FAKE_A + 4, 4, 4, 4), 0),          # C overlaps A
])
def test_host_buffers_reject_malformed_requests(g, args, mode):
    assert g.gemm_f32_host(*args, mode=mode) == g.GEMM_F32_EINVAL
    assert g.gemm_f32_last_launches() == 0


def test_general_alpha_zero_needs_no_operands(g):
    # alpha == 0: A and B are not used, so they may be null; no GPU here
    rc = g.gemm_f32_general(*_with(alpha=0.0, A=0, B=0))
    assert rc == g.GEMM_F32_EDEVICE


def test_empty_outputs_are_a_no_op(g):
    # M == 0 or N == 0: nothing to write, no CUDA call, success
    assert g.gemm_f32_ex(FAKE_A, FAKE_B, FAKE_C, 0, 5, 5) == g.GEMM_F32_OK
    assert g.gemm_f32_last_kernel() == "none"
    assert g.gemm_f32_ex(FAKE_A, FAKE_B, FAKE_C, 5, 0, 5) == g.GEMM_F32_OK
    assert g.gemm_f32_ex(0, 0, 0, 0, 0, 0) == g.GEMM_F32_OK
    assert g.gemm_f32_last_launches() == 0
    for step in range(5):
        assert g.gemm_f32_ladder(FAKE_A, FAKE_B, FAKE_C, 0, 5, 5, step) == g.GEMM_F32_OK
    assert g.gemm_f32_general(*_with(M=0)) == g.GEMM_F32_OK
    assert g.gemm_f32_last_kernel() == "none"


def test_no_gpu_is_reported_as_unsupported_device(g):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = g.gemm_f32_ex(FAKE_A, FAKE_B, FAKE_C, 4, 4, 4)
    assert rc == g.GEMM_F32_EDEVICE
