"""ctypes binding of libgemm_f32.so: argument marshalling only.

Every computation happens in the library's CUDA kernels.  The library is
loaded on first use; if it is missing, that first call raises ImportError.
There is no fallback.  The environment variable GEMM_F32_LIBRARY, when set,
names the library file to load instead (the tests use it to run on the
bounds-checked debug build, libgemm_f32_checked.so).
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("GEMM_F32_LIBRARY") or os.path.join(_PKG, "libgemm_f32.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "gemm_f32.h")

GEMM_F32_OK = 0
GEMM_F32_EINVAL = -1
GEMM_F32_EDEVICE = -2
GEMM_F32_ELAUNCH = -3
GEMM_F32_ETIMEOUT = -4
GEMM_F32_ESCRATCH = -5
NOALLOC_SCRATCH_BYTES = 32 << 20

MODE_TC3X = 0
MODE_FFMA = 1
MODE_TC1X = 2
MODES = {"tc3x": MODE_TC3X, "ffma": MODE_FFMA, "tc1x": MODE_TC1X}

FLAG_FORCE_STAGED = 0x1
FLAG_TILE64 = 0x10
FLAG_TILE128 = 0x20
FLAG_TILE224 = 0x80
FLAG_TILE256 = 0x40
FLAG_ONE_TILE_PER_CTA = 0x100
FLAG_NO_SPLIT_K = 0x200
FLAG_CTA_PAIR = 0x400
FLAG_SINGLE_CTA = 0x800
FLAG_TEST_DROP_COPY = 0x1000

_ERRORS = {
    GEMM_F32_EINVAL: "invalid argument",
    GEMM_F32_EDEVICE: "unsupported device (needs sm_103, GB300)",
    GEMM_F32_ELAUNCH: "kernel launch refused by the CUDA runtime",
    GEMM_F32_ETIMEOUT: "a bounded device-side wait ran out",
    GEMM_F32_ESCRATCH: "the product needs more scratch than the library's fixed array",
}


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s failed: %s (%d)" % (what, _ERRORS.get(code, "unknown error"), code))
        self.code = code


class UnitRates(ctypes.Structure):
    """gemm_f32_unit_rates_t of include/gemm_f32.h."""
    _fields_ = [("tf32_flop_per_clk_sm", ctypes.c_double),
                ("tf32_pair_flop_per_clk_sm", ctypes.c_double),
                ("ffma_flop_per_clk_sm", ctypes.c_double),
                ("sm_mhz", ctypes.c_double),
                ("num_sms", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("%s is not built (run accelerator_row_major_gb300.build.build())" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci, cu = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
    lib.gemm_f32.argtypes = [vp, vp, vp, ci, ci, ci, vp]
    lib.gemm_f32.restype = ci
    lib.gemm_f32_ex.argtypes = [vp, vp, vp, ci, ci, ci, ci, cu, vp]
    lib.gemm_f32_ex.restype = ci
    lib.gemm_f32_status.argtypes = [vp, ctypes.POINTER(cu)]
    lib.gemm_f32_status.restype = ci
    lib.gemm_f32_last_launches.argtypes = []
    lib.gemm_f32_last_launches.restype = ci
    lib.gemm_f32_noalloc.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
    lib.gemm_f32_noalloc.restype = ci
    cf = ctypes.c_float
    lib.gemm_f32_general.argtypes = [ci, ci, ci, ci, ci, cf, vp, ci, vp, ci, cf, vp, ci, ci, vp]
    lib.gemm_f32_general.restype = ci
    lib.gemm_f32_host.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
    lib.gemm_f32_host.restype = ci
    lib.gemm_f32_ladder.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
    lib.gemm_f32_ladder.restype = ci
    lib.gemm_f32_last_kernel.argtypes = []
    lib.gemm_f32_last_kernel.restype = ctypes.c_char_p
    lib.gemm_f32_release.argtypes = []
    lib.gemm_f32_release.restype = ci
    lib.gemm_f32_version.argtypes = []
    lib.gemm_f32_version.restype = ctypes.c_char_p
    lib.gemm_f32_unit_rates.argtypes = [ctypes.POINTER(UnitRates)]
    lib.gemm_f32_unit_rates.restype = ci
    u64p = ctypes.POINTER(ctypes.c_ulonglong)
    lib.gemm_f32_clock_record.argtypes = [vp, u64p, u64p]
    lib.gemm_f32_clock_record.restype = ci
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once, on first use)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def declared_symbols(header: str = HEADER):
    """Function names declared in include/gemm_f32.h."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_f32\w*)\s*\(", text)))


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x.ctypes.data)          # numpy array (host memory)


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def gemm_f32(A, B, C, M: int, N: int, K: int, stream=None) -> int:
    """C = A * B (row-major, default mode).  A, B, C: device pointers (int)
    or CUDA tensors; stream: int handle, torch.cuda.Stream or None."""
    return lib().gemm_f32(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(stream))


def gemm_f32_ex(A, B, C, M: int, N: int, K: int, mode=MODE_TC3X, flags: int = 0, stream=None) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return lib().gemm_f32_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(mode), int(flags), _stream(stream))


def gemm_f32_noalloc(A, B, C, M: int, N: int, K: int, mode=MODE_TC3X, stream=None) -> int:
    """C = A * B in a tensor mode without any device allocation (scratch from
    a fixed array inside the library); see include/gemm_f32.h."""
    if isinstance(mode, str):
        mode = MODES[mode]
    return lib().gemm_f32_noalloc(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(mode), _stream(stream))


def gemm_f32_general(trans_a: int, trans_b: int, M: int, N: int, K: int, alpha: float, A, lda: int,
                     B, ldb: int, beta: float, C, ldc: int, mode=MODE_TC3X, stream=None) -> int:
    """C = alpha * op(A) * op(B) + beta * C on row-major storage with row
    strides lda, ldb, ldc; trans_a / trans_b select stored transposes (see
    include/gemm_f32.h)."""
    if isinstance(mode, str):
        mode = MODES[mode]
    return lib().gemm_f32_general(int(trans_a), int(trans_b), M, N, K, float(alpha), _ptr(A), lda,
                                  _ptr(B), ldb, float(beta), _ptr(C), ldc, int(mode), _stream(stream))


def gemm_f32_host(A, B, C, M: int, N: int, K: int, mode=MODE_TC3X, stream=None) -> int:
    """C = A * B with A, B, C in host memory (pinned torch tensors, numpy
    arrays or addresses); copies and product are queued on the library's
    streams, and `stream` waits for C (see include/gemm_f32.h)."""
    if isinstance(mode, str):
        mode = MODES[mode]
    return lib().gemm_f32_host(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(mode), _stream(stream))


LADDER_STEPS = (0, 1, 2, 3, 4)


def gemm_f32_ladder(A, B, C, M: int, N: int, K: int, step: int, stream=None) -> int:
    """C = A * B with the pages' teaching kernel v<step> (0 .. 4); see
    include/gemm_f32.h.  Not the product path."""
    return lib().gemm_f32_ladder(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(step), _stream(stream))


def gemm_f32_status(stream=None):
    """(code, site): synchronises the stream, reads and clears the error word."""
    site = ctypes.c_uint(0)
    rc = lib().gemm_f32_status(_stream(stream), ctypes.byref(site))
    return rc, site.value


def gemm_f32_clock_record(stream=None):
    """(sm_cycles, ns): the device's running sums of CTA 0's lifetime over the
    persistent kernels' launches (synchronises the stream); the difference of
    two readings gives the SM clock in between, cycles / ns GHz.  Raises
    GemmError on failure."""
    cycles, ns = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    check(lib().gemm_f32_clock_record(_stream(stream), ctypes.byref(cycles), ctypes.byref(ns)),
          "gemm_f32_clock_record")
    return cycles.value, ns.value


def gemm_f32_last_launches() -> int:
    return lib().gemm_f32_last_launches()


def gemm_f32_last_kernel() -> str:
    """Kernel the last successful call on this thread launched."""
    return lib().gemm_f32_last_kernel().decode()


def gemm_f32_release() -> int:
    """Frees the current device's workspaces (synchronises the device)."""
    return lib().gemm_f32_release()


def gemm_f32_unit_rates() -> dict:
    """Per-SM FLOP per clock of the tf32 tensor core (one SM, SM pairs) and
    of the fp32 FFMA pipe, measured on the current device, with the SM clock
    seen meanwhile; raises GemmError on failure."""
    r = UnitRates()
    check(lib().gemm_f32_unit_rates(ctypes.byref(r)), "gemm_f32_unit_rates")
    return {name: getattr(r, name) for name, _ in UnitRates._fields_}


def gemm_f32_version() -> str:
    return lib().gemm_f32_version().decode()


def check(rc: int, what: str = "gemm_f32") -> None:
    if rc != GEMM_F32_OK:
        raise GemmError(rc, what)
