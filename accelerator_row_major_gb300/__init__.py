"""Row-major FP32 GEMM for GB300 (sm_103a) behind a C ABI.

The library ``libgemm_f32.so`` (built by ``accelerator_row_major_gb300.build``)
computes C = A * B for row-major fp32 matrices on the GPU.  This package is
its thin Python binding; PyTorch is used only to hold device memory and
streams.

    import torch, accelerator_row_major_gb300 as g
    C = g.matmul(A, B)                     # A, B: contiguous fp32 CUDA tensors
    g.gemm_f32(A, B, C, M, N, K, stream)   # the C-ABI call, same arguments
"""
from ._binding import (FLAG_CTA_PAIR, FLAG_FORCE_STAGED, FLAG_SINGLE_CTA, FLAG_TILE64, FLAG_TILE128, FLAG_TILE256,  # noqa: F401
                       FLAG_NO_SPLIT_K, FLAG_ONE_TILE_PER_CTA, FLAG_TEST_DROP_COPY, GEMM_F32_EDEVICE, GEMM_F32_EINVAL,
                       GEMM_F32_ELAUNCH, GEMM_F32_ESCRATCH, GEMM_F32_ETIMEOUT, GEMM_F32_OK, LIB_PATH, MODE_FFMA,
                       MODE_TC1X, MODE_TC3X, MODES, GemmError, check, declared_symbols,
                       gemm_f32, gemm_f32_ex, gemm_f32_general, gemm_f32_host, gemm_f32_ladder, gemm_f32_last_kernel, gemm_f32_last_launches,
                       gemm_f32_noalloc, LADDER_STEPS,
                       gemm_f32_release, NOALLOC_SCRATCH_BYTES,
                       gemm_f32_clock_record, gemm_f32_status, gemm_f32_unit_rates,
                       gemm_f32_version)


def matmul(A, B, out=None, mode="tc3x", flags: int = 0, stream=None):
    """C = A @ B through the C ABI for contiguous 2-D fp32 CUDA tensors.

    Allocates C with torch when ``out`` is None; raises GemmError on a
    non-zero return code."""
    import torch

    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shapes %s and %s do not chain" % (tuple(A.shape), tuple(B.shape)))
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous float32 CUDA tensor" % name)
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif out.shape != (M, N) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of shape (%d, %d)" % (M, N))
    if stream is None:
        stream = torch.cuda.current_stream(A.device)
    check(gemm_f32_ex(A, B, out, M, N, K, mode, flags, stream))
    return out
