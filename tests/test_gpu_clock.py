"""gemm_f32_clock_record: the SM clock the persistent kernels ran at, from
clock64 and %globaltimer read by CTA 0 of each launch."""
import pytest

from tests._gpu import lib

pytestmark = pytest.mark.gpu

FLAG_CTA_PAIR = 0x400

# (M, K, N), mode, flags, the kernel that runs
CASES = [((4096, 1024, 4096), "tc3x", FLAG_CTA_PAIR, "tc_pair_kernel"),
         ((4096, 1024, 4096), "tc1x", FLAG_CTA_PAIR, "tc_pair_kernel"),
         ((2048, 1024, 2048), "ffma", 0, "ffma_gemm_kernel")]


@pytest.mark.parametrize("shape,mode,flags,kernel", CASES, ids=["%s-%s" % (c[3], c[1]) for c in CASES])
def test_clock_record_gives_the_sm_clock(shape, mode, flags, kernel):
    import torch

    g = lib()
    M, K, N = shape
    dev = torch.device("cuda:0")
    A = torch.randn(M, K, device=dev)
    B = torch.randn(K, N, device=dev)
    C = torch.empty(M, N, device=dev)
    stream = torch.cuda.current_stream()
    g.check(g.gemm_f32_ex(A, B, C, M, N, K, mode, flags, stream))
    assert g.gemm_f32_last_kernel() == kernel
    c0, n0 = g.gemm_f32_clock_record(stream)
    for _ in range(5):
        g.check(g.gemm_f32_ex(A, B, C, M, N, K, mode, flags, stream))
    c1, n1 = g.gemm_f32_clock_record(stream)
    assert c1 > c0 and n1 > n0
    ghz = (c1 - c0) / (n1 - n0)
    # SM clocks per nanosecond: between a deeply throttled part and the
    # 2.07 GHz maximum (with room for the timer's granularity)
    assert 0.3 < ghz < 2.3, ghz
    assert g.gemm_f32_status(stream) == (g.GEMM_F32_OK, 0)


@pytest.mark.parametrize("shape,kernel", [((100, 70, 37), "small_gemm_kernel"),
                                          ((65536, 256, 64), "tc_gemm_kernel")])
def test_other_kernels_leave_the_record_alone(shape, kernel):
    # the 16 x 16 tiled kernel is not a persistent grid, and the single-SM
    # tensor kernel keeps its prologue and exit free of the record
    import torch

    g = lib()
    M, K, N = shape
    dev = torch.device("cuda:0")
    A = torch.randn(M, K, device=dev)
    B = torch.randn(K, N, device=dev)
    C = torch.empty(M, N, device=dev)
    stream = torch.cuda.current_stream()
    before = g.gemm_f32_clock_record(stream)
    g.check(g.gemm_f32_ex(A, B, C, M, N, K, "tc3x", 0, stream))
    assert g.gemm_f32_last_kernel() == kernel
    assert g.gemm_f32_clock_record(stream) == before
