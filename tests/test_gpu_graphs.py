"""CUDA-graph capture of the C-ABI call: after one call of the same shape
and mode on the capturing stream (which sets up the device, configures the
kernel and sizes the split-tail workspace outside the capture), a captured
gemm_f32_ex replays correctly, and replays with new operand values written
into the same buffers give the new products."""
import numpy as np
import pytest

import workloads
from tests._gpu import TOL, assert_close, lib, oracle_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["tc3x", "ffma", "tc1x"])
@pytest.mark.parametrize("shape", [(1024, 512, 1024), (1001, 513, 777), (2304, 256, 2560)])
def test_captured_call_replays(mode, shape):
    import torch
    g = lib()
    M, K, N = shape
    dev = torch.device("cuda:0")
    s = torch.cuda.Stream(dev)
    A = torch.empty((M, K), device=dev)
    B = torch.empty((K, N), device=dev)
    C = torch.empty((M, N), device=dev)

    def call():
        g.check(g.gemm_f32_ex(A, B, C, M, N, K, mode, 0, s))

    with torch.cuda.stream(s):
        call()                       # set-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for seed in (0, 1):
        A_h, B_h = workloads.make_inputs(M, K, N, "uniform", 900 + seed)
        A.copy_(torch.from_numpy(A_h))
        B.copy_(torch.from_numpy(B_h))
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        rc, site = g.gemm_f32_status(s)
        assert rc == 0, site
        Co, absAB = oracle_full(A_h, B_h)
        assert_close(C.cpu().numpy(), Co, absAB, TOL[mode], "graph %s/%s/%d" % (shape, mode, seed))
