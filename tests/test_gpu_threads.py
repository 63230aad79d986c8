"""Host threads calling the library at the same time, each on its own
stream (ctypes releases the interpreter lock, so the calls overlap in the
library): per-device set-up, per-stream workspaces and copy buffers, the
thread-local last-call record and gemm_f32_host's shared slots must keep
every result right."""
import threading

import numpy as np
import pytest

import workloads
from tests._gpu import TOL, assert_close, lib, oracle_full

pytestmark = pytest.mark.gpu

# shapes covering the small kernel, the split tail, the pair kernel and
# operand copies (odd strides)
SHAPES = [(100, 37, 70), (1024, 512, 1024), (2304, 256, 2560), (1027, 1029, 1031), (512, 8192, 384)]


def test_threads_on_their_own_streams():
    import torch
    g = lib()
    dev = torch.device("cuda:0")
    cases = []
    for t, (M, K, N) in enumerate(SHAPES):
        A, B = workloads.make_inputs(M, K, N, "uniform", 300 + t)
        cases.append((A, B) + oracle_full(A, B))
    errors = []

    def worker(tid):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(dev)
            mode = ("tc3x", "ffma", "tc1x")[tid % 3]
            for rep in range(3):
                for idx in range(len(SHAPES)):
                    A, B, Co, absAB = cases[(idx + tid) % len(SHAPES)]
                    M, K = A.shape
                    N = B.shape[1]
                    a = torch.from_numpy(A).to(dev)
                    b = torch.from_numpy(B).to(dev)
                    c = torch.full((M, N), float("nan"), device=dev)
                    torch.cuda.synchronize(dev)
                    rc = g.gemm_f32_ex(a, b, c, M, N, K, mode, 0, s)
                    assert rc == 0, rc
                    kernel = g.gemm_f32_last_kernel()   # this thread's own call
                    assert kernel != "none"
                    st, site = g.gemm_f32_status(s)
                    assert st == 0, site
                    assert_close(c.cpu().numpy(), Co, absAB, TOL[mode],
                                 "thread %d %dx%dx%d %s %s" % (tid, M, K, N, mode, kernel))
        except Exception as e:   # collected and re-raised in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(6)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if errors:
        raise errors[0]


def test_threads_sharing_the_host_buffer_path():
    import torch
    g = lib()
    dev = torch.device("cuda:0")
    errors = []

    def worker(tid):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(dev)
            for rep in range(4):
                M, K, N = SHAPES[(tid + rep) % len(SHAPES)]
                A, B = workloads.make_inputs(M, K, N, "int8", 40 + tid)
                a = torch.from_numpy(A).pin_memory()
                b = torch.from_numpy(B).pin_memory()
                c = torch.full((M, N), float("nan")).pin_memory()
                rc = g.gemm_f32_host(a, b, c, M, N, K, "tc3x", s)
                assert rc == 0, rc
                st, site = g.gemm_f32_status(s)
                assert st == 0, site
                want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
                assert np.array_equal(c.numpy(), want), "thread %d shape %s" % (tid, (M, K, N))
        except Exception as e:
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if errors:
        raise errors[0]
