// CUDA-core kernel for small products, where launch and pipeline set-up,
// not arithmetic, set the time: measured on GB300 (CUDA-graph replay), the
// tensor-core kernels need about 6 us even for one tile, while this kernel
// does 100 x 37 x 70 in 2 us and 128^3 in 3.6 us.
//
// C[i][j] = sum_k A[i][k] * B[k][j] in fp32 fused multiply-adds, k ascending,
// so the result is within every mode's bound (1e-5 * (|A||B|)_ij).  One
// thread per output; 16 x 16 tiles of A and B pass through shared memory per
// K phase, zero-filled past the edges, with a barrier after the loads and
// one after the use: the shared-memory tiling of "Lesson 10: shared-memory
// tiled GEMM" (hpc.payai.win, section 2) and of the v2 step of "LeetGPU
// problem 2: matrix multiplication" (yekq.top, section v2), which on these
// sizes keeps more SMs busy than any coarser tiling.  No thread leaves before
// the last barrier.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"
#include "launch.h"

namespace gemm_f32_impl {
using namespace gemm_f32_dev;

namespace {

constexpr int kT = 16;

__global__ void __launch_bounds__(kT * kT) small_gemm_kernel(const float* __restrict__ A,
                                                             const float* __restrict__ B,
                                                             float* __restrict__ C, int M, int N,
                                                             int K, unsigned* err) {
  __shared__ float as[kT][kT];
  __shared__ float bs[kT][kT];
  grid_launch_dependents();
  grid_dependency_wait();   // global memory from here on
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.y * kT + ty;
  const int j = blockIdx.x * kT + tx;
  float acc = 0.0f;
  for (int k0 = 0; k0 < K; k0 += kT) {
    const size_t ia = static_cast<size_t>(i) * K + k0 + tx;
    const size_t ib = static_cast<size_t>(k0 + ty) * N + j;
    as[ty][tx] = (i < M && k0 + tx < K &&
                  GEMM_IN_EXTENT(ia, static_cast<size_t>(M) * K, err, kSiteBoundsA))
                     ? __ldg(A + ia)
                     : 0.0f;
    bs[ty][tx] = (k0 + ty < K && j < N &&
                  GEMM_IN_EXTENT(ib, static_cast<size_t>(K) * N, err, kSiteBoundsB))
                     ? __ldg(B + ib)
                     : 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kT; ++k) acc = fmaf(as[ty][k], bs[k][tx], acc);
    __syncthreads();
  }
  if (i < M && j < N &&
      GEMM_IN_EXTENT(static_cast<size_t>(i) * N + j, static_cast<size_t>(M) * N, err, kSiteBoundsC))
    C[static_cast<size_t>(i) * N + j] = acc;
}

}  // namespace

bool small_suits(const GemmArgs& g) {
  return static_cast<long long>(g.M) * g.N * g.K <= kSmallMaxWork && g.K <= kSmallMaxK &&
         (g.M + kT - 1) / kT <= 65535;
}

int launch_small(GemmArgs& g, cudaStream_t stream, int* launches) {
  *launches = 0;
  const dim3 grid((g.N + kT - 1) / kT, (g.M + kT - 1) / kT);
  if (launch_dependent(small_gemm_kernel, grid, dim3(kT, kT), 0, stream, g.A, g.B, g.C, g.M, g.N,
                       g.K, g.err) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  *launches = 1;
  g.kernel = "small_gemm_kernel";
  return GEMM_F32_OK;
}

}  // namespace gemm_f32_impl
