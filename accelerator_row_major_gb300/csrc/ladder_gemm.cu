// The pages' optimisation ladder for the FP32 GEMM, rebuilt for sm_103a so
// that its steps can be timed on this GPU beside the library's kernels.
// These are teaching kernels, not the product path: gemm_f32() never
// launches them.
//
// Every step computes C[i][j] = sum_k A[i][k] * B[k][j] (row-major, fp32
// fused multiply-adds in ascending k) and differs from the one before by one
// idea ("LeetGPU problem 2: matrix multiplication", yekq.top, sections
// v0 .. v4 and "benchmark summary"):
//   v0  one thread per output; threadIdx.x walks the rows of C, so a warp's
//       B and C accesses are a column apart (not coalesced);
//   v1  the same with threadIdx.x along the columns (coalesced B and C);
//   v2  16 x 16 shared-memory tiles of A and B per K phase, zero-filled past
//       the edges, a barrier after the loads and one after the use;
//   v3  1-D register coarsening: 64 x 64 block tiles, K phases of 16, and
//       each thread keeps 4 consecutive outputs of one row (one A value from
//       shared memory meets 4 B values per k);
//   v4  2-D register coarsening: each thread keeps a 4 x 4 block of outputs
//       (4 A and 4 B values per k feed 16 multiply-adds).
// The pages leave the block shapes of v2 .. v4 open apart from the 4- and
// 4 x 4-output thread tiles; the readings here are 16 x 16 threads (v0 ..
// v2, v4) and 16 x 64 threads (v3), with 64 x 64 x 16 block tiles for v3
// and v4.  Edges are guarded as on the pages: out-of-range loads read zero,
// out-of-range outputs are not written, and no thread returns before the
// last barrier.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"
#include "launch.h"

namespace gemm_f32_impl {
using namespace gemm_f32_dev;

namespace {

// Element loads and stores by index.  The checked build tests each index
// against its matrix's extent (A: M x K, B: K x N, C: M x N); the default
// build reads and writes as written.
__device__ __forceinline__ float ld_a(const float* __restrict__ A, size_t i, int M, int K,
                                     unsigned* err) {
  return GEMM_IN_EXTENT(i, static_cast<size_t>(M) * K, err, kSiteBoundsA) ? A[i] : 0.0f;
}
__device__ __forceinline__ float ld_b(const float* __restrict__ B, size_t i, int K, int N,
                                     unsigned* err) {
  return GEMM_IN_EXTENT(i, static_cast<size_t>(K) * N, err, kSiteBoundsB) ? B[i] : 0.0f;
}
__device__ __forceinline__ void st_c(float* __restrict__ C, size_t i, float v, int M, int N,
                                     unsigned* err) {
  if (GEMM_IN_EXTENT(i, static_cast<size_t>(M) * N, err, kSiteBoundsC)) C[i] = v;
}

constexpr int kTile = 16;                  // v0 .. v2 block edge
constexpr int kBM = 64, kBN = 64, kBK = 16;  // v3, v4 block tile
constexpr int kTN3 = 4;                    // v3 outputs per thread (one row)
constexpr int kTM4 = 4, kTN4 = 4;          // v4 outputs per thread

// v0: x -> row, y -> column.
__global__ void ladder_v0(const float* __restrict__ A, const float* __restrict__ B,
                          float* __restrict__ C, int M, int N, int K, unsigned* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int j = blockIdx.y * blockDim.y + threadIdx.y;
  if (i >= M || j >= N) return;   // no barrier in this kernel
  const size_t a0 = static_cast<size_t>(i) * K;
  float acc = 0.0f;
  for (int k = 0; k < K; ++k)
    acc = fmaf(ld_a(A, a0 + k, M, K, err), ld_b(B, static_cast<size_t>(k) * N + j, K, N, err), acc);
  st_c(C, static_cast<size_t>(i) * N + j, acc, M, N, err);
}

// v1: x -> column, y -> row.
__global__ void ladder_v1(const float* __restrict__ A, const float* __restrict__ B,
                          float* __restrict__ C, int M, int N, int K, unsigned* err) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y * blockDim.y + threadIdx.y;
  if (i >= M || j >= N) return;
  const size_t a0 = static_cast<size_t>(i) * K;
  float acc = 0.0f;
  for (int k = 0; k < K; ++k)
    acc = fmaf(ld_a(A, a0 + k, M, K, err), ld_b(B, static_cast<size_t>(k) * N + j, K, N, err), acc);
  st_c(C, static_cast<size_t>(i) * N + j, acc, M, N, err);
}

// v2: shared-memory tiles.  Thread (tx, ty) loads A[i][k0 + tx] and
// B[k0 + ty][j] and owns C[i][j], i = 16 by + ty, j = 16 bx + tx.
__global__ void ladder_v2(const float* __restrict__ A, const float* __restrict__ B,
                          float* __restrict__ C, int M, int N, int K, unsigned* err) {
  __shared__ float as[kTile][kTile];
  __shared__ float bs[kTile][kTile];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.y * kTile + ty;
  const int j = blockIdx.x * kTile + tx;
  float acc = 0.0f;
  for (int k0 = 0; k0 < K; k0 += kTile) {
    as[ty][tx] = (i < M && k0 + tx < K) ? ld_a(A, static_cast<size_t>(i) * K + k0 + tx, M, K, err)
                                        : 0.0f;
    bs[ty][tx] = (k0 + ty < K && j < N) ? ld_b(B, static_cast<size_t>(k0 + ty) * N + j, K, N, err)
                                        : 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kTile; ++k) acc = fmaf(as[ty][k], bs[k][tx], acc);
    __syncthreads();
  }
  if (i < M && j < N) st_c(C, static_cast<size_t>(i) * N + j, acc, M, N, err);
}

// Block-cooperative zero-filled copy of the A tile [kBM][kBK] at (m0, k0)
// and the B tile [kBK][kBN] at (k0, n0); `tid` of `nthreads`.
__device__ __forceinline__ void load_tiles(const float* __restrict__ A,
                                           const float* __restrict__ B, float (*as)[kBK],
                                           float (*bs)[kBN], int M, int N, int K, int m0,
                                           int n0, int k0, int tid, int nthreads, unsigned* err) {
  for (int e = tid; e < kBM * kBK; e += nthreads) {
    const int r = e / kBK, c = e % kBK;   // c fastest: a warp reads along a row of A
    as[r][c] = (m0 + r < M && k0 + c < K)
                   ? ld_a(A, static_cast<size_t>(m0 + r) * K + k0 + c, M, K, err)
                   : 0.0f;
  }
  for (int e = tid; e < kBK * kBN; e += nthreads) {
    const int r = e / kBN, c = e % kBN;   // a warp reads along a row of B
    bs[r][c] = (k0 + r < K && n0 + c < N)
                   ? ld_b(B, static_cast<size_t>(k0 + r) * N + n0 + c, K, N, err)
                   : 0.0f;
  }
}

// v3: block (16, 64); thread (tx, ty) owns C[m0 + ty][n0 + 4 tx .. +3].
__global__ void ladder_v3(const float* __restrict__ A, const float* __restrict__ B,
                          float* __restrict__ C, int M, int N, int K, unsigned* err) {
  __shared__ float as[kBM][kBK];
  __shared__ float bs[kBK][kBN];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * blockDim.x + tx;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  float acc[kTN3] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int k0 = 0; k0 < K; k0 += kBK) {
    load_tiles(A, B, as, bs, M, N, K, m0, n0, k0, tid, blockDim.x * blockDim.y, err);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      const float a = as[ty][k];
#pragma unroll
      for (int q = 0; q < kTN3; ++q) acc[q] = fmaf(a, bs[k][tx * kTN3 + q], acc[q]);
    }
    __syncthreads();
  }
  const int i = m0 + ty;
  if (i < M) {
#pragma unroll
    for (int q = 0; q < kTN3; ++q) {
      const int j = n0 + tx * kTN3 + q;
      if (j < N) st_c(C, static_cast<size_t>(i) * N + j, acc[q], M, N, err);   // each column checked
    }
  }
}

// v4: block (16, 16); thread (tx, ty) owns C[m0 + 4 ty .. +3][n0 + 4 tx .. +3].
__global__ void ladder_v4(const float* __restrict__ A, const float* __restrict__ B,
                          float* __restrict__ C, int M, int N, int K, unsigned* err) {
  __shared__ float as[kBM][kBK];
  __shared__ float bs[kBK][kBN];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * blockDim.x + tx;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  float acc[kTM4][kTN4];
#pragma unroll
  for (int r = 0; r < kTM4; ++r)
#pragma unroll
    for (int q = 0; q < kTN4; ++q) acc[r][q] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += kBK) {
    load_tiles(A, B, as, bs, M, N, K, m0, n0, k0, tid, blockDim.x * blockDim.y, err);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      float a[kTM4], b[kTN4];
#pragma unroll
      for (int r = 0; r < kTM4; ++r) a[r] = as[ty * kTM4 + r][k];
#pragma unroll
      for (int q = 0; q < kTN4; ++q) b[q] = bs[k][tx * kTN4 + q];
#pragma unroll
      for (int r = 0; r < kTM4; ++r)
#pragma unroll
        for (int q = 0; q < kTN4; ++q) acc[r][q] = fmaf(a[r], b[q], acc[r][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < kTM4; ++r) {
    const int i = m0 + ty * kTM4 + r;
#pragma unroll
    for (int q = 0; q < kTN4; ++q) {
      const int j = n0 + tx * kTN4 + q;
      if (i < M && j < N) st_c(C, static_cast<size_t>(i) * N + j, acc[r][q], M, N, err);
    }
  }
}

long ceil_div_l(long a, long b) { return (a + b - 1) / b; }

}  // namespace

int launch_ladder(GemmArgs& g, int step, cudaStream_t stream, int* launches) {
  *launches = 0;
  constexpr long kMaxGridYZ = 65535;
  dim3 grid, block;
  void (*kern)(const float*, const float*, float*, int, int, int, unsigned*) = nullptr;
  switch (step) {
    case 0:
      block = dim3(kTile, kTile);
      if (ceil_div_l(g.N, kTile) > kMaxGridYZ) return GEMM_F32_EINVAL;
      grid = dim3(ceil_div_l(g.M, kTile), ceil_div_l(g.N, kTile));
      kern = ladder_v0;
      g.kernel = "ladder_v0";
      break;
    case 1:
    case 2:
      block = dim3(kTile, kTile);
      if (ceil_div_l(g.M, kTile) > kMaxGridYZ) return GEMM_F32_EINVAL;
      grid = dim3(ceil_div_l(g.N, kTile), ceil_div_l(g.M, kTile));
      kern = step == 1 ? ladder_v1 : ladder_v2;
      g.kernel = step == 1 ? "ladder_v1" : "ladder_v2";
      break;
    case 3:
    case 4:
      block = step == 3 ? dim3(kBN / kTN3, kBM) : dim3(kBN / kTN4, kBM / kTM4);
      if (ceil_div_l(g.M, kBM) > kMaxGridYZ) return GEMM_F32_EINVAL;
      grid = dim3(ceil_div_l(g.N, kBN), ceil_div_l(g.M, kBM));
      kern = step == 3 ? ladder_v3 : ladder_v4;
      g.kernel = step == 3 ? "ladder_v3" : "ladder_v4";
      break;
    default:
      return GEMM_F32_EINVAL;
  }
  kern<<<grid, block, 0, stream>>>(g.A, g.B, g.C, g.M, g.N, g.K, g.err);
  if (cudaGetLastError() != cudaSuccess) return GEMM_F32_ELAUNCH;
  *launches = 1;
  return GEMM_F32_OK;
}

}  // namespace gemm_f32_impl
