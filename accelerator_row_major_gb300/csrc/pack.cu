// Operand repacking for the tensor-core path.  TMA reads a matrix only when
// its base is 16-byte aligned and its row stride is a multiple of 16 bytes,
// and only in the layout stored; an operand with an odd stride, or stored
// transposed (the general form), otherwise goes through the per-thread
// staged loads, which run at about half the TMA path's speed on large
// problems.  Copying it once into an aligned row-major buffer costs 8 bytes
// of HBM traffic per element and pays for itself above a few hundred rows
// and columns (the threshold sits in the launcher).
//
// pack_rows_kernel: dst[r][c] = src[r][c] (row strides ld_src, ld_dst); one
// launch copies one or two such matrices (A and B of a product: one launch
// instead of two, which is what a ragged mid-sized product notices).
// pack_transpose_kernel: dst[r][c] = src[c][r], through 32 x 33 shared-memory
// tiles so that both the reads and the writes are coalesced.
// Columns c >= cols of dst are left as they are: TMA reads them as out of
// bounds (zero) because the tensor map's width is `cols`.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"
#include "launch.h"

namespace gemm_f32_impl {
using namespace gemm_f32_dev;

namespace {

constexpr int kTile = 32;

struct RowCopy {
  const float* src;
  float* dst;
  long long ld_src, ld_dst;
  int rows, cols;
};

// Extents (elements) of one copy's source and destination windows, for the
// checked build.
__device__ __forceinline__ size_t src_extent(const RowCopy& m) {
  return stored_extent(m.rows, m.cols, m.ld_src);
}
__device__ __forceinline__ size_t dst_extent(const RowCopy& m) {
  return stored_extent(m.rows, m.cols, m.ld_dst);
}

__global__ void pack_rows_kernel(RowCopy x, RowCopy y, unsigned* err) {
  grid_launch_dependents();   // the product after this copy may start its set-up
  grid_dependency_wait();
  const long long nx = static_cast<long long>(x.rows) * x.cols;
  const long long total = nx + static_cast<long long>(y.rows) * y.cols;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool in_x = t < nx;
    const long long e = in_x ? t : t - nx;
    const int cols = in_x ? x.cols : y.cols;
    const long long r = e / cols, c = e % cols;
    const float* const src = in_x ? x.src : y.src;
    float* const dst = in_x ? x.dst : y.dst;
    const long long is = r * (in_x ? x.ld_src : y.ld_src) + c;
    const long long id = r * (in_x ? x.ld_dst : y.ld_dst) + c;
    if (GEMM_IN_EXTENT(is, src_extent(in_x ? x : y), err, kSiteBoundsPack) &&
        GEMM_IN_EXTENT(id, dst_extent(in_x ? x : y), err, kSiteBoundsPack))
      dst[id] = __ldg(src + is);
  }
}

int launch_rows(const RowCopy& x, const RowCopy& y, int num_sms, unsigned* err,
                cudaStream_t stream) {
  const long long total = static_cast<long long>(x.rows) * x.cols + static_cast<long long>(y.rows) * y.cols;
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
  if (launch_dependent(pack_rows_kernel, dim3(grid), dim3(256), 0, stream, x, y, err) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  return GEMM_F32_OK;
}

RowCopy row_copy(const float* src, int rows, int cols, int ld_src, float* dst, int ld_dst) {
  RowCopy m;
  m.src = src;
  m.dst = dst;
  m.ld_src = ld_src;
  m.ld_dst = ld_dst;
  m.rows = rows;
  m.cols = cols;
  return m;
}

// block (32, 8): tile (blockIdx.y, blockIdx.x) of dst, rows r0.., cols c0..
__global__ void pack_transpose_kernel(const float* __restrict__ src, int rows, int cols,
                                      long long ld_src, float* __restrict__ dst, long long ld_dst,
                                      unsigned* err) {
  __shared__ float tile[kTile][kTile + 1];
  grid_launch_dependents();
  grid_dependency_wait();
  const int r0 = blockIdx.y * kTile, c0 = blockIdx.x * kTile;
  // read src rows c0.. (dst columns), lanes along src columns (dst rows)
  for (int y = threadIdx.y; y < kTile; y += blockDim.y) {
    const int c = c0 + y, r = r0 + threadIdx.x;
    if (c < cols && r < rows &&
        GEMM_IN_EXTENT(static_cast<long long>(c) * ld_src + r, stored_extent(cols, rows, ld_src), err,
                       kSiteBoundsPack))
      tile[y][threadIdx.x] = __ldg(src + static_cast<long long>(c) * ld_src + r);
  }
  __syncthreads();
  for (int y = threadIdx.y; y < kTile; y += blockDim.y) {
    const int r = r0 + y, c = c0 + threadIdx.x;
    if (r < rows && c < cols &&
        GEMM_IN_EXTENT(static_cast<long long>(r) * ld_dst + c, stored_extent(rows, cols, ld_dst), err,
                       kSiteBoundsPack))
      dst[static_cast<long long>(r) * ld_dst + c] = tile[threadIdx.x][y];
  }
}

}  // namespace

int pack_operand(const float* src, int rows, int cols, int ld_src, bool transposed, float* dst,
                 int ld_dst, int num_sms, unsigned* err, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return GEMM_F32_OK;
  if (!transposed) {
    return launch_rows(row_copy(src, rows, cols, ld_src, dst, ld_dst),
                       row_copy(src, 0, 1, ld_src, dst, ld_dst), num_sms, err, stream);
  } else {
    const long long gy = (rows + kTile - 1) / kTile;
    if (gy > 65535) return GEMM_F32_EINVAL;
    const dim3 grid((cols + kTile - 1) / kTile, static_cast<unsigned>(gy));
    if (launch_dependent(pack_transpose_kernel, grid, dim3(kTile, 8), 0, stream, src, rows, cols,
                         static_cast<long long>(ld_src), dst, static_cast<long long>(ld_dst),
                         err) != cudaSuccess) {
      (void)cudaGetLastError();
      return GEMM_F32_ELAUNCH;
    }
  }
  if (cudaGetLastError() != cudaSuccess) return GEMM_F32_ELAUNCH;
  return GEMM_F32_OK;
}

int pack_for_tma(GemmArgs& g, cudaStream_t stream, int* launches) {
  if ((g.flags & GEMM_F32_FLAG_FORCE_STAGED) || tma_addressable(g)) return GEMM_F32_OK;
  if (static_cast<long long>(g.M) * g.N * g.K < kPackMinWork) return GEMM_F32_OK;
  const bool pack_a = g.trans_a || g.lda % 4 != 0 || reinterpret_cast<uintptr_t>(g.A) % 16 != 0;
  const bool pack_b = g.trans_b || g.ldb % 4 != 0 || reinterpret_cast<uintptr_t>(g.B) % 16 != 0;
  const int lda = (g.K + 3) & ~3, ldb = (g.N + 3) & ~3;
  const size_t a_bytes =
      pack_a ? (static_cast<size_t>(g.M) * lda * sizeof(float) + 255) & ~static_cast<size_t>(255) : 0;
  const size_t b_bytes = pack_b ? static_cast<size_t>(g.K) * ldb * sizeof(float) : 0;
  float* const buf = static_cast<float*>(acquire_pack_buffer(g.device, stream, a_bytes + b_bytes));
  if (!buf) return GEMM_F32_OK;   // no memory for copies: the staged loads serve
  float* const b_dst = buf + a_bytes / sizeof(float);
  if (pack_a && pack_b && !g.trans_a && !g.trans_b) {
    // both plain row copies: one launch
    const int rc = launch_rows(row_copy(g.A, g.M, g.K, g.lda, buf, lda),
                               row_copy(g.B, g.K, g.N, g.ldb, b_dst, ldb), g.num_sms, g.err,
                               stream);
    if (rc != GEMM_F32_OK) return rc;
    g.A = buf;
    g.lda = lda;
    g.B = b_dst;
    g.ldb = ldb;
    ++*launches;
    return GEMM_F32_OK;
  }
  if (pack_a) {
    const int rc =
        pack_operand(g.A, g.M, g.K, g.lda, g.trans_a != 0, buf, lda, g.num_sms, g.err, stream);
    if (rc != GEMM_F32_OK) return rc;
    g.A = buf;
    g.lda = lda;
    g.trans_a = 0;
    ++*launches;
  }
  if (pack_b) {
    const int rc =
        pack_operand(g.B, g.K, g.N, g.ldb, g.trans_b != 0, b_dst, ldb, g.num_sms, g.err, stream);
    if (rc != GEMM_F32_OK) return rc;
    g.B = b_dst;
    g.ldb = ldb;
    g.trans_b = 0;
    ++*launches;
  }
  return GEMM_F32_OK;
}

}  // namespace gemm_f32_impl
