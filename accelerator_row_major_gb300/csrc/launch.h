// Private interface between the C-ABI front end (gemm_f32.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

namespace gemm_f32_impl {

// Launches `kernel` with programmatic stream serialization: it may begin as
// the previous kernel on `stream` lets its dependents start, and waits
// (griddepcontrol.wait, device_common.cuh) before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct GemmArgs {
  const float* A;
  const float* B;
  float* C;
  int M, N, K;          // K >= 1, M >= 1, N >= 1 here (the front end handles the rest)
  unsigned* err;        // device error word of the current device
  int num_sms;          // multiprocessors of the current device
  int device;           // current device ordinal
  unsigned flags;       // GEMM_F32_FLAG_* bits
  const char* kernel = "none";   // set by the launcher: the kernel it launched
  // General form C = alpha op(A) op(B) + beta C (row-major storage).  The
  // plain product has lda = K, ldb = N, ldc = N, no transposes, alpha = 1,
  // beta = 0 and scale = 0.
  int lda = 0, ldb = 0, ldc = 0;   // row strides (elements) of the stored A, B, C
  int trans_a = 0;                 // 1: A is stored K x M and op(A) = its transpose
  int trans_b = 0;                 // 1: B is stored N x K and op(B) = its transpose
  float alpha = 1.0f, beta = 0.0f;
  int scale = 0;                   // 1 when alpha != 1 or beta != 0
};

// The plain product C = A * B on dense row-major storage (what gemm_f32 and
// gemm_f32_ex compute): the kernels have separate code for it.
inline bool plain_form(const GemmArgs& g) {
  return !g.trans_a && !g.trans_b && g.lda == g.K && g.ldb == g.N && g.ldc == g.N && !g.scale;
}

// Whether the operands can be read by TMA tiles: untransposed, row strides a
// multiple of 16 bytes, 16-byte aligned bases.
inline bool tma_addressable(const GemmArgs& g) {
  return !g.trans_a && !g.trans_b && g.lda % 4 == 0 && g.ldb % 4 == 0 &&
         reinterpret_cast<uintptr_t>(g.A) % 16 == 0 && reinterpret_cast<uintptr_t>(g.B) % 16 == 0;
}

// The library's workspace for `stream` on `device` (one per device and
// stream), grown to at least `bytes` with cudaMalloc when needed (which
// synchronises the device) and zeroed when allocated.  Its split-tail
// counters stay valid from call to call, even after a kernel gave up on a
// bounded wait (device_common.cuh).  Returns nullptr if the memory cannot be
// had; the caller then does without.
void* acquire_workspace(int device, cudaStream_t stream, size_t bytes);

// Tensor-core path (tcgen05.mma kind::tf32).  nprod = 3 (split hi/lo, three
// products) or 1 (operands rounded to TF32, one product).  Returns 0 or a
// negative GEMM_F32_E* code.  *launches receives the kernels launched.
int launch_tc(GemmArgs& g, int nprod, cudaStream_t stream, int* launches);

// Tensor-core path on CTA pairs (256 x 256 tiles, cta_group::2), and whether
// a problem in a mode of `nprod` products should take it (a wave of pair
// tiles and, on the TMA path, a deep enough K; or forced by flags).
bool tc_pair_suits(const GemmArgs& g, int nprod);
int launch_tc_pair(GemmArgs& g, int nprod, cudaStream_t stream, int* launches);

// Tensor-core path on the single-CTA kernel whose split-tail scratch is the
// fixed array inside the library at `scratch` (no allocation, no operand
// packing).  Returns GEMM_F32_ESCRATCH if the product would need more than
// GEMM_F32_NOALLOC_SCRATCH_BYTES, GEMM_F32_EDEVICE if `scratch` is null.
// fixed_scratch_address() gives the array's device address on the current
// device (nullptr if the runtime cannot give it).
int launch_tc_fixed_scratch(GemmArgs& g, int nprod, void* scratch, cudaStream_t stream,
                            int* launches);
void* fixed_scratch_address();

// 2-D fp32 tensor map of a row-major [rows x cols] matrix with row stride ld
// (elements) and box [box_rows x box_cols]; out-of-bounds reads give zero.
// False when the driver entry point or the encoding fails.
bool tma_encode_2d(CUtensorMap* map, const float* ptr, int rows, int cols, int ld, int box_cols,
                   int box_rows, CUtensorMapSwizzle swz);

// CUDA-core FFMA path.
int launch_ffma(GemmArgs& g, cudaStream_t stream, int* launches);

// Operand repacking for the TMA path (pack.cu).  pack_operand writes op(X),
// rows x cols (X itself, or the transpose of X stored cols x rows), row-major
// with row stride ld_dst.  pack_for_tma rewrites g's A and B (pointers,
// strides, transpose flags) to packed copies in the stream's pack buffer
// when TMA cannot read them and the product has at least kPackMinWork
// multiply-adds; it packs nothing otherwise (or without memory) and counts
// its kernels in *launches.
constexpr long long kPackMinWork = 1LL << 27;
int pack_operand(const float* src, int rows, int cols, int ld_src, bool transposed, float* dst,
                 int ld_dst, int num_sms, unsigned* err, cudaStream_t stream);
int pack_for_tma(GemmArgs& g, cudaStream_t stream, int* launches);

// The library's pack buffer for `stream` on `device`, grown to at least
// `bytes` (1 MiB granules, cudaMalloc, which synchronises the device when it
// grows); nullptr when the memory cannot be had.  Freed by gemm_f32_release.
void* acquire_pack_buffer(int device, cudaStream_t stream, size_t bytes);

// Small products (at most kSmallMaxWork multiply-adds, K <= kSmallMaxK) on a
// latency-lean CUDA-core kernel, in every mode: below these sizes launch and
// pipeline set-up dominate the tensor-core kernels' time.
constexpr long long kSmallMaxWork = 1LL << 23;
constexpr int kSmallMaxK = 256;
bool small_suits(const GemmArgs& g);
int launch_small(GemmArgs& g, cudaStream_t stream, int* launches);

// The pages' ladder kernels v0 .. v4 (step), for timing and teaching.
int launch_ladder(GemmArgs& g, int step, cudaStream_t stream, int* launches);

}  // namespace gemm_f32_impl
