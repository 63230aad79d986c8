// Private interface between the C-ABI front end (gemm_f32.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

namespace gemm_f32_impl {

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
};

// The library's workspace for `stream` on `device` (one per device and
// stream), grown to at least `bytes` with cudaMalloc when needed (which
// synchronises the device) and zeroed when allocated.  *must_clear is set
// when the caller must re-zero the split-tail counters before using it (a
// kernel on this device gave up on a bounded wait since it was last used).
// Returns nullptr if the memory cannot be had; the caller then does without.
void* acquire_workspace(int device, cudaStream_t stream, size_t bytes, int* must_clear);

// Tensor-core path (tcgen05.mma kind::tf32).  nprod = 3 (split hi/lo, three
// products) or 1 (operands rounded to TF32, one product).  Returns 0 or a
// negative GEMM_F32_E* code.  *launches receives the kernels launched.
int launch_tc(GemmArgs& g, int nprod, cudaStream_t stream, int* launches);

// Tensor-core path on CTA pairs (256 x 256 tiles, cta_group::2), and whether
// a problem should take it (large M and N, or forced by flags).
bool tc_pair_suits(const GemmArgs& g);
int launch_tc_pair(GemmArgs& g, int nprod, cudaStream_t stream, int* launches);

// Tensor-core path whose split-tail scratch comes from a fixed array inside
// the library (no allocation).  Returns GEMM_F32_ESCRATCH if the product
// would need more than GEMM_F32_NOALLOC_SCRATCH_BYTES.
int launch_tc_fixed_scratch(GemmArgs& g, int nprod, cudaStream_t stream, int* launches);

// CUDA-core FFMA path.
int launch_ffma(GemmArgs& g, cudaStream_t stream, int* launches);

// The pages' ladder kernels v0 .. v4 (step), for timing and teaching.
int launch_ladder(GemmArgs& g, int step, cudaStream_t stream, int* launches);

}  // namespace gemm_f32_impl
