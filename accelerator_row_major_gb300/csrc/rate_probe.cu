// Per-SM arithmetic rates of the two units the GEMM kernels use, measured on
// the current device: the roofline's compute peak ("Lesson 10: shared-memory
// tiled GEMM", hpc.payai.win, section 1: a kernel is judged against the
// peak of the unit that does its work, or against memory bandwidth).
//
//   tf32_rate_kernel<false>  back-to-back tcgen05.mma.cta_group::1.kind::tf32
//                            M = 128, N = 256, K = 8 (A from tensor memory,
//                            B from shared memory), one CTA per SM, no loads
//   tf32_rate_kernel<true>   the same with cta_group::2, M = 256 on SM pairs
//   ffma_rate_kernel         chains of fma.rn.f32x2 on 16 warps per SM
//
// Each CTA counts the SM clock (%clock64) over its own work and reads
// %globaltimer at both ends, so the rates come out per clock (independent of
// the clock the GPU runs at) and the clock itself comes out too.  The
// operands are zeros: throughput per clock does not depend on the values.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"

namespace {
using namespace gemm_f32_dev;

constexpr int kRateThreads = 128;
constexpr int kRateSmem = 120 * 1024;   // more than half an SM's shared memory: one CTA per SM
constexpr int kMmaM = 128, kMmaN = 256, kMmaK = 8;
constexpr int kBRows = kMmaN;           // shared-memory operand: 256 rows x 8 k (64-byte swizzle atoms)
constexpr int kFfmaThreads = 512;
constexpr int kFfmaChains = 8;          // independent fma.rn.f32x2 chains per thread
constexpr int kFfmaUnroll = 32;         // chain steps per loop iteration (loop overhead < 1 %)

struct ProbeOut {
  unsigned long long cycles;   // SM clock cycles of this CTA's timed work
  unsigned long long ns;       // globaltimer nanoseconds of the same span
};

__device__ __forceinline__ uint32_t probe_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void probe_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void probe_tmem_alloc(uint32_t slot) {
  if (PAIR)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(slot)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(slot)
                 : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void probe_tmem_dealloc(uint32_t taddr) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(taddr) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(taddr) : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void probe_mma(uint32_t d, uint32_t a, uint64_t b_desc, uint32_t idesc) {
  if (PAIR)
    asm volatile("tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, 1;" ::"r"(d), "r"(a),
                 "l"(b_desc), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, 1;" ::"r"(d), "r"(a),
                 "l"(b_desc), "r"(idesc)
                 : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void probe_commit(uint32_t bar) {
  if (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar),
        "h"(static_cast<uint16_t>(0x3))
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// One issuing thread per CTA (per pair with PAIR) issues `iters` MMAs into
// one accumulator and waits, bounded, for their completion.
template <bool PAIR>
__global__ void __launch_bounds__(kRateThreads, 1) tf32_rate_kernel(ProbeOut* out, unsigned* err,
                                                                    int iters) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  const uint32_t dyn0 = smem_addr(smem_dyn);
  const uint32_t base = (dyn0 + 1023u) & ~1023u;
  uint32_t* const b_ptr = reinterpret_cast<uint32_t*>(smem_dyn + (base - dyn0));
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = PAIR ? probe_cluster_rank() : 0u;

  for (int i = threadIdx.x; i < kBRows * kMmaK * 2; i += kRateThreads) b_ptr[i] = 0u;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  if (warp == 0) probe_tmem_alloc<PAIR>(smem_addr(&slot));
  tc_fence_before_sync();
  __syncthreads();
  if (PAIR) probe_cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&slot);
  // A operand: columns 256 .. 263 of every lane, zeroed
  {
    const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st_8cols(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256u, z);
    tmem_wait_st();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (PAIR) probe_cluster_sync();
  tc_fence_after_sync();

  const bool issuer = threadIdx.x == 0 && rank == 0;
  unsigned long long c0 = 0, t0 = 0;
  if (threadIdx.x == 0) {
    c0 = clock64();
    t0 = globaltimer_ns();
  }
  if (issuer) {
    // 64-byte swizzle atoms of 8 rows x 64 bytes (the stage layout of the
    // GEMM kernels at 16-deep stages)
    const uint64_t b_desc = smem_desc(base, 16, 512, 4);
    const uint32_t idesc = idesc_tf32(PAIR ? 2 * kMmaM : kMmaM, kMmaN, false, false);
#pragma unroll 1
    for (int i = 0; i < iters; ++i) probe_mma<PAIR>(tmem, tmem + 256u, b_desc, idesc);
    probe_commit<PAIR>(smem_addr(&bar));
  }
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(smem_addr(&bar), 0, err, kSiteDrainMma);
    const unsigned long long c1 = clock64();
    const unsigned long long t1 = globaltimer_ns();
    out[blockIdx.x].cycles = ok ? c1 - c0 : 0ull;
    out[blockIdx.x].ns = ok ? t1 - t0 : 0ull;
  }
  tc_fence_before_sync();
  __syncthreads();
  if (PAIR) probe_cluster_sync();   // the pair's MMAs are done with both CTAs' memory
  if (warp == 0) {
    tc_fence_after_sync();
    probe_tmem_dealloc<PAIR>(tmem);
  }
}

__device__ __forceinline__ uint64_t probe_fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// kFfmaChains independent chains acc = acc * m + c per thread; the results
// feed a store that never happens unless a value is NaN, so nothing is
// optimised away.
__global__ void __launch_bounds__(kFfmaThreads, 1) ffma_rate_kernel(ProbeOut* out, float* sink,
                                                                    int iters) {
  uint64_t acc[kFfmaChains];
#pragma unroll
  for (int j = 0; j < kFfmaChains; ++j) {
    const float x = static_cast<float>(threadIdx.x + j) * 1e-3f;
    acc[j] = (static_cast<uint64_t>(__float_as_uint(x)) << 32) | __float_as_uint(-x);
  }
  const uint64_t m = (static_cast<uint64_t>(__float_as_uint(0.999f)) << 32) | __float_as_uint(0.999f);
  const uint64_t c = (static_cast<uint64_t>(__float_as_uint(1e-4f)) << 32) | __float_as_uint(1e-4f);
  __syncthreads();
  unsigned long long c0 = 0, t0 = 0;
  if (threadIdx.x == 0) {
    c0 = clock64();
    t0 = globaltimer_ns();
  }
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int u = 0; u < kFfmaUnroll; ++u)
#pragma unroll
      for (int j = 0; j < kFfmaChains; ++j) acc[j] = probe_fma2(acc[j], m, c);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    out[blockIdx.x].cycles = clock64() - c0;
    out[blockIdx.x].ns = globaltimer_ns() - t0;
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kFfmaChains; ++j)
    s += __uint_as_float(static_cast<uint32_t>(acc[j])) + __uint_as_float(static_cast<uint32_t>(acc[j] >> 32));
  if (s != s) sink[threadIdx.x] = s;
}

double median(std::vector<double> v) {
  if (v.empty()) return 0.0;
  std::sort(v.begin(), v.end());
  const size_t h = v.size() / 2;
  return v.size() % 2 ? v[h] : 0.5 * (v[h - 1] + v[h]);
}

// Launches `kern` on `grid` CTAs, returns the median over CTAs (the issuing
// CTA of each pair only, with `stride` 2) of FLOP per cycle and of MHz.
template <class Launch>
int run_probe(Launch launch, int grid, int stride, double flop_per_cta, ProbeOut* d_out,
              unsigned* d_err, double* flop_per_clk, double* mhz) {
  if (cudaMemset(d_out, 0, sizeof(ProbeOut) * grid) != cudaSuccess ||
      cudaMemset(d_err, 0, sizeof(unsigned)) != cudaSuccess)
    return GEMM_F32_ELAUNCH;
  launch();
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return GEMM_F32_ELAUNCH;
  std::vector<ProbeOut> h(grid);
  unsigned err = 0;
  if (cudaMemcpy(h.data(), d_out, sizeof(ProbeOut) * grid, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&err, d_err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_F32_ELAUNCH;
  if (err) return GEMM_F32_ETIMEOUT;
  std::vector<double> rate, clk;
  for (int i = 0; i < grid; i += stride) {
    if (!h[i].cycles || !h[i].ns) return GEMM_F32_ETIMEOUT;
    rate.push_back(flop_per_cta / static_cast<double>(h[i].cycles));
    clk.push_back(1e3 * static_cast<double>(h[i].cycles) / static_cast<double>(h[i].ns));
  }
  *flop_per_clk = median(rate);
  *mhz = median(clk);
  return GEMM_F32_OK;
}

int unit_rates(gemm_f32_unit_rates_t* r) {
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GEMM_F32_EDEVICE;
  if (major != 10 || minor != 3 || sms < 2) return GEMM_F32_EDEVICE;
  if (cudaFuncSetAttribute(tf32_rate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kRateSmem) != cudaSuccess ||
      cudaFuncSetAttribute(tf32_rate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kRateSmem) != cudaSuccess)
    return GEMM_F32_ELAUNCH;
  void* buf = nullptr;
  const size_t out_bytes = sizeof(ProbeOut) * static_cast<size_t>(sms);
  if (cudaMalloc(&buf, out_bytes + 256 + kFfmaThreads * sizeof(float)) != cudaSuccess)
    return GEMM_F32_ELAUNCH;
  ProbeOut* const d_out = static_cast<ProbeOut*>(buf);
  unsigned* const d_err = reinterpret_cast<unsigned*>(static_cast<char*>(buf) + out_bytes);
  float* const d_sink = reinterpret_cast<float*>(static_cast<char*>(buf) + out_bytes + 256);
  const int mma_iters = 8192, ffma_iters = 512;
  const int pair_grid = sms & ~1;
  double mhz_tf32 = 0, mhz_pair = 0, mhz_ffma = 0;
  int rc = run_probe(
      [&] { tf32_rate_kernel<false><<<sms, kRateThreads, kRateSmem>>>(d_out, d_err, mma_iters); },
      sms, 1, 2.0 * kMmaM * kMmaN * kMmaK * mma_iters, d_out, d_err, &r->tf32_flop_per_clk_sm,
      &mhz_tf32);
  if (rc == GEMM_F32_OK) {
    // one issuing CTA per pair; its work covers two SMs
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(pair_grid);
    cfg.blockDim = dim3(kRateThreads);
    cfg.dynamicSmemBytes = kRateSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    rc = run_probe(
        [&] { (void)cudaLaunchKernelEx(&cfg, tf32_rate_kernel<true>, d_out, d_err, mma_iters); },
        pair_grid, 2, 2.0 * kMmaM * kMmaN * kMmaK * mma_iters, d_out, d_err,
        &r->tf32_pair_flop_per_clk_sm, &mhz_pair);
  }
  if (rc == GEMM_F32_OK)
    rc = run_probe(
        [&] { ffma_rate_kernel<<<sms, kFfmaThreads>>>(d_out, d_sink, ffma_iters); }, sms, 1,
        4.0 * kFfmaThreads * kFfmaChains * kFfmaUnroll * ffma_iters, d_out, d_err,
        &r->ffma_flop_per_clk_sm, &mhz_ffma);
  (void)cudaFree(buf);
  if (rc != GEMM_F32_OK) {
    (void)cudaGetLastError();
    return rc;
  }
  r->sm_mhz = median({mhz_tf32, mhz_pair, mhz_ffma});
  r->num_sms = sms;
  return GEMM_F32_OK;
}

}  // namespace

extern "C" int gemm_f32_unit_rates(gemm_f32_unit_rates_t* rates) {
  if (!rates) return GEMM_F32_EINVAL;
  return unit_rates(rates);
}
