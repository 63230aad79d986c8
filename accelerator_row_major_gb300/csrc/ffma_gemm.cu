// CUDA-core FP32 GEMM (FFMA) for sm_103a: persistent CTAs, 8 x 16 outputs
// per thread, a 4-stage cp.async shared-memory ring, and the paired fp32
// fused multiply-add (fma.rn.f32x2: two FMAs per lane per instruction, each
// rounded once like fmaf).  Block tiles of 256 threads, one CTA per SM:
// 128 x 256, and 512 x 64 for N <= 64 and 64 x 512 for M <= 64, so that
// skinny products spend no multiply-adds on rows or columns beyond the
// matrix.
//
// Computes C[i][j] = sum_k A[i][k] * B[k][j] (row-major) in fp32 fused
// multiply-adds, k ascending per output.  The structure follows the pages'
// last step -- 2-D register coarsening, where each thread keeps a tile of C
// in registers and reuses every loaded A and B value across it ("LeetGPU
// problem 2: matrix multiplication", yekq.top, section v4) -- on top of
// shared-memory K tiles ("Lesson 10: shared-memory tiled GEMM",
// hpc.payai.win, section 2).  Differences: the K tiles are copied by
// cp.async several tiles ahead (no register staging), one barrier per K
// tile instead of two (the stage being filled is never the one being read),
// 16-byte copies where the strides allow, and a persistent grid.
// Out-of-range elements are zero-filled by the copy and never stored; no
// thread leaves before the last barrier ("Lesson 10", section 3).
//
// The last partial wave is split along K like the tensor-core path's (see
// device_common.cuh): partial tiles go through the library's workspace.
//
// Thread (tx, ty) of the TX x TY grid (TX = BN / 16, TY = BM / 8) owns rows
// ty + TY i (i < 8) and columns (BN / 4) g + 4 tx .. +3 (g < 4).  A warp
// covers min(TX, 8) values of tx and the rest of its lanes along ty, so per
// K step its 16-byte A reads hit 4 or 8 consecutive rows (distinct banks
// with the 20-float row pitch) and its B reads one 128- or 64-byte segment.
// The block tile is a template parameter: the pages' last step makes the
// block and thread tiles (BM, BN, TM, TN) parameters of the kernel for the
// same reason ("LeetGPU problem 2", section v4).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"
#include "launch.h"

namespace gemm_f32_impl {
using namespace gemm_f32_dev;

namespace {

constexpr int kBK = 16;
constexpr int kAPitch = kBK + 4;               // floats per A row in shared memory
constexpr int kRasterGroup = 8;

// A block tile of BM x BN outputs, 8 x 16 per thread.
template <int BM_, int BN_, int STAGES_ = 4>
struct FfmaTile {
  static constexpr int BM = BM_, BN = BN_;
  static constexpr int STAGES = STAGES_;                  // shared-memory ring depth
  static constexpr int TY = BM / 8, TX = BN / 16;       // threads along rows / columns
  static constexpr int THREADS = TX * TY;
  static constexpr int LX = TX < 8 ? TX : 8;              // lanes of a warp along columns
  static constexpr int WX = TX / LX;                      // warps along columns
  static constexpr int CG = BN / 4;                       // column-group stride
  static constexpr int CTAS_PER_SM = 256 / THREADS;       // 8 warps per SM
  static constexpr int A_STAGE = BM * kAPitch;            // floats, per-thread copies
  static constexpr int B_STAGE = kBK * BN;                // floats
  static constexpr int SMEM = STAGES * (A_STAGE + B_STAGE) * 4;
  // TMA loads: A stages dense (BM rows of 16 floats, 64-byte swizzle), in
  // boxes of at most 256 rows; B stages of 16 rows, in boxes of at most 256
  // columns ([box][16][A_BOX... B_BOX]); 1024-byte aligned.
  static constexpr int A_BOX = BM < 256 ? BM : 256;
  static constexpr int B_BOX = BN < 256 ? BN : 256;
  static constexpr int A_STAGE_TMA = BM * kBK;            // floats
  static constexpr int STAGE_BYTES_TMA = (A_STAGE_TMA + B_STAGE) * 4;
  static constexpr int SMEM_TMA = STAGES * STAGE_BYTES_TMA + 1024;
  static_assert(THREADS % 32 == 0 && BM * 4 % THREADS == 0 && BN * 4 % THREADS == 0, "tile");
  // a thread's rows ty + TY i share one swizzle phase ((row >> 1) & 3)
  static_assert(TY % 8 == 0 && BM % A_BOX == 0 && BN % B_BOX == 0, "TMA tile");
  static_assert((A_STAGE_TMA * 4) % 1024 == 0 && STAGE_BYTES_TMA % 1024 == 0, "TMA alignment");
};
// The skinny tiles keep 256 threads in one CTA per SM: measured on GB300
// (per-CTA timestamps), two 128-thread CTAs sharing an SM do not share it
// evenly -- one finishes its (equal) work in 57 % of the time of the other,
// which then runs on 4 warps, too few to keep the FMA pipe busy (64 x 4096
// x 65536 with 64 x 256 tiles: CTAs ending at 360-370 us and 640-647 us, an
// average of 6.3 resident warps out of 8).
using TileWide = FfmaTile<128, 256>;     // default
using TileTall = FfmaTile<512, 64>;      // N <= 64
using TileShort = FfmaTile<64, 512>;     // M <= 64
constexpr int kMaxPending = 8;               // split tiles one CTA may have to reduce
// An FFMA K iteration costs ~6x a tensor-core one, so splitting the tail pays
// off at far fewer iterations per CTA (measured on GB300: 2.5x on 1024 x 512 x
// 1024 with 8, none with the tensor-core kernels' 64).
constexpr int kMinSplitItersFfma = 8;

struct FfmaParams {
  const float* __restrict__ A;
  const float* __restrict__ B;
  float* __restrict__ C;
  int M, N, K;
  int tiles_m, tiles_n, k_iters;
  int dp_tiles;          // tiles 0 .. dp_tiles-1 are computed whole, round robin
  int sk_ctas;           // CTAs 0 .. sk_ctas-1 share the K iterations of the rest
  long long sk_work;     // (tiles - dp_tiles) * k_iters
  int max_seg;           // most CTAs sharing one tail tile
  float* partials;       // [tail tile][max_seg][BM][BN] fp32
  unsigned long long* counters;   // [tail tile]: generation and partials published
  int drop_first_copy;   // testing only (TMA loads): CTA 0 never fills its first stage
  unsigned* err;
};

// The general form's parameters: row strides, transposed storage (4-byte
// copies only), alpha / beta (scale = 1), and whether rows of C take 16-byte
// stores.  A separate kernel argument: measured on GB300, growing FfmaParams
// changed the plain kernel's register allocation and cost it 2 %.
struct FfmaGeneral {
  int lda, ldb, ldc;
  int trans_a, trans_b;
  float alpha, beta;
  int scale;
  int c_vec;
};

// Two fused multiply-adds per lane: d.x = a.x * b.x + c.x, d.y = a.y * b.y + c.y
// (each rounded once, as fmaf), on 64-bit register pairs.
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t pair(float x, float y) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(x), "f"(y));
  return d;
}

__device__ __forceinline__ float2 unpair(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copies K tile `kt` of the block's A panel and B panel into one stage with
// 4-byte cp.async copies (any alignment, any stride, transposed storage);
// out-of-range elements are zero-filled.
template <class T, bool GEN>
__device__ __forceinline__ void load_stage(const FfmaParams& p, const FfmaGeneral& gp, int m0,
                                           int n0, int kt,
                                           uint32_t a_dst, uint32_t b_dst) {
  const int tid = threadIdx.x;
  const int k0 = kt * kBK;
  const int lda = GEN ? gp.lda : p.K, ldb = GEN ? gp.ldb : p.N;
  const bool trans_a = GEN && gp.trans_a, trans_b = GEN && gp.trans_b;
  [[maybe_unused]] const size_t a_extent =
      trans_a ? stored_extent(p.K, p.M, lda) : stored_extent(p.M, p.K, lda);
  [[maybe_unused]] const size_t b_extent =
      trans_b ? stored_extent(p.N, p.K, ldb) : stored_extent(p.K, p.N, ldb);
  // A: BM rows x 16 k = 4 BM chunks of 4 floats; thread -> chunks tid + THREADS h
#pragma unroll
  for (int h = 0; h < T::BM * 4 / T::THREADS; ++h) {
    const int c = tid + h * T::THREADS;
    const int r = c >> 2, kc = (c & 3) * 4;
    const int gm = m0 + r, gk = k0 + kc;
    const uint32_t dst = a_dst + (r * kAPitch + kc) * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const size_t at = trans_a ? static_cast<size_t>(gk + e) * lda + gm
                                : static_cast<size_t>(gm) * lda + gk + e;
      const bool in = gm < p.M && gk + e < p.K &&
                      GEMM_IN_EXTENT(at, a_extent, p.err, kSiteBoundsA);
      cp_async_4(dst + 4 * e, in ? p.A + at : p.A, in ? 4u : 0u);
    }
  }
  // B: 16 k x BN columns = 4 BN chunks; thread -> chunks tid + THREADS h
#pragma unroll
  for (int h = 0; h < T::BN * 4 / T::THREADS; ++h) {
    const int c = tid + h * T::THREADS;
    const int k = c / (T::BN / 4), nc = (c % (T::BN / 4)) * 4;
    const int gk = k0 + k, gn = n0 + nc;
    const uint32_t dst = b_dst + (k * T::BN + nc) * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const size_t at = trans_b ? static_cast<size_t>(gn + e) * ldb + gk
                                : static_cast<size_t>(gk) * ldb + gn + e;
      const bool in = gk < p.K && gn + e < p.N &&
                      GEMM_IN_EXTENT(at, b_extent, p.err, kSiteBoundsB);
      cp_async_4(dst + 4 * e, in ? p.B + at : p.B, in ? 4u : 0u);
    }
  }
}

// One stage of the inner product: acc += A tile x B tile over its 16 k.
// `a_at(i, kg)` gives the shared-memory float offset of the float4 of row
// ty + TY i, k 4 kg .. 4 kg + 3; `b_at(k, g)` that of the float4 of row k,
// columns CG g + 4 tx .. + 3.
template <class T, class AAt, class BAt>
__device__ __forceinline__ void stage_product(const float* as, const float* bs, AAt a_at, BAt b_at,
                                              uint64_t (&acc)[8][8]) {
#pragma unroll
  for (int kg = 0; kg < kBK / 4; ++kg) {
    float4 a4[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a4[i] = *reinterpret_cast<const float4*>(as + a_at(i, kg));
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint64_t b[8];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(bs + b_at(kg * 4 + kk, g));
        b[2 * g] = v.x;
        b[2 * g + 1] = v.y;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float a = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
        const uint64_t aa = pair(a, a);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][q] = fma2(aa, b[q], acc[i][q]);
      }
    }
  }
}

// VEC: operands the tensor-memory accelerator can read (untransposed, row
// strides a multiple of 4 floats, 16-byte aligned bases): one thread loads
// each stage with TMA boxes, completion counted on the stage's mbarrier, and
// every thread waits on it (bounded, as in the tensor-core kernels).
// Otherwise every thread copies 4-byte elements with cp.async.
// GEN: the general form (row strides, stored transposes, alpha / beta); a
// separate instantiation, so that the plain product's code is unchanged.
template <class T, bool VEC, bool GEN>
__global__ void __launch_bounds__(T::THREADS, T::CTAS_PER_SM)
    ffma_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const FfmaParams p,
                     const FfmaGeneral gp) {
  constexpr int BM = T::BM, BN = T::BN, TY = T::TY, CG = T::CG;
  constexpr int kStages = T::STAGES;
  // extents (elements) of C and of the partial tiles, for the checked build
  [[maybe_unused]] const size_t c_extent = stored_extent(p.M, p.N, GEN ? gp.ldc : p.N);
  [[maybe_unused]] const size_t work_extent =
      static_cast<size_t>(p.tiles_m * p.tiles_n - p.dp_tiles) * p.max_seg * (BM * BN);
  extern __shared__ __align__(16) float smem_f[];
  __shared__ WorkItem pending[kMaxPending];   // split tiles this CTA must reduce
  __shared__ int pending_count;
  __shared__ __align__(8) uint64_t full_bar[kStages];   // TMA loads: stage filled
  __shared__ unsigned long long clk_mark[2];            // the clock record's start
  clock_start(clk_mark);
  const uint32_t dyn0 = smem_addr(smem_f);
  const uint32_t base = VEC ? (dyn0 + 1023u) & ~1023u : dyn0;
  float* const As = smem_f + (base - dyn0) / 4;      // [stage][BM][16 or kAPitch]
  constexpr int A_ST = VEC ? T::A_STAGE_TMA : T::A_STAGE;
  float* const Bs = As + kStages * A_ST;             // [stage][B box][16][B_BOX]
  const uint32_t as_addr = smem_addr(As), bs_addr = smem_addr(Bs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tx = (warp % T::WX) * T::LX + lane % T::LX;
  const int ty = (warp / T::WX) * (32 / T::LX) + lane / T::LX;
  if (threadIdx.x == 0) {
    pending_count = 0;
    if (VEC) {
      for (int st = 0; st < kStages; ++st) mbar_init(smem_addr(&full_bar[st]), 1);
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
    }
  }
  __syncthreads();
  grid_launch_dependents();
  grid_dependency_wait();   // global memory from here on

  // TMA loads: fills issued (thread 0) and stages consumed (every thread),
  // counted over all work items, so stage = n % S and parity = (n / S) & 1
  uint32_t fills = 0, uses = 0;
  int dropped = -1;     // test hook: the stage that was never filled
  bool ok = true;
  const int sw = (ty >> 1) & 3;   // 64-byte swizzle phase of this thread's A rows
  auto a_at_tma = [&](int i, int kg) { return (ty + TY * i) * kBK + ((kg ^ sw) << 2); };
  auto a_at_copy = [&](int i, int kg) { return (ty + TY * i) * kAPitch + kg * 4; };
  auto b_at_tma = [&](int k, int g) {
    const int col = g * CG + tx * 4;
    return (col / T::B_BOX) * (kBK * T::B_BOX) + k * T::B_BOX + col % T::B_BOX;
  };
  auto b_at_copy = [&](int k, int g) { return k * BN + g * CG + tx * 4; };

  WorkList list(p);
  WorkItem w;
  while (ok && list.next(p, w)) {
    const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup);
    const int m0 = c.tm * BM, n0 = c.tn * BN;
    const int nk = w.k1 - w.k0;
    // acc[i][q] holds C columns 2q, 2q+1 of row i of this thread's 8 x 16
    uint64_t acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[i][q] = 0ull;

    if constexpr (VEC) {
      // one thread fills stage fills % S with K tile kt; the stage it
      // overwrites was consumed at least one barrier ago
      auto issue = [&](int kt) {
        const uint32_t st = fills % kStages;
        const uint32_t bar = smem_addr(&full_bar[st]);
        if (p.drop_first_copy && blockIdx.x == 0 && fills == 0) {
          dropped = 0;   // never armed: the waits on it run out
        } else {
          mbar_arrive_expect_tx(bar, T::STAGE_BYTES_TMA);
          const uint32_t a_dst = as_addr + st * (T::A_STAGE_TMA * 4);
          const uint32_t b_dst = bs_addr + st * (T::B_STAGE * 4);
#pragma unroll
          for (int h = 0; h < BM / T::A_BOX; ++h)
            tma_load_2d(a_dst + h * (T::A_BOX * kBK * 4), &tmA, bar, kt * kBK, m0 + h * T::A_BOX);
#pragma unroll
          for (int h = 0; h < BN / T::B_BOX; ++h)
            tma_load_2d(b_dst + h * (T::B_BOX * kBK * 4), &tmB, bar, n0 + h * T::B_BOX, kt * kBK);
        }
        ++fills;
      };
      if (threadIdx.x == 0)
        for (int st = 0; st < kStages - 1 && st < nk; ++st) issue(w.k0 + st);
      for (int j = 0; j < nk; ++j) {
        const uint32_t st = uses % kStages;
        const bool got = mbar_wait(smem_addr(&full_bar[st]), (uses / kStages) & 1u, p.err,
                                   kSiteTransformFull);
        // every thread's copy of the verdict; also the barrier after which
        // stage (j - 1) % S, read by the iteration before, may be refilled
        if (!__syncthreads_and(got)) {
          ok = false;
          break;
        }
        if (threadIdx.x == 0 && j + kStages - 1 < nk) issue(w.k0 + j + kStages - 1);
        stage_product<T>(As + st * T::A_STAGE_TMA, Bs + st * T::B_STAGE, a_at_tma, b_at_tma,
                         acc);
        ++uses;
      }
      if (!ok) break;
      __syncthreads();
    } else {
      // prologue: the first kStages-1 tiles in flight (empty groups keep the count)
#pragma unroll
      for (int st = 0; st < kStages - 1; ++st) {
        if (st < nk)
          load_stage<T, GEN>(p, gp, m0, n0, w.k0 + st, as_addr + st * T::A_STAGE * 4,
                             bs_addr + st * T::B_STAGE * 4);
        cp_async_commit();
      }
      for (int j = 0; j < nk; ++j) {
        cp_async_wait<kStages - 2>();   // this thread's copies of tile j have landed
        __syncthreads();                // everyone's have; stage (j-1) % S is free
        const int nxt = j + kStages - 1;
        if (nxt < nk) {
          const int st = nxt % kStages;
          load_stage<T, GEN>(p, gp, m0, n0, w.k0 + nxt, as_addr + st * T::A_STAGE * 4,
                             bs_addr + st * T::B_STAGE * 4);
        }
        cp_async_commit();
        stage_product<T>(As + (j % kStages) * T::A_STAGE, Bs + (j % kStages) * T::B_STAGE,
                         a_at_copy, b_at_copy, acc);
      }
      cp_async_wait<0>();
      __syncthreads();   // the next item's prologue overwrites stages still being read
    }

    if (w.nseg == 1) {
      // epilogue: rows ty + TY i, columns CG g + 4 tx .. +3
      if constexpr (!GEN) {
        const bool c_vec = VEC && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = m0 + ty + TY * i;
          if (r >= p.M) continue;
          float* crow = p.C + static_cast<size_t>(r) * p.N;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int n = n0 + g * CG + tx * 4;
            const float2 lo = unpair(acc[i][2 * g]), hi = unpair(acc[i][2 * g + 1]);
            const float v[4] = {lo.x, lo.y, hi.x, hi.y};
            if (c_vec && n + 3 < p.N) {
              if (GEMM_IN_EXTENT(crow + n + 3 - p.C, c_extent, p.err, kSiteBoundsC))
                *reinterpret_cast<float4*>(crow + n) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (n + q < p.N && GEMM_IN_EXTENT(crow + n + q - p.C, c_extent, p.err, kSiteBoundsC))
                  crow[n + q] = v[q];
            }
          }
        }
      } else {
        // general form: row stride ldc; alpha * sum (+ beta * C_old, read
        // only when beta != 0)
        const bool c_vec = VEC && gp.c_vec != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = m0 + ty + TY * i;
          if (r >= p.M) continue;
          float* crow = p.C + static_cast<size_t>(r) * gp.ldc;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int n = n0 + g * CG + tx * 4;
            const float2 lo = unpair(acc[i][2 * g]), hi = unpair(acc[i][2 * g + 1]);
            float v[4] = {lo.x, lo.y, hi.x, hi.y};
            if (gp.scale) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                v[q] *= gp.alpha;
                if (gp.beta != 0.0f && n + q < p.N &&
                    GEMM_IN_EXTENT(crow + n + q - p.C, c_extent, p.err, kSiteBoundsC))
                  v[q] = fmaf(gp.beta, crow[n + q], v[q]);
              }
            }
            if (c_vec && n + 3 < p.N) {
              if (GEMM_IN_EXTENT(crow + n + 3 - p.C, c_extent, p.err, kSiteBoundsC))
                *reinterpret_cast<float4*>(crow + n) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (n + q < p.N && GEMM_IN_EXTENT(crow + n + q - p.C, c_extent, p.err, kSiteBoundsC))
                  crow[n + q] = v[q];
            }
          }
        }
      }
    } else {
      // part of a split tile: publish it; the CTA that publishes last reduces
      // the tile after its work list
      float* const slot =
          p.partials + (static_cast<size_t>(w.tail) * p.max_seg + w.seg) * (BM * BN);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float2 lo = unpair(acc[i][2 * g]), hi = unpair(acc[i][2 * g + 1]);
          float* const to = slot + (ty + TY * i) * BN + g * CG + tx * 4;
          if (GEMM_IN_EXTENT(to + 3 - p.partials, work_extent, p.err, kSiteBoundsWork))
            *reinterpret_cast<float4*>(to) = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0 &&
          tail_arrive(p.counters, w.tail) == static_cast<unsigned>(w.nseg)) {
        // only the first and the last item of a CTA's share can be partial
        if (pending_count < kMaxPending)
          pending[pending_count++] = w;
        else
          record_error(p.err, kSitePendingOverflow);
      }
    }
  }

  if (!ok) {
    // a wait ran out (reported in the error word): C of this call is left
    // as it is; the loads still in flight land before the CTA's shared
    // memory goes away
    if (threadIdx.x == 0)
      for (uint32_t f = uses; f < fills; ++f)
        if (static_cast<int>(f) != dropped)
          mbar_wait(smem_addr(&full_bar[f % kStages]), (f / kStages) & 1u, p.err, kSiteDrainTma);
    __syncthreads();
    clock_stop(p.err, clk_mark);
    if (p.sk_ctas > 0 && threadIdx.x == 0) tail_launch_done(p.counters);
    return;
  }
  __syncthreads();
  const int npend = pending_count;
  if (npend > 0) {
    __threadfence();
    for (int e = 0; e < npend; ++e) {
      const WorkItem pw = pending[e];
      const TileCoord c = tile_coord(pw.tile, p.tiles_m, p.tiles_n, kRasterGroup);
      const size_t at = static_cast<size_t>(pw.tail) * p.max_seg * (BM * BN);
      const float* parts = p.partials + at;
      const BoundsRef br{p.err, work_extent - at, c_extent};
      if constexpr (!GEN)
        reduce_partials<BM, BN, T::THREADS, 16>(parts, pw.nseg, c.tm * BM, c.tn * BN, p.M, p.N,
                                                p.C, br);
      else
        reduce_partials_general<BM, BN, T::THREADS, 16>(parts, pw.nseg, c.tm * BM, c.tn * BN,
                                                        p.M, p.N, p.C, gp.ldc, gp.scale, gp.alpha,
                                                        gp.beta, br);
    }
  }
  clock_stop(p.err, clk_mark);
  if (p.sk_ctas > 0 && threadIdx.x == 0) tail_launch_done(p.counters);
}

constexpr int kMaxDevices = 64;

// Configures the kernel once per device (its dynamic shared memory, and all
// of the unified L1 / shared memory as shared memory: the 512 x 64 tile's
// four stages take 176 KB) and returns how many of its CTAs an SM holds (0 on
// failure), which the persistent grid is planned with.
template <class T, bool VEC, bool GEN>
int resident_ctas(int device) {
  static std::atomic<int> per_sm[kMaxDevices];   // 0: not configured yet
  const int d = device % kMaxDevices;
  int n = per_sm[d].load();
  if (n > 0) return n;
  auto kern = ffma_gemm_kernel<T, VEC, GEN>;
  constexpr int smem = VEC ? T::SMEM_TMA : T::SMEM;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, T::THREADS, smem) != cudaSuccess ||
      n < 1) {
    (void)cudaGetLastError();
    return 0;
  }
  n = std::min(n, T::CTAS_PER_SM);
  per_sm[d].store(n);
  return n;
}

template <class T, bool VEC, bool GEN>
int launch_vec(const CUtensorMap& ma, const CUtensorMap& mb, const FfmaParams& p,
               const FfmaGeneral& gp, int grid, cudaStream_t stream) {
  if (launch_dependent(ffma_gemm_kernel<T, VEC, GEN>, dim3(grid), dim3(T::THREADS),
                       VEC ? T::SMEM_TMA : T::SMEM, stream, ma, mb, p, gp) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  return GEMM_F32_OK;
}

// Plans and launches the product on block tiles T: persistent CTAs
// (CTAS_PER_SM per SM), the last partial wave split along K when that
// leaves every CTA at least kMinSplitItersFfma K tiles.
template <class T>
int launch_tile(GemmArgs& g, cudaStream_t stream, int* launches) {
  *launches = 0;
  FfmaParams p;
  p.A = g.A;
  p.B = g.B;
  p.C = g.C;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles_m = (g.M + T::BM - 1) / T::BM;
  p.tiles_n = (g.N + T::BN - 1) / T::BN;
  p.k_iters = (g.K + kBK - 1) / kBK;
  p.partials = nullptr;
  p.counters = nullptr;
  p.drop_first_copy = (g.flags & GEMM_F32_FLAG_TEST_DROP_COPY) ? 1 : 0;
  p.err = g.err;
  FfmaGeneral gp;
  gp.lda = g.lda;
  gp.ldb = g.ldb;
  gp.ldc = g.ldc;
  gp.trans_a = g.trans_a;
  gp.trans_b = g.trans_b;
  gp.alpha = g.alpha;
  gp.beta = g.beta;
  gp.scale = g.scale;
  gp.c_vec = g.ldc % 4 == 0 && reinterpret_cast<uintptr_t>(g.C) % 16 == 0;
  const long tiles = static_cast<long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fffffffL) return GEMM_F32_EINVAL;
  p.dp_tiles = static_cast<int>(tiles);
  p.sk_ctas = 0;
  p.sk_work = 0;
  p.max_seg = 1;
  // TMA loads: untransposed operands, row strides a multiple of 4 floats,
  // 16-byte aligned bases (ragged edges read as zero); otherwise 4-byte copies
  alignas(64) CUtensorMap ma, mb;
  bool vec = tma_addressable(g) &&
             tma_encode_2d(&ma, g.A, g.M, g.K, g.lda, kBK, T::A_BOX, CU_TENSOR_MAP_SWIZZLE_64B) &&
             tma_encode_2d(&mb, g.B, g.K, g.N, g.ldb, T::B_BOX, kBK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!vec) {
    memset(&ma, 0, sizeof(ma));
    memset(&mb, 0, sizeof(mb));
  }
  const bool gen = !plain_form(g);
  const int per_sm = gen ? (vec ? resident_ctas<T, true, true>(g.device)
                                : resident_ctas<T, false, true>(g.device))
                         : (vec ? resident_ctas<T, true, false>(g.device)
                                : resident_ctas<T, false, false>(g.device));
  if (per_sm < 1) return GEMM_F32_ELAUNCH;
  const int slots = g.num_sms * per_sm;   // CTAs resident at once
  int grid = (g.flags & GEMM_F32_FLAG_ONE_TILE_PER_CTA)
                 ? static_cast<int>(tiles)
                 : static_cast<int>(std::min<long>(tiles, slots));
  if (!(g.flags & (GEMM_F32_FLAG_ONE_TILE_PER_CTA | GEMM_F32_FLAG_NO_SPLIT_K))) {
    FfmaParams q = p;
    const size_t ws_bytes =
        plan_split_tail(q, tiles, slots, sizeof(float) * T::BM * T::BN, kMinSplitItersFfma);
    void* ws = ws_bytes ? acquire_workspace(g.device, stream, ws_bytes) : nullptr;
    if (ws) {
      p = q;
      grid = slots;
      p.counters = static_cast<unsigned long long*>(ws);
      p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
    }
  }
  int rc;
  if (gen)
    rc = vec ? launch_vec<T, true, true>(ma, mb, p, gp, grid, stream)
             : launch_vec<T, false, true>(ma, mb, p, gp, grid, stream);
  else
    rc = vec ? launch_vec<T, true, false>(ma, mb, p, gp, grid, stream)
             : launch_vec<T, false, false>(ma, mb, p, gp, grid, stream);
  if (rc == GEMM_F32_OK) {
    *launches += 1;
    g.kernel = "ffma_gemm_kernel";
  }
  return rc;
}

}  // namespace

// Block tiles by shape: a tile taller than wide for N <= 64 and one wider
// than tall for M <= 64, where the 128 x 256 tile would spend three quarters
// (N = 64) or half (M = 64) of its multiply-adds beyond the matrix.
int launch_ffma(GemmArgs& g, cudaStream_t stream, int* launches) {
  if (g.N <= TileTall::BN && g.M > TileShort::BM) return launch_tile<TileTall>(g, stream, launches);
  if (g.M <= TileShort::BM) return launch_tile<TileShort>(g, stream, launches);
  return launch_tile<TileWide>(g, stream, launches);
}

}  // namespace gemm_f32_impl
