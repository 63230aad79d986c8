// Tensor-core FP32 GEMM for sm_103a: tcgen05.mma kind::tf32 with a TMEM
// accumulator, fed by TMA (or by masked per-thread loads where TMA cannot
// address the operands), with the 3xTF32 split done in shared memory.
//
// Computes C[i][j] = sum_k A[i][k] * B[k][j] for row-major A (M x K),
// B (K x N), C (M x N): the product of "LeetGPU problem 2: matrix
// multiplication" (yekq.top, section "problem statement").  The pages tile
// the product in shared memory with two barriers per K phase ("Lesson 10:
// shared-memory tiled GEMM", hpc.payai.win, section 2); here the K phases
// flow through a ring of stages guarded by mbarriers instead, and ragged
// edges are zero-filled on load and masked on store as in the pages'
// guarded tiles (same lesson, section 3; "LeetGPU problem 2", v3 tail fix).
//
// Tile: 128 columns of C (n) by TM rows (m).  Row-major B is N-contiguous,
// and a kind::tf32 MMA only accepts K-major operands, so B is transposed on
// its way into the tensor core: the transform warps read the raw B tile
// (thread t owns column n0 + t) and write its TF32 hi/lo parts into tensor
// memory, where lane t holds column t and one 32-bit column holds one k.
// That is the MMA's A operand (M = 128 lanes); the A tile, K-major as it
// sits in memory, is the MMA's shared-memory B operand (N = TM).  The MMA
// therefore accumulates the transposed tile, D[n][m] = C[m][n], which also
// makes the epilogue's stores coalesced (lane t writes column n0 + t).
// For N <= 64 the tile is 64 columns wide (TN = 64).  With one product the
// MMA has M = 64, whose rows live in lanes 0-15 of each 32-lane quarter
// (measured on GB300), and the transform and the epilogue follow that
// layout, as does the 256-row tile with three products; in shorter tiles
// with three products B^T hi fills lanes 0-63 and B^T lo lanes 64-127 of an
// M = 128 operand (two MMAs per K step, on A hi and on A lo), and the
// epilogue adds lanes 64 + n to lanes n through shared memory.  Tiles of 64 rows with
// three products read A hi and A lo as one operand of 128 rows (they are
// adjacent in the stage), so each K step takes two N = 128 MMAs instead of
// three N = 64 ones (an N = 64 MMA costs about 72 cycles in this kernel, an
// N = 128 one about 73), and the lo x lo product comes along; the epilogue
// adds the accumulator's hi-row and lo-row halves.
//
// Template parameters: tile height TM (256, 128, 64), stage depth BK (16,
// 32), products NPROD (3: 3xTF32, 1: 1xTF32), operand loader LOAD (TMA;
// per-thread loads of the plain product; per-thread loads of the general
// form with row strides and stored transposes) and tile width TN.  The
// general form's alpha / beta and strides arrive in a separate argument, so
// that the plain product's code is left as it is.
//
// Roles inside one persistent CTA (one CTA per SM, 16 warps):
//   warp 0        TMA producer: A tile [TM x BK] (swizzled) and B tile
//                 [BK x 128] per K phase into stage s
//   warp 1        TMEM allocator and MMA issuer (one thread)
//   warps 4..7    epilogue: TMEM -> registers -> C (masked, coalesced)
//   warps 8..15   transform: A tile -> TF32 lo in shared memory (the raw
//                 tile is the hi part; with one product the tensor core reads
//                 it truncated); B tile -> TF32 hi/lo of its transpose in TMEM
//                 (warps w and w+4 share TMEM lanes 32(w%4).., each taking
//                 half of the tile's K rows).
//                 On the staged path (operands TMA cannot address) these
//                 warps load both tiles from global memory themselves, all of
//                 a stage's loads issued before any is used.
// Every role walks the same list of work items (below) and the same K-phase
// count per item, so no role leaves a barrier phase unfinished (the
// uniform-control rule of "Lesson 10", section 3).
//
// Work list of CTA c (grid G): first whole tiles c, c+G, ... of the leading
// full waves; then, when the tile count is not a multiple of G, an equal
// share of the remaining tiles' K iterations (the tail is cut along K, so
// every CTA finishes at about the same time).  A CTA that computes only part
// of a tile's K range writes its partial tile to a workspace and bumps the
// tile's counter; the CTA that arrives last adds all partials in segment
// order (fixed, so the result does not depend on which CTA is last) and
// writes C.  No CTA waits for another.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"
#include "launch.h"

namespace gemm_f32_impl {
using namespace gemm_f32_dev;

namespace {

constexpr int kTN = 128;                     // columns of C per tile = TMEM lanes = MMA M
constexpr int kTNNarrow = 64;                // the same for N <= 64: an M = 64 MMA, whose
                                             // rows sit in lanes 0-15 of each lane quarter
constexpr int kWarps = 16;                   // see role table above
constexpr int kThreads = kWarps * 32;
constexpr int kEpilogueWarp0 = 4;
constexpr int kTransformWarp0 = 8;
constexpr int kTransformThreads = 256;       // two warps per TMEM lane quarter
constexpr int kEpilogueThreads = 128;
constexpr int kEpilogueBarrier = 1;          // named barrier of the epilogue warps
constexpr int kSmemLimit = 232448;           // opt-in dynamic shared memory per block
constexpr int kTmemCols = 512;
constexpr int kRasterGroup = 8;              // tile-rows per L2 group
constexpr int kMaxPending = 8;               // split tiles one CTA may have to reduce

struct TcParams {
  const float* A;
  const float* B;
  float* C;
  int M, N, K;
  int tiles_m, tiles_n, k_iters;
  int dp_tiles;          // tiles 0 .. dp_tiles-1 are computed whole, round robin
  int sk_ctas;           // CTAs 0 .. sk_ctas-1 share the K iterations of the rest
  long long sk_work;     // (tiles - dp_tiles) * k_iters
  int max_seg;           // most CTAs sharing one tail tile
  float* partials;       // [tail tile][max_seg][TM][128] fp32
  unsigned long long* counters;   // [tail tile]: generation and partials published
  int drop_first_copy;   // testing only: CTA 0 skips its first copy
  unsigned* err;
};

// The general form C = alpha op(A) op(B) + beta C: row strides, stored
// transposes (staged loader only) and alpha / beta.  A separate kernel
// argument, so that the plain product's parameters keep their layout.
struct TcGeneral {
  int lda, ldb, ldc;
  int trans_a, trans_b;
  float alpha, beta;
  int scale;             // C = alpha * acc (+ beta * C when beta != 0)
};

template <int TM, int BK, int NPROD, int TN = kTN>
struct TcCfg {
  static constexpr int A_BYTES = TM * BK * 4;                       // A hi (TMA target)
  static constexpr int A_LO_BYTES = NPROD == 3 ? A_BYTES : 0;       // A lo
  static constexpr int B_RAW_BYTES = BK * TN * 4;                   // raw B tile [BK][TN]
  static constexpr int STAGE_BYTES = A_BYTES + A_LO_BYTES + B_RAW_BYTES;
  // Tiles of 64 rows with three products stack A hi and A lo (adjacent in
  // the stage, rows 64..127 of one N = 128 operand): one MMA per B part and
  // K step, 2 x N = 128 instead of 3 x N = 64, the fourth product lo x lo
  // coming along for free.  The accumulator then has 2 TM columns (hi rows,
  // lo rows), summed by the epilogue.
  // Narrow tiles (64 columns) of up to 128 rows with three products stack by
  // lanes instead (at 256 rows the three M = 64 MMAs measured 1 % faster):
  // B^T hi in TMEM lanes 0..63 and B^T lo in lanes 64..127 make one M = 128
  // operand, so each K step takes two M = 128 MMAs (on A hi and on A lo)
  // instead of three M = 64 ones, and the accumulator's lanes 64 + n (the
  // B-lo sums) are added to lanes n by the epilogue through shared memory.
  static constexpr bool LSTACK = TN == kTNNarrow && NPROD == 3 && TM <= 128;
  static constexpr bool STACK = TM == 64 && NPROD == 3 && !LSTACK;
  static constexpr int MMA_M = LSTACK ? 128 : TN;                   // TMEM lanes of the MMA
  static constexpr int ACC_W = STACK ? 2 * TM : TM;                 // columns per accumulator
  static constexpr int NACC = (TM >= 224 || STACK) ? 1 : 2;         // accumulators in TMEM
  static constexpr int ACC_COLS = NACC * ACC_W;
  static constexpr int BT_COLS = (NPROD == 3 && !LSTACK) ? 2 * BK : BK;   // B^T columns per stage
  static constexpr int XCHG_BYTES = LSTACK ? 64 * 33 * 4 : 0;       // epilogue exchange buffer
  static constexpr int FIT_SMEM = (kSmemLimit - 2048 - XCHG_BYTES) / STAGE_BYTES;
  static constexpr int FIT_TMEM = (kTmemCols - ACC_COLS) / BT_COLS;
  static constexpr int S0 = FIT_SMEM < FIT_TMEM ? FIT_SMEM : FIT_TMEM;
  static constexpr int STAGES = S0 < 8 ? S0 : 8;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 1024 + XCHG_BYTES;
  static constexpr uint32_t A_SWZ_MASK = BK == 32 ? 7u : 3u;       // 128B or 64B swizzle
  static constexpr uint32_t A_LAYOUT = BK == 32 ? 2u : 4u;         // descriptor layout code
  static constexpr uint32_t A_SBO = BK == 32 ? 1024u : 512u;       // 8-row group stride
  static_assert(STAGES >= 2, "at least two stages");
  static_assert(BK == 16 || BK == 32, "BK");
  static_assert(TM == 64 || TM == 128 || TM == 224 || TM == 256, "TM");
  static_assert(A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "1024-byte aligned atoms");
  static_assert(ACC_COLS + STAGES * BT_COLS <= kTmemCols, "TMEM budget");
};

// Byte offset of a swizzled tile element from its plain (row-major in the
// tile) offset: the 16-byte chunk index is XORed with bits 7.. of the offset,
// which is how TMA writes and tcgen05 reads 64B / 128B swizzled tiles.
__device__ __forceinline__ uint32_t swizzle(uint32_t o, uint32_t mask) {
  return o ^ (((o >> 7) & mask) << 4);
}

// Final value of one element of C: the accumulated sum, or with the general
// form alpha * sum + beta * C_old (C_old read only when beta != 0).
__device__ __forceinline__ float scaled_c(float acc, const float* dst, float alpha, float beta) {
  const float r = alpha * acc;
  return beta != 0.0f ? fmaf(beta, *dst, r) : r;
}

// The operand parts the tensor core is given for one fp32 element: with
// three products, hi = the raw bits (read as trunc(x)) and lo = the rounded
// remainder; with one product, hi = x rounded to the nearest TF32 value (B
// always; A on the staged path, which writes the tile anyway).
template <int NPROD>
__device__ __forceinline__ void split_operand(uint32_t x, uint32_t& hi, uint32_t& lo) {
  if (NPROD == 3) {
    hi = x;
    lo = tf32_lo_of_truncated(x);
  } else {
    hi = tf32_round_bits(x);
    lo = 0u;
  }
}

template <int NC>
__device__ __forceinline__ void tmem_store_cols(uint32_t taddr, const uint32_t (&v)[NC]);
template <>
__device__ __forceinline__ void tmem_store_cols<8>(uint32_t taddr, const uint32_t (&v)[8]) {
  tmem_st_8cols(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_store_cols<16>(uint32_t taddr, const uint32_t (&v)[16]) {
  tmem_st_16cols(taddr, v);
}

__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync %0, %1;" ::"r"(kEpilogueBarrier), "r"(kEpilogueThreads) : "memory");
}

// True on every epilogue thread iff `v` is true on all of them (a barrier:
// every epilogue thread reaches it after its own bounded wait, so a wait
// that runs out on some threads and not on others cannot split the group).
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(kEpilogueBarrier), "r"(kEpilogueThreads)
      : "memory");
  return r != 0;
}

template <int TM, int BK, int NPROD, int LOAD, int TN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p,
                   const TcGeneral gp) {
  constexpr bool TMA = LOAD == kLoadTma;
  constexpr bool GEN = LOAD == kLoadStagedGeneral;
  constexpr bool PLAIN_C = LOAD == kLoadStaged;   // C = the sum, row stride N
  const int ldc = PLAIN_C ? p.N : gp.ldc;
  const bool scale = !PLAIN_C && gp.scale;
  const int lda = GEN ? gp.lda : p.K, ldb = GEN ? gp.ldb : p.N;
  const bool trans_a = GEN && gp.trans_a, trans_b = GEN && gp.trans_b;
  using Cfg = TcCfg<TM, BK, NPROD, TN>;
  static_assert(TN == kTN || (TN == kTNNarrow && LOAD == kLoadTma), "narrow tiles: TMA only");
  // extents (elements) of the arrays indexed by hand, for the checked build
  [[maybe_unused]] const size_t a_extent =
      trans_a ? stored_extent(p.K, p.M, lda) : stored_extent(p.M, p.K, lda);
  [[maybe_unused]] const size_t b_extent =
      trans_b ? stored_extent(p.N, p.K, ldb) : stored_extent(p.K, p.N, ldb);
  [[maybe_unused]] const size_t c_extent = stored_extent(p.M, p.N, ldc);
  [[maybe_unused]] const size_t work_extent =
      static_cast<size_t>(p.tiles_m * p.tiles_n - p.dp_tiles) * p.max_seg * (TM * TN);
  constexpr int S = Cfg::STAGES;
  constexpr int NACC = Cfg::NACC;
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t dyn0 = smem_addr(smem_dyn);
  const uint32_t base = (dyn0 + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_dyn + (base - dyn0);
  const uint32_t bars = base + S * Cfg::STAGE_BYTES;
  // barrier map (8 bytes each)
  auto full_bar = [&](int s) { return bars + 8u * s; };              // TMA landed
  auto ready_bar = [&](int s) { return bars + 8u * (S + s); };       // operands split
  auto empty_bar = [&](int s) { return bars + 8u * (2 * S + s); };   // MMAs done with stage
  auto accf_bar = [&](int b) { return bars + 8u * (3 * S + b); };    // accumulator b complete
  auto acce_bar = [&](int b) { return bars + 8u * (3 * S + NACC + b); };  // accumulator b drained
  const uint32_t drain_bar = bars + 8u * (3 * S + 2 * NACC);
  const uint32_t tmem_slot = drain_bar + 8u;
  // split tiles this CTA published last, reduced after the work list
  volatile int* const pending_count = reinterpret_cast<volatile int*>(base_ptr + (tmem_slot + 8u - base));
  WorkItem* const pending = reinterpret_cast<WorkItem*>(base_ptr + (tmem_slot + 16u - base));
  static_assert(8 * (3 * S + 2 * NACC + 2) + 16 + kMaxPending * sizeof(WorkItem) <= 1024,
                "barriers and pending work fit the 1024 bytes after the stages");
  // LSTACK: the epilogue's exchange of B-lo sums, [64 columns][33] floats
  float* const xchg = reinterpret_cast<float*>(base_ptr + S * Cfg::STAGE_BYTES + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *pending_count = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(ready_bar(s), kTransformThreads);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpilogueThreads);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (TMA && warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  grid_launch_dependents();
  grid_dependency_wait();   // global memory from here on

  WorkItem w;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (TMA && lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t armed = 0;    // bit s: stage s was armed at least once
      uint32_t last_ph = 0;  // bit s: parity of the last arming of stage s
      bool ok = true;
      bool first = true;
      WorkList list(p);
      while (ok && list.next(p, w)) {
        const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup);
        for (int kt = w.k0; kt < w.k1; ++kt) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t st = base + s * Cfg::STAGE_BYTES;
          if (p.drop_first_copy && blockIdx.x == 0 && first) {
            // test hook: this stage is never filled, so every role that
            // depends on it runs into its bounded wait
            first = false;
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
            continue;
          }
          first = false;
          mbar_arrive_expect_tx(full_bar(s), Cfg::A_BYTES + Cfg::B_RAW_BYTES);
          armed |= 1u << s;
          last_ph = (last_ph & ~(1u << s)) | (ph << s);
          tma_load_2d(st, &tmA, full_bar(s), kt * BK, c.tm * TM);
          tma_load_2d(st + Cfg::A_BYTES + Cfg::A_LO_BYTES, &tmB, full_bar(s), c.tn * TN, kt * BK);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // copies still in flight must land before the CTA's shared memory goes away
      for (int q = 0; q < S; ++q)
        if (armed & (1u << q)) mbar_wait(full_bar(q), (last_ph >> q) & 1u, p.err, kSiteDrainTma);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(Cfg::MMA_M, Cfg::ACC_W, false, false);
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      WorkList list(p);
      while (ok && list.next(p, w)) {
        if (!mbar_wait(acce_bar(acc), acc_ph ^ 1u, p.err, kSiteMmaAccEmpty)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_W);
        for (int kt = w.k0; kt < w.k1; ++kt) {
          if (!mbar_wait(ready_bar(s), ph, p.err, kSiteMmaReady)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = base + s * Cfg::STAGE_BYTES;
          const uint32_t bt = tmem_base + static_cast<uint32_t>(Cfg::ACC_COLS + s * Cfg::BT_COLS);
#pragma unroll
          for (int kk = 0; kk < BK / 8; ++kk) {
            const uint64_t a_hi = smem_desc(st + kk * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
            mma_tf32_tmem_a(d_tmem, bt + kk * 8, a_hi, idesc, (kt > w.k0 || kk > 0) ? 1u : 0u);
            if (Cfg::LSTACK) {
              // the TMEM operand holds B^T hi and lo in its two lane halves
              const uint64_t a_lo =
                  smem_desc(st + Cfg::A_BYTES + kk * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
              mma_tf32_tmem_a(d_tmem, bt + kk * 8, a_lo, idesc, 1u);
            } else if (Cfg::STACK) {
              // a_hi spans [A hi; A lo] here: B_hi * both, then B_lo * both
              mma_tf32_tmem_a(d_tmem, bt + BK + kk * 8, a_hi, idesc, 1u);
            } else if (NPROD == 3) {
              const uint64_t a_lo =
                  smem_desc(st + Cfg::A_BYTES + kk * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
              mma_tf32_tmem_a(d_tmem, bt + kk * 8, a_lo, idesc, 1u);        // B_hi * A_lo
              mma_tf32_tmem_a(d_tmem, bt + BK + kk * 8, a_hi, idesc, 1u);   // B_lo * A_hi
            }
          }
          mma_commit(empty_bar(s));  // stage s is free once these MMAs finish
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf_bar(acc));   // accumulator complete once all MMAs finish
        if (++acc == NACC) {
          acc = 0;
          acc_ph ^= 1u;
        }
      }
      mma_commit(drain_bar);
      mbar_wait(drain_bar, 0, p.err, kSiteDrainMma);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // this warp may read TMEM lanes 32q .. 32q+31
    // this thread's column within the tile; with narrow tiles of one product
    // only lanes 0-15 of each quarter hold accumulator rows, with LSTACK
    // quarters 2 and 3 hold the B-lo sums of quarters 0 and 1
    const bool live = TN == kTN || (Cfg::LSTACK ? q < 2 : lane < 16);
    const int nl = TN == kTN ? q * 32 + lane
                             : (Cfg::LSTACK ? (q & 1) * 32 + lane : q * 16 + (lane & 15));
    int acc = 0;
    uint32_t acc_ph = 0;
    WorkList list(p);
    while (list.next(p, w)) {
      const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup);
      if (!epilogue_all(mbar_wait(accf_bar(acc), acc_ph, p.err, kSiteEpilogueFull))) break;
      tc_fence_after_sync();
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::ACC_W);
      // rows chunk*32 .. +31 of the tile's accumulator (with STACK the sum of
      // its hi-row and lo-row columns)
      auto load_rows = [&](int chunk, uint32_t (&v)[32]) {
        tmem_ld_32cols(t_acc + chunk * 32, v);
        if constexpr (Cfg::STACK) {
          uint32_t u[32];
          tmem_ld_32cols(t_acc + TM + chunk * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(u[j]));
        } else if constexpr (Cfg::LSTACK) {
          tmem_wait_ld();
          if (q >= 2) {
            float* const row = xchg + ((q - 2) * 32 + lane) * 33;
#pragma unroll
            for (int j = 0; j < 32; ++j) row[j] = __uint_as_float(v[j]);
          }
          epilogue_sync();
          if (q < 2) {
            const float* const row = xchg + (q * 32 + lane) * 33;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + row[j]);
          }
          epilogue_sync();   // the buffer is free for the next chunk
        } else {
          tmem_wait_ld();
        }
      };
      const int n = c.tn * TN + nl;   // this thread's column of C
      const bool n_ok = live && n < p.N;
      if (w.nseg > 1) {
        // part of a split tile: publish this partial; the CTA that publishes
        // last reduces the tile after its work list (see teardown)
        float* const mine = p.partials +
                            (static_cast<size_t>(w.tail) * p.max_seg + w.seg) * (TM * TN) + nl;
#pragma unroll 1
        for (int chunk = 0; chunk < TM / 32; ++chunk) {
          uint32_t v[32];
          load_rows(chunk, v);
          if (live) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (GEMM_IN_EXTENT(mine + (chunk * 32 + j) * TN - p.partials, work_extent, p.err,
                                 kSiteBoundsWork))
                mine[(chunk * 32 + j) * TN] = __uint_as_float(v[j]);
          }
        }
        __threadfence();
        epilogue_sync();
        if (q == 0 && lane == 0 &&
            tail_arrive(p.counters, w.tail) == static_cast<unsigned>(w.nseg)) {
          // only the first and the last item of a CTA's share can be partial
          if (*pending_count < kMaxPending)
            pending[(*pending_count)++] = w;
          else
            record_error(p.err, kSitePendingOverflow);
        }
      } else {
#pragma unroll 1
        for (int chunk = 0; chunk < TM / 32; ++chunk) {
          uint32_t v[32];
          load_rows(chunk, v);
          const int m0 = c.tm * TM + chunk * 32;
          if (n_ok) {
            float* dst = p.C + static_cast<size_t>(m0) * static_cast<size_t>(ldc) + n;
            const int rows = min(32, p.M - m0);
            if (!scale) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < rows && GEMM_IN_EXTENT(dst + static_cast<size_t>(j) * ldc - p.C, c_extent,
                                               p.err, kSiteBoundsC))
                  dst[static_cast<size_t>(j) * ldc] = __uint_as_float(v[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (j < rows &&
                    GEMM_IN_EXTENT(dst + static_cast<size_t>(j) * ldc - p.C, c_extent, p.err,
                                   kSiteBoundsC)) {
                  float* d = dst + static_cast<size_t>(j) * ldc;
                  *d = scaled_c(__uint_as_float(v[j]), d, gp.alpha, gp.beta);
                }
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(acce_bar(acc));
      if (++acc == NACC) {
        acc = 0;
        acc_ph ^= 1u;
      }
    }
  } else if (warp >= kTransformWarp0) {
    // ------------------------------------------------------------ transform
    constexpr int KH = BK / 2;                            // K rows of B per thread
    const int tt = threadIdx.x - kTransformWarp0 * 32;    // 0 .. 255
    const int q = (warp - kTransformWarp0) & 3;           // this warp's TMEM lane quarter
    // this thread's column of the tile (its TMEM lane: 32q + lane); with
    // narrow tiles of one product lanes 16-31 of a quarter are not read by
    // the MMA and carry a copy of lane - 16's column; with LSTACK quarters 2
    // and 3 carry the lo parts of quarters 0 and 1's columns
    const int col = TN == kTN ? q * 32 + lane
                              : (Cfg::LSTACK ? (q & 1) * 32 + lane : q * 16 + (lane & 15));
    const int kh0 = (tt >> 7) * KH;                       // first K row of its half
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    WorkList list(p);
    while (ok && list.next(p, w)) {
      const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup);
      for (int kt = w.k0; kt < w.k1; ++kt) {
        uint8_t* const st = base_ptr + s * Cfg::STAGE_BYTES;
        // the MMAs of this stage's previous round must be done before its
        // TMEM columns are overwritten (implied on the TMA path, cheap to check)
        if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err, kSiteTransformEmpty)) {
          ok = false;
          break;
        }
        if (TMA && !mbar_wait(full_bar(s), ph, p.err, kSiteTransformFull)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t bh[KH], bl[KH];
        if (TMA) {
          // A: three products read the raw tile as the high part; only the
          // low part is written.
          uint4* const hi = reinterpret_cast<uint4*>(st);
          uint4* const lo = reinterpret_cast<uint4*>(st + Cfg::A_BYTES);
          // One product leaves the tile as it is: the tensor core reads it
          // truncated to TF32 (B is rounded to nearest below), which keeps
          // the per-product error under 2^-10 + 2^-11 and saves a read and
          // a write of the tile in shared memory.
          if (NPROD == 3) {
#pragma unroll 4
            for (int i = tt; i < Cfg::A_BYTES / 16; i += kTransformThreads) {
              const uint4 x = hi[i];
              lo[i] = make_uint4(tf32_lo_of_truncated(x.x), tf32_lo_of_truncated(x.y),
                                 tf32_lo_of_truncated(x.z), tf32_lo_of_truncated(x.w));
            }
          }
          // B: column `col` of the raw tile, K rows kh0 .. kh0+KH-1
          const uint32_t* braw =
              reinterpret_cast<const uint32_t*>(st + Cfg::A_BYTES + Cfg::A_LO_BYTES);
#pragma unroll
          for (int k = 0; k < KH; ++k) split_operand<NPROD>(braw[(kh0 + k) * TN + col], bh[k], bl[k]);
        } else {
          const int m0 = c.tm * TM, n0 = c.tn * TN, k0 = kt * BK;
          // This thread's loads for the stage are issued before any of them
          // is used (A in chunks of at most 16, the first with all of B), so
          // a few latencies cover the stage.
          constexpr int AV = TM * BK / kTransformThreads;   // A elements per thread
          constexpr int CH = AV <= 16 ? AV : (KH >= 16 ? 8 : 16);   // within 128 registers
          uint32_t bv[KH];
          const int gn = n0 + col;
#pragma unroll
          for (int c0 = 0; c0 < AV; c0 += CH) {
            uint32_t av[CH];
            // A tile: element e = tt + 256 j is row r, column k of the tile,
            // with lanes along k (or along m when A is stored transposed), so
            // that they read consecutive addresses
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const int e = tt + (c0 + j) * kTransformThreads;
              const int r = trans_a ? e % TM : e / BK, k = trans_a ? e / TM : e % BK;
              const int gm = m0 + r, gk = k0 + k;
              const size_t at = trans_a ? static_cast<size_t>(gk) * lda + gm
                                          : static_cast<size_t>(gm) * lda + gk;
              av[j] = (gm < p.M && gk < p.K &&
                       GEMM_IN_EXTENT(at, a_extent, p.err, kSiteBoundsA))
                          ? __float_as_uint(__ldg(p.A + at))
                          : 0u;
            }
            if (c0 == 0) {
              // B tile: column n0 + col, K rows of this thread's half (lanes along n)
#pragma unroll
              for (int k = 0; k < KH; ++k) {
                const int gk = k0 + kh0 + k;
                const size_t bt_at = trans_b ? static_cast<size_t>(gn) * ldb + gk
                                               : static_cast<size_t>(gk) * ldb + gn;
                bv[k] = (gn < p.N && gk < p.K &&
                         GEMM_IN_EXTENT(bt_at, b_extent, p.err, kSiteBoundsB))
                            ? __float_as_uint(__ldg(p.B + bt_at))
                            : 0u;
              }
            }
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const int e = tt + (c0 + j) * kTransformThreads;
              const int r = trans_a ? e % TM : e / BK, k = trans_a ? e / TM : e % BK;
              uint32_t h, l;
              split_operand<NPROD>(av[j], h, l);
              const uint32_t o = swizzle(static_cast<uint32_t>(r * BK * 4 + k * 4), Cfg::A_SWZ_MASK);
              *reinterpret_cast<uint32_t*>(st + o) = h;
              if (NPROD == 3) *reinterpret_cast<uint32_t*>(st + Cfg::A_BYTES + o) = l;
            }
          }
#pragma unroll
          for (int k = 0; k < KH; ++k) split_operand<NPROD>(bv[k], bh[k], bl[k]);
        }
        const uint32_t bt =
            lane_base + static_cast<uint32_t>(Cfg::ACC_COLS + s * Cfg::BT_COLS + kh0);
        if (Cfg::LSTACK) {
          // lanes 0..63 take B^T hi, lanes 64..127 B^T lo (warp-uniform)
          if (q >= 2)
            tmem_store_cols<KH>(bt, bl);
          else
            tmem_store_cols<KH>(bt, bh);
        } else {
          tmem_store_cols<KH>(bt, bh);
          if (NPROD == 3) tmem_store_cols<KH>(bt + BK, bl);
        }
        tmem_wait_st();
        fence_proxy_async_smem();  // A hi/lo: generic-proxy writes -> tensor-core reads
        tc_fence_before_sync();
        mbar_arrive(ready_bar(s));
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // Split tiles whose last partial this CTA published: every thread of the
  // CTA sums the partials in segment order (fixed, whichever CTA gets here)
  // and writes C.  Many independent 16-byte loads per thread keep the L2
  // reads in flight.  (Written out here rather than through the shared
  // reduce_partials(): measured on GB300, that call made this kernel's
  // mainloop about 8 % slower.)
  const int npend = *pending_count;
  if (npend > 0) {
    __threadfence();
    for (int e = 0; e < npend; ++e) {
      const WorkItem pw = pending[e];
      const TileCoord c = tile_coord(pw.tile, p.tiles_m, p.tiles_n, kRasterGroup);
      const float4* const parts = reinterpret_cast<const float4*>(
          p.partials + static_cast<size_t>(pw.tail) * p.max_seg * (TM * TN));
      constexpr int kVec = TM * TN / 4;           // float4s per partial
      constexpr int kPer = kVec / kThreads;       // per thread
      constexpr int kH = (kPer + 1) / 2;          // per thread and half (the last may be short)
      static_assert(kVec % kThreads == 0, "partial tile shape");
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float4 sum[kH];
#pragma unroll
        for (int i = 0; i < kH; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int sg = 0; sg < pw.nseg; ++sg) {
          float4 x[kH];
#pragma unroll
          for (int i = 0; i < kH; ++i) {
            if (half * kH + i >= kPer) {
              x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              continue;
            }
            const size_t f4 = static_cast<size_t>(sg) * kVec + threadIdx.x +
                              (half * kH + i) * kThreads;
            x[i] = GEMM_IN_EXTENT(
                       4 * (f4 + (parts - reinterpret_cast<const float4*>(p.partials))) + 3,
                       work_extent, p.err, kSiteBoundsWork)
                       ? __ldcg(parts + f4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < kH; ++i) {
            sum[i].x += x[i].x;
            sum[i].y += x[i].y;
            sum[i].z += x[i].z;
            sum[i].w += x[i].w;
          }
        }
#pragma unroll
        for (int i = 0; i < kH; ++i) {
          if (half * kH + i >= kPer) continue;
          const int f = threadIdx.x + (half * kH + i) * kThreads;  // float4 index
          const int m = c.tm * TM + f / (TN / 4);
          const int n = c.tn * TN + (f % (TN / 4)) * 4;
          if (m < p.M) {
            float* dst = p.C + static_cast<size_t>(m) * static_cast<size_t>(ldc) + n;
            const float vals[4] = {sum[i].x, sum[i].y, sum[i].z, sum[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (n + q < p.N &&
                  GEMM_IN_EXTENT(dst + q - p.C, c_extent, p.err, kSiteBoundsC))
                dst[q] = scale ? scaled_c(vals[q], dst + q, gp.alpha, gp.beta) : vals[q];
          }
        }
      }
    }
  }
  if (p.sk_ctas > 0 && threadIdx.x == 0) tail_launch_done(p.counters);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      (void)cudaGetLastError();
  });
  return g_encode;
}

}  // namespace

// 2-D fp32 map of a row-major [rows x cols] matrix with row stride ld
// (elements), box [box_rows x box_cols]; out-of-bounds boxes read as zero.
bool tma_encode_2d(CUtensorMap* map, const float* ptr, int rows, int cols, int ld, int box_cols,
               int box_rows, CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4u};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

constexpr int kMaxDevices = 64;

template <int TM, int BK, int NPROD, int LOAD, int TN = kTN>
int launch_one(const GemmArgs& g, const TcParams& p, const TcGeneral& gp, const CUtensorMap& ma,
               const CUtensorMap& mb, int grid, cudaStream_t stream) {
  using Cfg = TcCfg<TM, BK, NPROD, TN>;
  static std::atomic<unsigned long long> configured{0};  // bit per device
  auto kern = tc_gemm_kernel<TM, BK, NPROD, LOAD, TN>;
  const unsigned long long bit = 1ull << (g.device % kMaxDevices);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return GEMM_F32_ELAUNCH;
    }
    configured.fetch_or(bit);
  }
  if (launch_dependent(kern, dim3(grid), dim3(kThreads), Cfg::SMEM, stream, ma, mb, p, gp) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  return GEMM_F32_OK;
}

template <int BK, int NPROD, int LOAD, int TN = kTN>
int launch_tm(int tm, const GemmArgs& g, const TcParams& p, const TcGeneral& gp,
              const CUtensorMap& ma, const CUtensorMap& mb, int grid, cudaStream_t stream) {
  switch (tm) {
    case 64: return launch_one<64, BK, NPROD, LOAD, TN>(g, p, gp, ma, mb, grid, stream);
    case 128: return launch_one<128, BK, NPROD, LOAD, TN>(g, p, gp, ma, mb, grid, stream);
    case 224:
      if constexpr (LOAD == kLoadTma)
        return launch_one<224, BK, NPROD, LOAD, TN>(g, p, gp, ma, mb, grid, stream);
      return GEMM_F32_EINVAL;
    default: return launch_one<256, BK, NPROD, LOAD, TN>(g, p, gp, ma, mb, grid, stream);
  }
}

// Tile heights 64 and 128 are also built with BK = 32 for three products:
// fewer, larger stages (the MMA thread's wait on a stage costs about as much
// as the stage's MMAs at these heights).
template <int NPROD, int LOAD, int TN = kTN>
int launch_tm_bk(int tm, int bk, const GemmArgs& g, const TcParams& p, const TcGeneral& gp,
                 const CUtensorMap& ma, const CUtensorMap& mb, int grid, cudaStream_t stream) {
  if (NPROD == 1) {
    if constexpr (LOAD != kLoadTma)
      if (bk == 16) return launch_tm<16, 1, LOAD, TN>(tm, g, p, gp, ma, mb, grid, stream);
    return launch_tm<32, 1, LOAD, TN>(tm, g, p, gp, ma, mb, grid, stream);
  }
  // three products take 16-deep stages only with 224- and 256-row tiles (bk_for)
  if (bk == 16) {
    if constexpr (LOAD == kLoadTma)
      if (tm == 224) return launch_one<224, 16, 3, LOAD, TN>(g, p, gp, ma, mb, grid, stream);
    return tm == 256 ? launch_one<256, 16, 3, LOAD, TN>(g, p, gp, ma, mb, grid, stream)
                     : GEMM_F32_EINVAL;
  }
  return tm == 64 ? launch_one<64, 32, 3, LOAD, TN>(g, p, gp, ma, mb, grid, stream)
                  : launch_one<128, 32, 3, LOAD, TN>(g, p, gp, ma, mb, grid, stream);
}

// The loader for a launch: TMA when the operands allow, else the staged
// loads of the plain product or of the general form.
template <int NPROD>
int launch_loader(bool tma, int tm, int bk, const GemmArgs& g, const TcParams& p,
                  const TcGeneral& gp, const CUtensorMap& ma, const CUtensorMap& mb, int grid,
                  cudaStream_t stream) {
  if (tma) return launch_tm_bk<NPROD, kLoadTma>(tm, bk, g, p, gp, ma, mb, grid, stream);
  if (plain_form(g))
    return launch_tm_bk<NPROD, kLoadStaged>(tm, bk, g, p, gp, ma, mb, grid, stream);
  return launch_tm_bk<NPROD, kLoadStagedGeneral>(tm, bk, g, p, gp, ma, mb, grid, stream);
}

// K depth of a stage.  Three products: 32 at tile heights up to 128, 16 at
// 256 (where 32 would leave room for two stages only).  One product: 32 on
// the TMA path, 16 on the staged one (measured on GB300: 1.4x faster there,
// the per-thread loads of a 32-deep stage waiting far longer on memory).
int bk_for(int nprod, int tm, bool tma) {
  if (nprod == 1) return tma ? 32 : 16;
  return tm <= 128 ? 32 : 16;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

TcGeneral general_of(const GemmArgs& g) {
  TcGeneral gp;
  gp.lda = g.lda;
  gp.ldb = g.ldb;
  gp.ldc = g.ldc;
  gp.trans_a = g.trans_a;
  gp.trans_b = g.trans_b;
  gp.alpha = g.alpha;
  gp.beta = g.beta;
  gp.scale = g.scale;
  return gp;
}

// Tile height TM.  With the split tail the schedule no longer quantises to
// whole waves, so the most efficient height is used (256; 128 or 64 when M
// is that small).  Without it (too few K iterations to split, ONE_TILE_PER_CTA
// or NO_SPLIT_K), the height whose schedule gives the busiest SM the least
// time: rounds of tiles x TM / (relative efficiency), the efficiencies being
// measured throughputs of TM = 224, 128 and 64 relative to TM = 256: 8192^3
// for tiles 128 columns wide, 65536 x 1024 x 64 and 131072 x 1024 x 64 for
// narrow ones (where 128-row tiles cost 4 % more per row than 256-row ones).
// 224-row tiles exist on the TMA path only; they turn 1.68 waves of 256-row
// tiles (65536 rows on 152 SMs) into two nearly full ones.
int choose_tm(const GemmArgs& g, bool split_tail, int width, bool tma) {
  if (g.flags & GEMM_F32_FLAG_TILE64) return 64;
  if (g.flags & GEMM_F32_FLAG_TILE128) return 128;
  if (g.flags & GEMM_F32_FLAG_TILE224) return tma ? 224 : 256;
  if (g.flags & GEMM_F32_FLAG_TILE256) return 256;
  if (split_tail) return g.M <= 64 ? 64 : (g.M <= 128 ? 128 : 256);
  const long tn = ceil_div(g.N, width);
  long best_cost = -1;
  int best = 256;
  const int tms[4] = {256, 224, 128, 64};
  const long wide_pct[4] = {100, 98, 81, 56}, narrow_pct[4] = {100, 98, 96, 51};
  const long* const eff_pct = width == kTN ? wide_pct : narrow_pct;
  for (int i = 0; i < 4; ++i) {
    if (tms[i] == 224 && !tma) continue;
    const long tiles = tn * ceil_div(g.M, tms[i]);
    const long rounds = (tiles + g.num_sms - 1) / g.num_sms;
    const long cost = rounds * tms[i] * 100 / eff_pct[i];
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = tms[i];
    }
  }
  return best;
}

// A shorter tile height that fills one wave without splitting K, when the
// tallest tiles would leave SMs idle and K is short enough that the split's
// fixed cost matters: measured on GB300, 1536^3 runs 33 us in 144 tiles of
// 128 rows against 43 us in 72 tiles of 256 split along K, while at K = 4096
// the split of 256-row tiles wins (1536 x 1536 x 4096: 69 against 82 us).
// Returns 0 when the usual choice stands (or a flag fixes the height).
constexpr int kOneWaveMaxK = 2048;

int one_wave_height(const GemmArgs& g, int tn) {
  if (g.flags & (GEMM_F32_FLAG_TILE64 | GEMM_F32_FLAG_TILE128 | GEMM_F32_FLAG_TILE224 |
                 GEMM_F32_FLAG_TILE256 | GEMM_F32_FLAG_ONE_TILE_PER_CTA))
    return 0;
  if (g.K > kOneWaveMaxK) return 0;
  const long tiles_n = ceil_div(g.N, tn);
  if (g.M <= 128 || tiles_n * ceil_div(g.M, 256) >= g.num_sms) return 0;
  for (int tm : {128, 64}) {
    const long tiles = tiles_n * ceil_div(g.M, tm);
    if (4 * tiles >= 3L * g.num_sms && tiles <= g.num_sms) return tm;
  }
  return 0;
}

}  // namespace

// Least K iterations per CTA in a split tail that follows at least one full
// wave of whole tiles.
constexpr int kMinSplitItersMultiWave = 64;

// Where a launch's split-tail scratch comes from: the library's workspace
// for the stream (allocated on first use), or, for gemm_f32_noalloc, a
// fixed region that is never grown.
struct TailScratch {
  void* fixed = nullptr;    // non-null: this region of fixed_bytes, no allocation
  size_t fixed_bytes = 0;
};

// One launch with tiles `tn` columns wide (kTN, or kTNNarrow on the TMA
// path only: returns kRetryWide, having launched nothing, when TMA cannot be
// used after all).  With a fixed scratch region, a split tail that needs
// more than it holds returns GEMM_F32_ESCRATCH, having launched nothing.
constexpr int kRetryWide = 1;

int launch_tc_tn(GemmArgs& g, int nprod, int tn, const TailScratch& scratch, cudaStream_t stream,
                 int* launches) {
  *launches = 0;
  int bk = 0;
  TcParams p;
  p.A = g.A;
  p.B = g.B;
  p.C = g.C;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles_n = ceil_div(g.N, tn);
  p.drop_first_copy = (g.flags & GEMM_F32_FLAG_TEST_DROP_COPY) ? 1 : 0;
  p.err = g.err;
  const TcGeneral gp = general_of(g);
  p.partials = nullptr;
  p.counters = nullptr;
  p.sk_ctas = 0;
  p.sk_work = 0;
  p.max_seg = 1;

  // TMA when the operands allow (it decides the stage depth of one product)
  const bool tma_ok = !(g.flags & GEMM_F32_FLAG_FORCE_STAGED) && tma_addressable(g);

  // Split tail when it applies (with the tallest useful tile); otherwise
  // whole tiles with the height that best fills the waves.
  int tm = 0;
  size_t ws_bytes = 0;
  const int one_wave_tm = one_wave_height(g, tn);
  if (!one_wave_tm && !(g.flags & (GEMM_F32_FLAG_ONE_TILE_PER_CTA | GEMM_F32_FLAG_NO_SPLIT_K))) {
    tm = choose_tm(g, true, tn, tma_ok);
    bk = bk_for(nprod, tm, tma_ok);
    p.k_iters = ceil_div(g.K, bk);
    p.tiles_m = ceil_div(g.M, tm);
    const long tiles = static_cast<long>(p.tiles_m) * p.tiles_n;
    if (tiles <= 0x7fffffffL)
      ws_bytes = plan_split_tail(p, tiles, g.num_sms, static_cast<size_t>(tm) * tn * sizeof(float),
                                 tiles >= g.num_sms ? kMinSplitItersMultiWave : kMinSplitIters);
  }
  void* ws = nullptr;
  if (ws_bytes) {
    if (scratch.fixed) {
      if (ws_bytes > scratch.fixed_bytes) return GEMM_F32_ESCRATCH;
      ws = scratch.fixed;
    } else {
      ws = acquire_workspace(g.device, stream, ws_bytes);
    }
  }
  if (!ws) {
    tm = one_wave_tm ? one_wave_tm : choose_tm(g, false, tn, tma_ok);
    bk = bk_for(nprod, tm, tma_ok);
    p.k_iters = ceil_div(g.K, bk);
    p.tiles_m = ceil_div(g.M, tm);
    p.sk_ctas = 0;
    p.sk_work = 0;
    p.max_seg = 1;
  }
  const long tiles = static_cast<long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fffffffL) return GEMM_F32_EINVAL;
  int grid;
  if (ws) {
    grid = g.num_sms;
    p.counters = static_cast<unsigned long long*>(ws);
    p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
  } else {
    p.dp_tiles = static_cast<int>(tiles);
    grid = (g.flags & GEMM_F32_FLAG_ONE_TILE_PER_CTA)
               ? static_cast<int>(tiles)
               : static_cast<int>(std::min<long>(tiles, g.num_sms));
  }

  // TMA needs 16-byte aligned bases and row strides (K % 4 == 0, N % 4 == 0);
  // if the maps cannot be made after all, the staged loader runs with the
  // stage depth already planned (both depths exist for it).
  bool tma = tma_ok;
  alignas(64) CUtensorMap ma, mb;
  if (tma) {
    tma = tma_encode_2d(&ma, g.A, g.M, g.K, g.lda, bk, tm,
                    bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) &&
          tma_encode_2d(&mb, g.B, g.K, g.N, g.ldb, tn, bk, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!tma) {
    if (tn != kTN) return kRetryWide;
    memset(&ma, 0, sizeof(ma));
    memset(&mb, 0, sizeof(mb));
  }
  int rc;
  if (tn == kTNNarrow)
    rc = nprod == 3
             ? launch_tm_bk<3, kLoadTma, kTNNarrow>(tm, bk, g, p, gp, ma, mb, grid, stream)
             : launch_tm_bk<1, kLoadTma, kTNNarrow>(tm, bk, g, p, gp, ma, mb, grid, stream);
  else
    rc = nprod == 3 ? launch_loader<3>(tma, tm, bk, g, p, gp, ma, mb, grid, stream)
                    : launch_loader<1>(tma, tm, bk, g, p, gp, ma, mb, grid, stream);
  if (rc == GEMM_F32_OK) {
    *launches += 1;
    g.kernel = "tc_gemm_kernel";
  }
  return rc;
}

// The single-CTA kernel for a problem: tiles 64 columns wide for N <= 64 on
// the TMA path, so that no MMA work is spent on columns beyond N (measured on
// GB300: 65536 x 1024 x 64 had the tensor pipe 79 % busy with half of each
// M = 128 MMA discarded), 128 columns otherwise.
int launch_tc_single(GemmArgs& g, int nprod, const TailScratch& scratch, cudaStream_t stream,
                     int* launches) {
  if (g.N <= kTNNarrow && !(g.flags & GEMM_F32_FLAG_FORCE_STAGED) && tma_addressable(g)) {
    const int rc = launch_tc_tn(g, nprod, kTNNarrow, scratch, stream, launches);
    if (rc != kRetryWide) return rc;
  }
  return launch_tc_tn(g, nprod, kTN, scratch, stream, launches);
}

int launch_tc_kernels(GemmArgs& g, int nprod, cudaStream_t stream, int* launches);

int launch_tc(GemmArgs& g, int nprod, cudaStream_t stream, int* launches) {
  // operands TMA cannot read, in a large product: copy them first (measured
  // on GB300, the staged loads run at about half the TMA path's speed)
  int packs = 0;
  const int prc = pack_for_tma(g, stream, &packs);
  if (prc != GEMM_F32_OK) return prc;
  const int rc = launch_tc_kernels(g, nprod, stream, launches);
  if (rc == GEMM_F32_OK) *launches += packs;
  return rc;
}

int launch_tc_kernels(GemmArgs& g, int nprod, cudaStream_t stream, int* launches) {
  // Below a wave of pair tiles the single-SM kernel is faster in both modes
  // (measured on GB300, one product, CUDA-graph replay: 2048^3 25.2 against
  // 28.8 us; M = 1001, K = 777, N = 513 15.9 against 21.7 us; M = N = 1024,
  // K = 8192 42.1 against 46.6 us).
  if (tc_pair_suits(g, nprod)) return launch_tc_pair(g, nprod, stream, launches);
  return launch_tc_single(g, nprod, TailScratch(), stream, launches);
}

// ---------------------------------------------------------------- fixed-scratch variant
// The split tail's scratch (tile counters and partial tiles) for
// gemm_f32_noalloc, compiled into the library instead of allocated: every
// device that loads this module holds these bytes until the process exits.
// All calls on a device share it, so calls that overlap on the GPU race.
// Being zero at load, its tile counters start in a valid state; afterwards
// they keep themselves valid (generation scheme, device_common.cuh).
static __device__ __align__(256) unsigned char g_fixed_scratch[GEMM_F32_NOALLOC_SCRATCH_BYTES];

void* fixed_scratch_address() {
  // In host code g_fixed_scratch only names the array: its device address on
  // the current device is asked of the runtime.  Under lazy module loading
  // this loads this file's module (and so places the array) if it was not
  // loaded yet.
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_fixed_scratch) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return ptr;
}

int launch_tc_fixed_scratch(GemmArgs& g, int nprod, void* scratch, cudaStream_t stream,
                            int* launches) {
  *launches = 0;
  if (!scratch) return GEMM_F32_EDEVICE;
  TailScratch fixed;
  fixed.fixed = scratch;
  fixed.fixed_bytes = GEMM_F32_NOALLOC_SCRATCH_BYTES;
  return launch_tc_single(g, nprod, fixed, stream, launches);
}

}  // namespace gemm_f32_impl
