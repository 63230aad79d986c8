// Tensor-core FP32 GEMM on CTA pairs (tcgen05 cta_group::2) for sm_103a.
//
// Same product and the same 3xTF32 / 1xTF32 arithmetic as tc_gemm.cu
// (C[i][j] = sum_k A[i][k] * B[k][j], row-major; "LeetGPU problem 2: matrix
// multiplication", yekq.top, section "problem statement"), but each output
// tile of 256 columns of C by 256 rows is computed by a cluster of two CTAs
// on two SMs with one M = 256 MMA issued by the even CTA:
//   - CTA r holds columns n0 + 128 r .. +127 of the tile: the transposed B
//     tile's TF32 parts in its tensor memory (the MMA's A operand, 128
//     lanes per CTA) and that half of the accumulator (128 lanes x 256
//     columns = all 256 rows of C);
//   - CTA r holds rows m0 + 128 r .. +127 of the A tile in shared memory
//     (the MMA's B operand is split by rows across the pair, and the pair's
//     tensor cores exchange the halves).
// Against one CTA per 128 x 256 tile, every SM reads half as much of the A
// tile from L2 and its shared memory serves half as many MMA operand bytes.
//
// Roles per CTA: warp 0 TMA producer (own halves); warp 1 TMEM allocation
// (both CTAs, cta_group::2) and MMA issue (even CTA only); warps 2, 3, 16
// and 17 forward finished stages to the even CTA; warps 4..7 epilogue (own
// accumulator half); warps 8..15 transform (own halves).  The even CTA's MMA
// waits for both CTAs' stages (one cluster-scope arrive per CTA and stage)
// and for both epilogues to drain the accumulator; its commits arrive on
// both CTAs' barriers (multicast).  Waits are bounded as in
// tc_gemm.cu; the split tail of the last wave works per CTA half.  Where TMA
// cannot address the operands the transform warps load them (LOAD selects
// the plain product's loads or the general form's, as in tc_gemm.cu), with
// stages 16 deep.
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

constexpr int kHalf = 128;                   // rows of A / columns of C per CTA
constexpr int kPairTile = 256;               // the pair's tile: 256 x 256
constexpr int kWarps = 18;                   // 16 + two more forwarding warps
constexpr int kThreads = kWarps * 32;
constexpr int kForwarders = 4;               // warps 2, 3, 16, 17
constexpr int kEpilogueWarp0 = 4;
constexpr int kTransformWarp0 = 8;
constexpr int kTransformWarps = 8;
constexpr int kEpilogueWarps = 4;
constexpr int kEpilogueBarrier = 1;
constexpr int kSmemLimit = 232448;
constexpr int kTmemCols = 512;
constexpr int kRasterGroup = 8;
constexpr int kMaxPending = 8;

struct PairParams {
  const float* A;
  const float* B;
  float* C;
  int M, N, K;
  int tiles_m, tiles_n, k_iters;     // tiles of 256 x 256
  int dp_tiles, sk_ctas;             // split-tail plan over CTA pairs
  long long sk_work;
  int max_seg;
  float* partials;                   // [tail][max_seg][2][256 m][128 n]
  unsigned long long* counters;      // [tail][2]: generation and partials published
  int drop_first_copy;
  unsigned* err;
};

// The general form (see tc_gemm.cu): a separate kernel argument.
struct PairGeneral {
  int lda, ldb, ldc;
  int trans_a, trans_b;
  float alpha, beta;
  int scale;
};

// alpha * acc (+ beta * C_old, read only when beta != 0).
__device__ __forceinline__ float pair_scaled_c(float acc, const float* dst, float alpha,
                                              float beta) {
  const float r = alpha * acc;
  return beta != 0.0f ? fmaf(beta, *dst, r) : r;
}

template <int BK, int NPROD>
struct PairCfg {
  static constexpr int A_BYTES = kHalf * BK * 4;
  static constexpr int A_LO_BYTES = NPROD == 3 ? A_BYTES : 0;
  static constexpr int B_RAW_BYTES = BK * kHalf * 4;
  static constexpr int STAGE_BYTES = A_BYTES + A_LO_BYTES + B_RAW_BYTES;
  static constexpr int ACC_COLS = kPairTile;                       // one accumulator
  static constexpr int BT_COLS = BK * (NPROD == 3 ? 2 : 1);
  static constexpr int FIT_SMEM = (kSmemLimit - 2048) / STAGE_BYTES;
  static constexpr int FIT_TMEM = (kTmemCols - ACC_COLS) / BT_COLS;
  static constexpr int S0 = FIT_SMEM < FIT_TMEM ? FIT_SMEM : FIT_TMEM;
  static constexpr int STAGES = S0 < 8 ? S0 : 8;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 1024;
  static constexpr uint32_t A_SWZ_MASK = BK == 32 ? 7u : 3u;
  static constexpr uint32_t A_LAYOUT = BK == 32 ? 2u : 4u;
  static constexpr uint32_t A_SBO = BK == 32 ? 1024u : 512u;
  static_assert(STAGES >= 2, "at least two stages");
  static_assert(A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "1024-byte aligned atoms");
  static_assert(ACC_COLS + STAGES * BT_COLS <= kTmemCols, "TMEM budget");
};

// ---------------------------------------------------------------- pair primitives
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Non-blocking test: the waits below spin on it, since a blocking try_wait
// on a barrier that another SM arrives on was measured to wake late.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait on a barrier that threads of the other CTA arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, unsigned* err,
                                                  unsigned site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitBudgetNs) {
      record_error(err, site);
      return false;
    }
  }
}


__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (both CTAs' TMEM) (+)= A (both CTAs' TMEM lanes) * B (rows split across
// both CTAs' shared memory).  Issued by the even CTA.
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The barrier at `bar` in both CTAs receives one arrive once the MMAs this
// thread issued before have completed.
__device__ __forceinline__ void mma_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ uint32_t swizzle(uint32_t o, uint32_t mask) {
  return o ^ (((o >> 7) & mask) << 4);
}

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
  asm volatile("bar.sync %0, %1;" ::"r"(kEpilogueBarrier), "r"(kEpilogueWarps * 32) : "memory");
}

__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(kEpilogueBarrier), "r"(kEpilogueWarps * 32)
      : "memory");
  return r != 0;
}

// The work list of a CTA pair: as WorkList, with the pair as the unit.
struct PairWorkList {
  int unit, units, next_dp;
  long long x, x_end;

  __device__ __forceinline__ explicit PairWorkList(const PairParams& p) {
    unit = static_cast<int>(blockIdx.x >> 1);
    units = static_cast<int>(gridDim.x >> 1);
    next_dp = unit;
    x = x_end = 0;
    if (unit < p.sk_ctas) {
      x = sk_start(unit, p.sk_ctas, p.sk_work);
      x_end = sk_start(unit + 1, p.sk_ctas, p.sk_work);
    }
  }

  __device__ __forceinline__ bool next(const PairParams& p, WorkItem& w) {
    if (next_dp < p.dp_tiles) {
      w.tile = next_dp;
      w.k0 = 0;
      w.k1 = p.k_iters;
      w.tail = -1;
      w.seg = 0;
      w.nseg = 1;
      // Odd waves walk K backwards: they start on the K slices the previous
      // wave read last, which are still in L2, and the A row panels a wave
      // shares with the one before it are then read mostly from L2.
      w.rev = ((next_dp / units) & 1) != 0;
      next_dp += units;
      return true;
    }
    if (x < x_end) {
      const long long ki = p.k_iters;
      const int i = static_cast<int>(x / ki);
      w.tile = p.dp_tiles + i;
      w.tail = i;
      w.k0 = static_cast<int>(x - i * ki);
      w.k1 = static_cast<int>(min(ki, w.k0 + (x_end - x)));
      const int first = sk_owner(i * ki, p.sk_ctas, p.sk_work);
      const int last = sk_owner((i + 1) * ki - 1, p.sk_ctas, p.sk_work);
      w.seg = unit - first;
      w.nseg = last - first + 1;
      w.rev = false;
      x += w.k1 - w.k0;
      return true;
    }
    return false;
  }
};

template <int BK, int NPROD, int LOAD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const PairParams p, const PairGeneral gp) {
  constexpr bool TMA = LOAD == kLoadTma;
  constexpr bool GEN = LOAD == kLoadStagedGeneral;
  constexpr bool PLAIN_C = LOAD == kLoadStaged;   // C = the sum, row stride N
  const int ldc = PLAIN_C ? p.N : gp.ldc;
  const bool scale = !PLAIN_C && gp.scale;
  const int lda = GEN ? gp.lda : p.K, ldb = GEN ? gp.ldb : p.N;
  const bool trans_a = GEN && gp.trans_a, trans_b = GEN && gp.trans_b;
  using Cfg = PairCfg<BK, NPROD>;
  constexpr int S = Cfg::STAGES;
  // extents (elements) of the arrays indexed by hand, for the checked build
  [[maybe_unused]] const size_t a_extent =
      trans_a ? stored_extent(p.K, p.M, lda) : stored_extent(p.M, p.K, lda);
  [[maybe_unused]] const size_t b_extent =
      trans_b ? stored_extent(p.N, p.K, ldb) : stored_extent(p.K, p.N, ldb);
  [[maybe_unused]] const size_t c_extent = stored_extent(p.M, p.N, ldc);
  [[maybe_unused]] const size_t work_extent =
      static_cast<size_t>(p.tiles_m * p.tiles_n - p.dp_tiles) * p.max_seg * 2 * (kPairTile * kHalf);
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t dyn0 = smem_addr(smem_dyn);
  const uint32_t base = (dyn0 + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_dyn + (base - dyn0);
  const uint32_t bars = base + S * Cfg::STAGE_BYTES;
  auto full_bar = [&](int s) { return bars + 8u * s; };              // own TMA landed
  auto ready_bar = [&](int s) { return bars + 8u * (S + s); };       // both CTAs split (even CTA's)
  auto empty_bar = [&](int s) { return bars + 8u * (2 * S + s); };   // pair MMAs done with stage
  auto done_bar = [&](int s) { return bars + 8u * (3 * S + s); };    // own transform finished stage
  const uint32_t accf_bar = bars + 8u * (4 * S);                     // accumulator complete
  const uint32_t acce_bar = bars + 8u * (4 * S + 1);                 // both halves drained (even CTA's)
  const uint32_t drain_bar = bars + 8u * (4 * S + 2);
  const uint32_t tmem_slot = bars + 8u * (4 * S + 3);
  volatile int* const pending_count =
      reinterpret_cast<volatile int*>(base_ptr + (tmem_slot + 8u - base));
  WorkItem* const pending = reinterpret_cast<WorkItem*>(base_ptr + (tmem_slot + 16u - base));
  static_assert(8 * (4 * S + 3) + 16 + kMaxPending * sizeof(WorkItem) <= 1024 - 16,
                "barriers and pending work fit the 1024 bytes after the stages");
  // the clock record's start mark: the last 16 bytes of that region
  unsigned long long(&clk_mark)[2] =
      *reinterpret_cast<unsigned long long(*)[2]>(base_ptr + (bars + 1008u - base));
  clock_start(clk_mark);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();

  if (threadIdx.x == 0) {
    *pending_count = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(ready_bar(s), 2);   // one arrive per CTA (from its forwarding warp)
      mbar_init(empty_bar(s), 1);
      mbar_init(done_bar(s), kTransformWarps * 32);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, 2 * kEpilogueWarps);
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  if (TMA && warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();      // barriers of both CTAs exist before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  grid_launch_dependents();
  grid_dependency_wait();   // global memory from here on

  WorkItem w;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (own halves)
    if (TMA && lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t armed = 0, last_ph = 0;
      bool ok = true, first = true;
      PairWorkList list(p);
      while (ok && list.next(p, w)) {
        const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup, true);
        for (int kt = w.k0; kt < w.k1; ++kt) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t st = base + s * Cfg::STAGE_BYTES;
          if (p.drop_first_copy && blockIdx.x == 0 && first) {
            first = false;   // test hook: this stage is never filled
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
          const int kc = k_tile_at(w, kt) * BK;
          tma_load_2d(st, &tmA, full_bar(s), kc, c.tm * kPairTile + static_cast<int>(rank) * kHalf);
          tma_load_2d(st + Cfg::A_BYTES + Cfg::A_LO_BYTES, &tmB, full_bar(s),
                      c.tn * kPairTile + static_cast<int>(rank) * kHalf, kc);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      for (int q = 0; q < S; ++q)
        if (armed & (1u << q)) mbar_wait(full_bar(q), (last_ph >> q) & 1u, p.err, kSiteDrainTma);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(2 * kHalf, kPairTile, false, false);
      int s = 0;
      uint32_t ph = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      PairWorkList list(p);
      while (ok && list.next(p, w)) {
        if (!mbar_wait_cluster(acce_bar, acc_ph ^ 1u, p.err, kSiteMmaAccEmpty)) break;
        tc_fence_after_sync();
        for (int kt = w.k0; kt < w.k1; ++kt) {
          if (!mbar_wait_cluster(ready_bar(s), ph, p.err, kSiteMmaReady)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = base + s * Cfg::STAGE_BYTES;
          const uint32_t bt = tmem_base + static_cast<uint32_t>(Cfg::ACC_COLS + s * Cfg::BT_COLS);
#pragma unroll
          for (int kk = 0; kk < BK / 8; ++kk) {
            const uint64_t a_hi = smem_desc(st + kk * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
            mma_pair(tmem_base, bt + kk * 8, a_hi, idesc, (kt > w.k0 || kk > 0) ? 1u : 0u);
            if (NPROD == 3) {
              const uint64_t a_lo =
                  smem_desc(st + Cfg::A_BYTES + kk * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
              mma_pair(tmem_base, bt + kk * 8, a_lo, idesc, 1u);
              mma_pair(tmem_base, bt + BK + kk * 8, a_hi, idesc, 1u);
            }
          }
          mma_commit_both(empty_bar(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_both(accf_bar);
        acc_ph ^= 1u;
      }
      mma_commit_local(drain_bar);
      mbar_wait(drain_bar, 0, p.err, kSiteDrainMma);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3 || warp >= 16) {
    // ------------------------------------------------------------ forwarders
    // A cluster-scope release arrive takes about as long as a stage of MMAs
    // when the arriving thread has just written the stage; these warps, with
    // nothing of their own to publish, pass each stage's completion on to the
    // even CTA (stage i by forwarder i mod 4) off the transform path.
    if (lane == 0) {
      const uint32_t leader_ready0 = map_rank(ready_bar(0), 0);
      const uint32_t mine = static_cast<uint32_t>(warp < 16 ? warp - 2 : warp - 14);
      int s = 0;
      uint32_t ph = 0, count = 0;
      bool ok = true;
      PairWorkList list(p);
      while (ok && list.next(p, w)) {
        for (int kt = w.k0; kt < w.k1; ++kt, ++count) {
          if (count % kForwarders == mine) {
            if (!mbar_wait(done_bar(s), ph, p.err, kSiteTransformFull)) {
              ok = false;
              break;
            }
            mbar_arrive_cluster(leader_ready0 + 8u * s);
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + kEpilogueWarps) {
    // ------------------------------------------------------------ epilogue (own half)
    const int q = warp & 3;
    const int nl = q * 32 + lane;
    const uint32_t leader_acce = map_rank(acce_bar, 0);
    uint32_t acc_ph = 0;
    PairWorkList list(p);
    while (list.next(p, w)) {
      const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup, true);
      if (!epilogue_all(mbar_wait(accf_bar, acc_ph, p.err, kSiteEpilogueFull))) break;
      tc_fence_after_sync();
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int n = c.tn * kPairTile + static_cast<int>(rank) * kHalf + nl;
      const bool n_ok = n < p.N;
      if (w.nseg > 1) {
        float* const mine =
            p.partials +
            ((static_cast<size_t>(w.tail) * p.max_seg + w.seg) * 2 + rank) * (kPairTile * kHalf) + nl;
#pragma unroll 1
        for (int chunk = 0; chunk < kPairTile / 32; ++chunk) {
          uint32_t v[32];
          tmem_ld_32cols(t_acc + chunk * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (GEMM_IN_EXTENT(mine + (chunk * 32 + j) * kHalf - p.partials, work_extent, p.err,
                               kSiteBoundsWork))
              mine[(chunk * 32 + j) * kHalf] = __uint_as_float(v[j]);
        }
        __threadfence();
        epilogue_sync();
        if (nl == 0 &&
            tail_arrive(p.counters, 2 * w.tail + static_cast<int>(rank)) ==
                static_cast<unsigned>(w.nseg)) {
          if (*pending_count < kMaxPending)
            pending[(*pending_count)++] = w;
          else
            record_error(p.err, kSitePendingOverflow);
        }
      } else {
#pragma unroll 1
        for (int chunk = 0; chunk < kPairTile / 32; ++chunk) {
          uint32_t v[32];
          tmem_ld_32cols(t_acc + chunk * 32, v);
          tmem_wait_ld();
          const int m0 = c.tm * kPairTile + chunk * 32;
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
                  *d = pair_scaled_c(__uint_as_float(v[j]), d, gp.alpha, gp.beta);
                }
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_acce);
      acc_ph ^= 1u;
    }
  } else if (warp >= kTransformWarp0 && warp < kTransformWarp0 + kTransformWarps) {
    // ------------------------------------------------------------ transform (own halves)
    constexpr int KH = BK / 2;
    const int tt = threadIdx.x - kTransformWarp0 * 32;
    const int col = tt & 127;
    const int kh0 = (tt >> 7) * KH;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(col & ~31) << 16);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    PairWorkList list(p);
    while (ok && list.next(p, w)) {
      const TileCoord c = tile_coord(w.tile, p.tiles_m, p.tiles_n, kRasterGroup, true);
      for (int kt = w.k0; kt < w.k1; ++kt) {
        uint8_t* const st = base_ptr + s * Cfg::STAGE_BYTES;
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
          uint4* const hi = reinterpret_cast<uint4*>(st);
          uint4* const lo = reinterpret_cast<uint4*>(st + Cfg::A_BYTES);
          // One product leaves the tile as it is: the tensor core reads it
          // truncated to TF32 (B is rounded to nearest below), which keeps
          // the per-product error under 2^-10 + 2^-11 and saves a read and
          // a write of the tile in shared memory.
          if (NPROD == 3) {
#pragma unroll 4
            for (int i = tt; i < Cfg::A_BYTES / 16; i += kTransformWarps * 32) {
              const uint4 x = hi[i];
              lo[i] = make_uint4(tf32_lo_of_truncated(x.x), tf32_lo_of_truncated(x.y),
                                 tf32_lo_of_truncated(x.z), tf32_lo_of_truncated(x.w));
            }
          }
          const uint32_t* braw =
              reinterpret_cast<const uint32_t*>(st + Cfg::A_BYTES + Cfg::A_LO_BYTES);
#pragma unroll
          for (int k = 0; k < KH; ++k) split_operand<NPROD>(braw[(kh0 + k) * kHalf + col], bh[k], bl[k]);
        } else {
          const int m0 = c.tm * kPairTile + static_cast<int>(rank) * kHalf;
          const int n0 = c.tn * kPairTile + static_cast<int>(rank) * kHalf;
          const int k0 = k_tile_at(w, kt) * BK;
          // This thread's loads for the stage are all issued before any of
          // them is used, so one latency covers the stage.
          constexpr int AV = kHalf * BK / (kTransformWarps * 32);   // 8
          constexpr int CH = AV;
          uint32_t bv[KH];
          const int gn = n0 + col;
#pragma unroll
          for (int c0 = 0; c0 < AV; c0 += CH) {
            uint32_t av[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              // element e = tt + 256 j: row r, column k of the half tile, lanes
              // along k (along m when A is stored transposed)
              const int e = tt + (c0 + j) * kTransformWarps * 32;
              const int r = trans_a ? e % kHalf : e / BK, k = trans_a ? e / kHalf : e % BK;
              const int gm = m0 + r, gk = k0 + k;
              const size_t at = trans_a ? static_cast<size_t>(gk) * lda + gm
                                          : static_cast<size_t>(gm) * lda + gk;
              av[j] = (gm < p.M && gk < p.K &&
                       GEMM_IN_EXTENT(at, a_extent, p.err, kSiteBoundsA))
                          ? __float_as_uint(__ldg(p.A + at))
                          : 0u;
            }
            if (c0 == 0) {
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
              const int e = tt + (c0 + j) * kTransformWarps * 32;
              const int r = trans_a ? e % kHalf : e / BK, k = trans_a ? e / kHalf : e % BK;
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
        tmem_store_cols<KH>(bt, bh);
        if (NPROD == 3) tmem_store_cols<KH>(bt + BK, bl);
        tmem_wait_st();
        fence_proxy_async_smem();   // A hi/lo: generic-proxy writes -> tensor-core reads
        tc_fence_before_sync();
        mbar_arrive(done_bar(s));   // local; a forwarding warp tells the even CTA
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
  cluster_sync();   // the even CTA's MMAs have finished with this CTA's memory
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  // Split tiles whose last partial (of this CTA's half) this CTA published:
  // every thread sums the partials in segment order and writes C.
  const int npend = *pending_count;
  if (npend > 0) {
    __threadfence();
    for (int e = 0; e < npend; ++e) {
      const WorkItem pw = pending[e];
      const TileCoord c = tile_coord(pw.tile, p.tiles_m, p.tiles_n, kRasterGroup, true);
      const float4* const parts = reinterpret_cast<const float4*>(p.partials) +
                                  static_cast<size_t>(pw.tail) * p.max_seg * 2 * (kPairTile * kHalf / 4);
      constexpr int kVec = kPairTile * kHalf / 4;   // float4s of one half partial
      constexpr int kBatch = 8;                     // float4s per thread in flight
#pragma unroll 1
      for (int base = 0; base < kVec; base += kBatch * kThreads) {
        float4 sum[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int sg = 0; sg < pw.nseg; ++sg) {
          const float4* src = parts + (static_cast<size_t>(sg) * 2 + rank) * kVec;
          float4 x[kBatch];
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            const int f = base + threadIdx.x + i * kThreads;
            x[i] = f < kVec && GEMM_IN_EXTENT(
                                   4 * (src + f - reinterpret_cast<const float4*>(p.partials)) + 3,
                                   work_extent, p.err, kSiteBoundsWork)
                       ? __ldcg(src + f)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            sum[i].x += x[i].x;
            sum[i].y += x[i].y;
            sum[i].z += x[i].z;
            sum[i].w += x[i].w;
          }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int f = base + threadIdx.x + i * kThreads;   // float4 index in the half tile
          if (f >= kVec) continue;
          const int m = c.tm * kPairTile + f / (kHalf / 4);
          const int n = c.tn * kPairTile + static_cast<int>(rank) * kHalf + (f % (kHalf / 4)) * 4;
          if (m < p.M) {
            float* dst = p.C + static_cast<size_t>(m) * static_cast<size_t>(ldc) + n;
            const float vals[4] = {sum[i].x, sum[i].y, sum[i].z, sum[i].w};
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              if (n + qq < p.N)
                if (GEMM_IN_EXTENT(dst + qq - p.C, c_extent, p.err, kSiteBoundsC))
                  dst[qq] = scale ? pair_scaled_c(vals[qq], dst + qq, gp.alpha, gp.beta) : vals[qq];
          }
        }
      }
    }
  }
  clock_stop(p.err, clk_mark);
  if (p.sk_ctas > 0 && threadIdx.x == 0) tail_launch_done(p.counters);
}

// ---------------------------------------------------------------- host side
constexpr int kMaxDevices = 64;

template <int BK, int NPROD, int LOAD>
int launch_pair_one(const GemmArgs& g, const PairParams& p, const PairGeneral& gp,
                    const CUtensorMap& ma, const CUtensorMap& mb, int grid, cudaStream_t stream) {
  using Cfg = PairCfg<BK, NPROD>;
  static std::atomic<unsigned long long> configured{0};
  auto kern = tc_pair_kernel<BK, NPROD, LOAD>;
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

}  // namespace

// Least K for the pair kernel on the TMA path, with three products and with
// one.  Its single accumulator makes each tile's MMAs wait for the previous
// tile's epilogue (about 7,000 clocks), against a tile's MMA work of 48 K
// clocks (three products) or 16 K (one).  Measured on GB300 (CUDA-graph
// replay, against single-SM tiles): three products, 4096^3 391.6 against
// 399.5 us and 8192^3 3191 against 3346 us, but 4096 x 1024 x 4096 123.3
// against 115.1 us and a tie at K = 2048 - 3072; one product, 8192^3 1499
// against 1535 us, but 4096^3 206.3 against 198.7 us and 4096 x 1024 x 4096
// 64.9 against 51.2 us.
constexpr int kPairMinK3 = 3072;
constexpr int kPairMinK1 = 6144;

bool tc_pair_suits(const GemmArgs& g, int nprod) {
  if (g.flags & GEMM_F32_FLAG_SINGLE_CTA) return false;
  if (g.flags & GEMM_F32_FLAG_CTA_PAIR) return true;
  if (g.flags & (GEMM_F32_FLAG_TILE64 | GEMM_F32_FLAG_TILE128 | GEMM_F32_FLAG_TILE224 |
                 GEMM_F32_FLAG_TILE256 | GEMM_F32_FLAG_ONE_TILE_PER_CTA))
    return false;
  const long tiles = static_cast<long>((g.M + kPairTile - 1) / kPairTile) *
                     ((g.N + kPairTile - 1) / kPairTile);
  if (g.M < kPairTile || g.N < kPairTile || tiles < g.num_sms / 2) return false;
  if (!(g.flags & GEMM_F32_FLAG_FORCE_STAGED) && tma_addressable(g))
    return g.K >= (nprod == 1 ? kPairMinK1 : kPairMinK3);
  return true;   // per-thread loads: the pair kernel halves each SM's share
}

int launch_tc_pair(GemmArgs& g, int nprod, cudaStream_t stream, int* launches) {
  *launches = 0;
  const int pairs = g.num_sms / 2;
  if (pairs < 1) return GEMM_F32_EDEVICE;
  // Operand path first: it sets the K depth of a stage (one product on the
  // TMA path: 32; otherwise 16, which keeps the staged loads of one product
  // within the 96 registers this 18-warp block gets).
  bool tma = !(g.flags & GEMM_F32_FLAG_FORCE_STAGED) && tma_addressable(g);
  int bk = (nprod == 1 && tma) ? 32 : 16;
  alignas(64) CUtensorMap ma, mb;
  if (tma) {
    tma = tma_encode_2d(&ma, g.A, g.M, g.K, g.lda, bk, kHalf,
                    bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) &&
          tma_encode_2d(&mb, g.B, g.K, g.N, g.ldb, kHalf, bk, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!tma) {
    bk = 16;
    memset(&ma, 0, sizeof(ma));
    memset(&mb, 0, sizeof(mb));
  }
  PairParams p;
  p.A = g.A;
  p.B = g.B;
  p.C = g.C;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles_m = (g.M + kPairTile - 1) / kPairTile;
  p.tiles_n = (g.N + kPairTile - 1) / kPairTile;
  p.k_iters = (g.K + bk - 1) / bk;
  p.drop_first_copy = (g.flags & GEMM_F32_FLAG_TEST_DROP_COPY) ? 1 : 0;
  p.err = g.err;
  PairGeneral gp;
  gp.lda = g.lda;
  gp.ldb = g.ldb;
  gp.ldc = g.ldc;
  gp.trans_a = g.trans_a;
  gp.trans_b = g.trans_b;
  gp.alpha = g.alpha;
  gp.beta = g.beta;
  gp.scale = g.scale;
  p.partials = nullptr;
  p.counters = nullptr;
  const long tiles = static_cast<long>(p.tiles_m) * p.tiles_n;
  if (tiles > 0x7fffffffL) return GEMM_F32_EINVAL;
  p.dp_tiles = static_cast<int>(tiles);
  p.sk_ctas = 0;
  p.sk_work = 0;
  p.max_seg = 1;
  int units = static_cast<int>(std::min<long>(tiles, pairs));
  if (!(g.flags & GEMM_F32_FLAG_NO_SPLIT_K)) {
    PairParams q = p;
    const size_t ws_bytes =
        plan_split_tail(q, tiles, pairs, sizeof(float) * 2 * kPairTile * kHalf, kMinSplitIters, 2);
    void* ws = ws_bytes ? acquire_workspace(g.device, stream, ws_bytes) : nullptr;
    if (ws) {
      p = q;
      units = pairs;
      p.counters = static_cast<unsigned long long*>(ws);
      p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
    }
  }
  const int grid = 2 * units;
  int rc;
  if (nprod == 3)
    rc = tma ? launch_pair_one<16, 3, kLoadTma>(g, p, gp, ma, mb, grid, stream)
         : plain_form(g) ? launch_pair_one<16, 3, kLoadStaged>(g, p, gp, ma, mb, grid, stream)
                         : launch_pair_one<16, 3, kLoadStagedGeneral>(g, p, gp, ma, mb, grid, stream);
  else
    rc = tma ? launch_pair_one<32, 1, kLoadTma>(g, p, gp, ma, mb, grid, stream)
         : plain_form(g) ? launch_pair_one<16, 1, kLoadStaged>(g, p, gp, ma, mb, grid, stream)
                         : launch_pair_one<16, 1, kLoadStagedGeneral>(g, p, gp, ma, mb, grid, stream);
  if (rc == GEMM_F32_OK) {
    *launches += 1;
    g.kernel = "tc_pair_kernel";
  }
  return rc;
}

}  // namespace gemm_f32_impl
