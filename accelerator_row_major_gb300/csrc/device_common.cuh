// Device-side building blocks shared by the GEMM kernels (sm_103a only):
// the persistent tile order, bounded mbarrier waits that report instead of
// hanging, and thin inline-PTX wrappers for mbarrier, TMA and tcgen05.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>

namespace gemm_f32_dev {

// ---------------------------------------------------------------- errors
// A wait that runs past this budget records its site in the error word and
// returns false; the kernel then unwinds without touching C any further.
constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s

// Sites reported through gemm_f32_status().
enum WaitSite : unsigned {
  kSiteProducerEmpty = 1,   // TMA producer waiting for a free stage
  kSiteTransformFull = 2,   // transform warps waiting for TMA data
  kSiteTransformEmpty = 3,  // staged loaders waiting for a free stage
  kSiteMmaReady = 4,        // MMA issuer waiting for split operands
  kSiteMmaAccEmpty = 5,     // MMA issuer waiting for a drained accumulator
  kSiteEpilogueFull = 6,    // epilogue waiting for a finished accumulator
  kSiteDrainMma = 7,        // teardown: waiting for the last MMAs
  kSiteDrainTma = 8,        // teardown: waiting for copies in flight
  kSitePendingOverflow = 9, // split-tail bookkeeping exceeded its bound
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(unsigned* err, unsigned site) {
  atomicCAS(err, 0u, site);
}

// ---------------------------------------------------------------- clock record
// The error word is the first of a 32-byte block of device words; bytes
// 16..31 hold two 64-bit sums, the clock record.  The first thread of CTA 0
// of the pair and FFMA kernels adds its CTA's lifetime to them, in SM clocks
// (clock64) and in nanoseconds (%globaltimer).  CTA 0 of a persistent grid
// lives through the whole launch, so cycles / ns over a run of launches is
// the SM clock they ran at, whatever the driver's sampled clock says.  The
// start mark is kept in shared memory, so the record holds no register
// through the kernel.
struct ClockRecord {
  unsigned long long cycles, ns;
};

__device__ __forceinline__ ClockRecord* clock_record(unsigned* err) {
  return reinterpret_cast<ClockRecord*>(err + 4);
}

__device__ __forceinline__ void clock_start(unsigned long long (&mark)[2]) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    mark[0] = clock64();
    mark[1] = globaltimer_ns();
  }
}

__device__ __forceinline__ void clock_stop(unsigned* err, const unsigned long long (&mark)[2]) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const unsigned long long c = clock64() - mark[0];
    const unsigned long long t = globaltimer_ns() - mark[1];
    ClockRecord* const r = clock_record(err);
    atomicAdd(&r->cycles, c);
    atomicAdd(&r->ns, t);
  }
}

// ---------------------------------------------------------------- bounds checks
// The debug build (-DGEMM_BOUNDS_CHECK, libgemm_f32_checked.so) checks every
// global load and store that a kernel indexes by hand -- the per-thread
// operand loads, the FFMA copies, the C stores, the partial tiles of the
// split tail, the operand packing and the teaching kernels -- against the
// extent of the array it addresses.  An index outside records its site in
// the error word (the first one wins, as for the waits), and the access is
// skipped: a load gives 0, a store does not happen.  Out-of-range elements
// load 0 and are never written, the rule of "Lesson 10: shared-memory tiled
// GEMM" (hpc.payai.win, section 3); here it is checked, not assumed.  In the
// default build the check is the constant true and costs nothing.
enum BoundsSite : unsigned {
  kSiteBoundsA = 16,        // a read of A outside its stored extent
  kSiteBoundsB = 17,        // a read of B outside its stored extent
  kSiteBoundsC = 18,        // a read or write of C outside its window's extent
  kSiteBoundsWork = 19,     // a partial tile outside the split-tail workspace
  kSiteBoundsPack = 20,     // operand packing outside its source or destination
};

#ifdef GEMM_BOUNDS_CHECK
__device__ __forceinline__ bool in_extent(size_t index, size_t extent, unsigned* err,
                                          unsigned site) {
  if (index < extent) return true;
  record_error(err, site);
  return false;
}
#define GEMM_IN_EXTENT(index, extent, err, site) \
  ::gemm_f32_dev::in_extent(static_cast<size_t>(index), static_cast<size_t>(extent), (err), (site))
#else
#define GEMM_IN_EXTENT(index, extent, err, site) true
#endif

// Elements spanned by a row-major array of `rows` rows of `cols` elements
// with row stride `ld` (first to last element touched).
__host__ __device__ __forceinline__ size_t stored_extent(long long rows, long long cols,
                                                         long long ld) {
  return rows > 0 && cols > 0 ? static_cast<size_t>((rows - 1) * ld + cols) : 0;
}

// ---------------------------------------------------------------- tile order
// Output tiles are visited in groups of `group` tile-rows: inside a group the
// index runs down the rows first, so CTAs that run at the same time share
// the same few B column panels and A row panels in L2.
struct TileCoord {
  int tm, tn;
};

// With `snake`, odd groups run their columns right to left, so that the
// last tiles of one group and the first of the next share B column panels.
__device__ __forceinline__ TileCoord tile_coord(int t, int tiles_m, int tiles_n, int group,
                                                bool snake = false) {
  const int per_group = group * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group;
  const int rows_here = min(tiles_m - first_m, group);
  const int r = t - g * per_group;
  TileCoord c;
  c.tm = first_m + r % rows_here;
  c.tn = r / rows_here;
  if (snake && (g & 1)) c.tn = tiles_n - 1 - c.tn;
  return c;
}

// ---------------------------------------------------------------- split tail
// When the output tiles do not fill the last wave of CTAs, the remaining
// ("tail") tiles' K iterations are shared evenly by the CTAs.  Work list of
// CTA c (grid G): whole tiles c, c+G, ... below dp_tiles, then iterations
// [start(c), start(c+1)) of the tail's flattened (tile, K iteration) space.
// A CTA that computes only part of a tile writes it to a workspace slot and
// bumps the tile's counter; the CTA that bumps it last adds the partials in
// segment order (fixed: the sum does not depend on which CTA is last).
constexpr int kMinSplitIters = 64;       // least K iterations per CTA in the split tail

// Operand loaders of the tensor-core kernels (a template parameter):
// per-thread loads of the plain product, TMA tiles, or per-thread loads of
// the general form (row strides, stored transposes).  The plain product's
// staged kernel keeps its own code: the general form's indexing costs it
// registers (measured on GB300: 88 -> 122 at TM = 64, 8 % slower).
constexpr int kLoadStaged = 0;
constexpr int kLoadTma = 1;
constexpr int kLoadStagedGeneral = 2;

// Tile counters at the start of the workspace (kCounterBytes): one 64-bit
// word per tail tile (two for CTA-pair tiles, one per half) holding
// (generation << 32) | partials published, then, in the last 8 bytes, the
// number of CTAs of the running launch that have finished and the
// generation.  A launch with a split tail counts only arrivals made under
// the current generation, and the last of its CTAs to finish moves the
// generation on.  A launch that gave up on a bounded wait still finishes
// every CTA, so the counts it left half done belong to an old generation
// and the next launch on the workspace ignores them: no reset, on the host
// or in a graph replay, is needed after a timeout.  (The generation is 32
// bits: a stale count could only match again 2^32 split launches later.)
constexpr size_t kCounterBytes = 4096;
constexpr int kMaxTailWords = static_cast<int>((kCounterBytes - 64) / 8);   // 504

struct TailControl {
  unsigned done;   // CTAs of the running launch that have finished
  unsigned gen;    // generation of the running launch
};

__host__ __device__ __forceinline__ TailControl* tail_control(void* counters) {
  return reinterpret_cast<TailControl*>(static_cast<char*>(counters) + kCounterBytes - 8);
}

// Publishes one partial of a tail tile: returns how many partials of the
// tile (this one included) have been published in the current launch.
__device__ __forceinline__ unsigned tail_arrive(unsigned long long* words, int index) {
  const unsigned gen = *reinterpret_cast<volatile unsigned*>(&tail_control(words)->gen);
  unsigned long long* const w = words + index;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w);
  for (;;) {
    const unsigned count =
        static_cast<unsigned>(old >> 32) == gen ? static_cast<unsigned>(old) : 0u;
    const unsigned long long want = (static_cast<unsigned long long>(gen) << 32) | (count + 1u);
    const unsigned long long seen = atomicCAS(w, old, want);
    if (seen == old) return count + 1u;
    old = seen;
  }
}

// Called once per CTA (one thread) after the CTA's last use of the tile
// counters, by every CTA of a launch that has a split tail.
__device__ __forceinline__ void tail_launch_done(void* counters) {
  TailControl* const t = tail_control(counters);
  __threadfence();
  if (atomicAdd(&t->done, 1u) == gridDim.x - 1) {
    t->done = 0u;
    __threadfence();
    atomicAdd(&t->gen, 1u);
  }
}

// One unit of a CTA's work: K iterations [k0, k1) of one output tile.
struct WorkItem {
  int tile, k0, k1;
  int tail;        // index among the split tiles, or -1 for a whole tile
  int seg, nseg;   // this CTA's position among the CTAs sharing the tile
  bool rev;        // K iterations visited from k1 - 1 down to k0
};

// K iteration (tile column of A, tile row of B) that the n-th step of a work
// item loads, n = kt - k0 counted from the item's first step.
__device__ __forceinline__ int k_tile_at(const WorkItem& w, int kt) {
  return w.rev ? w.k0 + w.k1 - 1 - kt : kt;
}

__host__ __device__ __forceinline__ long long sk_start(long long c, long long ctas, long long work) {
  return c * work / ctas;
}
// CTA whose share of the split K iterations contains iteration x
__host__ __device__ __forceinline__ int sk_owner(long long x, long long ctas, long long work) {
  return static_cast<int>(((x + 1) * ctas - 1) / work);
}

// The work list of one CTA, walked identically by every role.  P provides
// k_iters, dp_tiles, sk_ctas and sk_work.
struct WorkList {
  int next_dp;
  long long x, x_end;

  template <class P>
  __device__ __forceinline__ explicit WorkList(const P& p) {
    next_dp = blockIdx.x;
    x = x_end = 0;
    if (static_cast<int>(blockIdx.x) < p.sk_ctas) {
      x = sk_start(blockIdx.x, p.sk_ctas, p.sk_work);
      x_end = sk_start(blockIdx.x + 1, p.sk_ctas, p.sk_work);
    }
  }

  template <class P>
  __device__ __forceinline__ bool next(const P& p, WorkItem& w) {
    if (next_dp < p.dp_tiles) {
      w.tile = next_dp;
      w.k0 = 0;
      w.k1 = p.k_iters;
      w.tail = -1;
      w.seg = 0;
      w.nseg = 1;
      w.rev = false;
      next_dp += gridDim.x;
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
      w.seg = static_cast<int>(blockIdx.x) - first;
      w.nseg = last - first + 1;
      w.rev = false;
      x += w.k1 - w.k0;
      return true;
    }
    return false;
  }
};

// Host: splits the last partial wave along K.  Fills p.dp_tiles / sk_ctas /
// sk_work / max_seg (p.k_iters must be set) and returns the workspace bytes
// the split needs, 0 when whole tiles are better (no split).
template <class P>
inline size_t plan_split_tail(P& p, long tiles, int grid, size_t partial_tile_bytes,
                              int min_iters = kMinSplitIters, int words_per_tile = 1) {
  p.dp_tiles = static_cast<int>(tiles);
  p.sk_ctas = 0;
  p.sk_work = 0;
  p.max_seg = 1;
  const long tail = tiles % grid;
  if (tail == 0) return 0;
  const long long work = static_cast<long long>(tail) * p.k_iters;
  const long long ctas = std::min<long long>(grid, work / min_iters);
  if (ctas <= tail) return 0;   // each CTA would still get whole tiles
  int max_seg = 1;
  for (long i = 0; i < tail; ++i) {
    const int first = sk_owner(i * p.k_iters, ctas, work);
    const int last = sk_owner((i + 1) * static_cast<long long>(p.k_iters) - 1, ctas, work);
    max_seg = std::max(max_seg, last - first + 1);
  }
  if (max_seg == 1 || tail * words_per_tile > kMaxTailWords) return 0;
  p.dp_tiles = static_cast<int>(tiles - tail);
  p.sk_ctas = static_cast<int>(ctas);
  p.sk_work = work;
  p.max_seg = max_seg;
  return kCounterBytes + static_cast<size_t>(tail) * max_seg * partial_tile_bytes;
}

// Device: every thread of the CTA (NTHREADS) adds the nseg partial tiles at
// `parts` ([seg][ROWS][COLS] fp32) in segment order and writes the sum to C
// rows m0.., columns n0.. (masked).  CHUNK independent 16-byte loads per
// thread per partial keep the L2 reads in flight; a kernel whose hot loops
// need few registers takes a small CHUNK so that this end-of-work code does
// not set its register count.
// What the checked build checks the reduction's accesses against: the error
// word, the elements of partials from `parts` on, and C's extent.
struct BoundsRef {
  unsigned* err;
  size_t parts_extent;
  size_t c_extent;
};

// sum[i] += chunk `base` + i of each of the nseg partial tiles at p4, in
// segment order.  The loads of two segments are issued together, so that a
// chunk of the usual two-segment tile costs one round trip to L2, not two.
template <int kChunk, int kVec, int NTHREADS>
__device__ __forceinline__ void add_segments(const float4* p4, int nseg, int base,
                                             float4 (&sum)[kChunk],
                                             [[maybe_unused]] const BoundsRef& br) {
  auto load = [&](int sg, int i) {
    const size_t f4 = static_cast<size_t>(sg) * kVec + threadIdx.x + (base + i) * NTHREADS;
    return GEMM_IN_EXTENT(4 * f4 + 3, br.parts_extent, br.err, kSiteBoundsWork)
               ? __ldcg(p4 + f4)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto add = [&](float4& a, const float4& x) {
    a.x += x.x;
    a.y += x.y;
    a.z += x.z;
    a.w += x.w;
  };
  int sg = 0;
#pragma unroll 1
  for (; sg + 1 < nseg; sg += 2) {
    float4 x0[kChunk], x1[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      x0[i] = load(sg, i);
      x1[i] = load(sg + 1, i);
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      add(sum[i], x0[i]);
      add(sum[i], x1[i]);
    }
  }
  if (sg < nseg) {
    float4 x0[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) x0[i] = load(sg, i);
#pragma unroll
    for (int i = 0; i < kChunk; ++i) add(sum[i], x0[i]);
  }
}

template <int ROWS, int COLS, int NTHREADS, int CHUNK>
__device__ __forceinline__ void reduce_partials(const float* parts, int nseg, int m0, int n0,
                                                int M, int N, float* C,
                                                [[maybe_unused]] const BoundsRef& br) {
  constexpr int kVec = ROWS * COLS / 4;            // float4s per partial
  constexpr int kPer = kVec / NTHREADS;            // per thread
  constexpr int kChunk = kPer < CHUNK ? kPer : CHUNK;
  static_assert(kVec % NTHREADS == 0 && kPer % kChunk == 0, "partial tile shape");
  const float4* const p4 = reinterpret_cast<const float4*>(parts);
#pragma unroll 1
  for (int base = 0; base < kPer; base += kChunk) {
    float4 sum[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    add_segments<kChunk, kVec, NTHREADS>(p4, nseg, base, sum, br);
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int f = threadIdx.x + (base + i) * NTHREADS;   // float4 index in the tile
      const int m = m0 + f / (COLS / 4);
      const int n = n0 + (f % (COLS / 4)) * 4;
      if (m < M) {
        float* dst = C + static_cast<size_t>(m) * static_cast<size_t>(N) + n;
        const float v[4] = {sum[i].x, sum[i].y, sum[i].z, sum[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (n + q < N && GEMM_IN_EXTENT(dst + q - C, br.c_extent, br.err, kSiteBoundsC))
            dst[q] = v[q];
      }
    }
  }
}

// The same for the general form: row stride ldc and, with `scale`,
// C = alpha * sum + beta * C_old (C_old read only when beta != 0).
template <int ROWS, int COLS, int NTHREADS, int CHUNK>
__device__ __forceinline__ void reduce_partials_general(const float* parts, int nseg, int m0,
                                                        int n0, int M, int N, float* C, int ldc,
                                                        int scale, float alpha, float beta,
                                                        [[maybe_unused]] const BoundsRef& br) {
  constexpr int kVec = ROWS * COLS / 4;            // float4s per partial
  constexpr int kPer = kVec / NTHREADS;            // per thread
  constexpr int kChunk = kPer < CHUNK ? kPer : CHUNK;
  static_assert(kVec % NTHREADS == 0 && kPer % kChunk == 0, "partial tile shape");
  const float4* const p4 = reinterpret_cast<const float4*>(parts);
#pragma unroll 1
  for (int base = 0; base < kPer; base += kChunk) {
    float4 sum[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    add_segments<kChunk, kVec, NTHREADS>(p4, nseg, base, sum, br);
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int f = threadIdx.x + (base + i) * NTHREADS;   // float4 index in the tile
      const int m = m0 + f / (COLS / 4);
      const int n = n0 + (f % (COLS / 4)) * 4;
      if (m < M) {
        float* dst = C + static_cast<size_t>(m) * static_cast<size_t>(ldc) + n;
        const float v[4] = {sum[i].x, sum[i].y, sum[i].z, sum[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (n + q >= N || !GEMM_IN_EXTENT(dst + q - C, br.c_extent, br.err, kSiteBoundsC))
            continue;
          float r = v[q];
          if (scale) {   // alpha * sum (+ beta * C_old when beta != 0)
            r *= alpha;
            if (beta != 0.0f) r = fmaf(beta, dst[q], r);
          }
          dst[q] = r;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- dependent launches
// Programmatic dependent launch: a kernel launched after one of these on the
// same stream (with the programmatic-serialization launch attribute) may
// start its CTAs as this one's CTAs finish.  Each kernel calls
// grid_launch_dependents() once its own set-up is done, and
// grid_dependency_wait() before its first global memory access: that wait
// returns once every earlier kernel of the stream has completed and its
// memory operations are visible, so a kernel may read what the previous one
// wrote (C becoming the next A, the split tail's counters).  Only set-up that
// touches nothing global (barriers, tensor memory, descriptor prefetch) runs
// before it.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- shared memory
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed.  Gives up after
// kWaitBudgetNs, records `site` and returns false.  The first look is a
// non-blocking test: measured on GB300, on a phase that has already completed
// it costs the MMA-issuing thread about 160 cycles less than try_wait.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err,
                                          unsigned site) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitBudgetNs) {
      record_error(err, site);
      return false;
    }
  }
}

// Generic-proxy writes to shared memory become visible to the async proxy
// (TMA, tensor cores) that is ordered after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(desc) : "memory");
}

// 2-D tiled copy global -> shared; completion is counted on `bar` in bytes.
// x is the innermost coordinate (elements); it must keep x * 4 bytes a
// multiple of 16 (the callers only pass multiples of 32).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* desc, uint32_t bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(desc), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]: A is read from tensor memory (lane =
// row of A, one 32-bit column per K element), B from shared memory.
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrive once every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// Each thread of the warp writes 8 / 16 / 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st_8cols(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor of tcgen05 (64 bits):
//   [0,14)  start address >> 4       [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4  [46,48) descriptor version (1)
//   [49,52) base offset (0: swizzle atoms start on their natural boundary)
//   [61,64) layout: 0 none, 2 = 128-byte swizzle, 4 = 64-byte swizzle
// For a K-major swizzled operand the leading offset is unused and the stride
// offset is the distance between groups of 8 rows.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout) << 61;
  return d;
}

// Instruction descriptor for kind::tf32 with an FP32 accumulator:
//   [4,6) D format (1 = f32)  [7,10) A format (2 = tf32)  [10,13) B format (2)
//   [15] A major (0 = K-major)  [16] B major (0 = K-major)
//   [17,23) N >> 3             [24,29) M >> 4
// Both operands are kept K-major: measured on GB300, a kind::tf32 MMA whose
// shared-memory B operand is described as MN-major completes without writing
// its accumulator.
__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(n) >> 3) << 17) |
         ((static_cast<uint32_t>(m) >> 4) << 24);
}

// ---------------------------------------------------------------- TF32 split
// The tensor core reads a 32-bit operand as TF32 by dropping its 13 low
// mantissa bits (measured on GB300 for both shared-memory and tensor-memory
// operands).  The helpers below therefore leave those bits as they are and
// only arrange that dropping them gives the intended TF32 value.

// Bits that the tensor core reads as the nearest TF32 value of x (10
// explicit mantissa bits), ties away from zero: half of the 13 dropped bits is
// added to the magnitude, and the truncation on read completes the rounding.
// A carry into the exponent is the correct round-up.  Finite inputs below
// 2^128 * (1 - 2^-12) only; larger ones round to infinity.
__device__ __forceinline__ uint32_t tf32_round_bits(uint32_t x) {
  return x + 0x1000u;
}

// Low part for an operand whose high part is the raw fp32 value: the high
// part the tensor core sees is trunc(x), x with the 13 low bits cleared.  The
// rest, x - trunc(x), is exact in fp32, and the returned bits make the tensor
// core read it rounded to the nearest TF32 value.
__device__ __forceinline__ uint32_t tf32_lo_of_truncated(uint32_t x) {
  const float r = __fsub_rn(__uint_as_float(x), __uint_as_float(x & 0xFFFFE000u));
  return tf32_round_bits(__float_as_uint(r));
}

}  // namespace gemm_f32_dev
