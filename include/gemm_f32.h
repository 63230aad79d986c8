/*
 * gemm_f32 -- row-major single-precision GEMM for NVIDIA GB300 (sm_103a).
 *
 * Operation (all entry points that compute):
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j],   0 <= i < M, 0 <= j < N
 * A is M x K, B is K x N and C is M x N, dense and row-major with leading
 * dimensions K, N and N.  This is the element formula in the problem
 * statement of "LeetGPU problem 2: matrix multiplication" (yekq.top, section
 * "problem statement") and the product of "Lesson 10: shared-memory tiled
 * GEMM" (hpc.payai.win, section 1).  C is overwritten (alpha = 1, beta = 0);
 * it need not be initialised.  The euler0525 page computes the same product
 * with the contraction named N; here K is always the contraction.
 *
 * Pointers: caller-owned DEVICE pointers (4-byte aligned), valid on the
 * current device.  The library keeps no reference to them after the call
 * returns.
 *
 * Workspace: when the output tiles do not fill the last wave of SMs, the
 * tensor modes split the remaining tiles along K across all SMs; partial
 * tiles then go through a workspace the library owns, one per (device,
 * stream).  The first call that needs it (or a larger one) allocates it with
 * cudaMalloc, which synchronises the device, so make such a call once before
 * capturing a stream into a CUDA graph; gemm_f32_release() frees it.  Calls
 * on different streams use different workspaces.
 *
 * Streams: every call is asynchronous on `stream` (0 = legacy default
 * stream) and never synchronises the host, like the stream-taking launcher
 * of "Lesson 10" (section "practice task").  A device-side failure (a
 * bounded wait that ran out) is reported later by gemm_f32_status().
 *
 * Sizes: any M, N, K >= 0 (M * N, M * K and K * N below 2^62).  M == 0 or
 * N == 0 is a no-op; K == 0 writes zeros into C.  Ragged sizes are masked
 * inside the kernels: no size needs to be a multiple of any tile.
 *
 * Return codes: 0 on success, else one of the negative GEMM_F32_E* codes.
 * No entry point aborts, prints or throws.
 */
#ifndef GEMM_F32_H
#define GEMM_F32_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t in the CUDA runtime headers. */
typedef struct CUstream_st* gemm_f32_stream_t;

enum gemm_f32_status_code {
    GEMM_F32_OK = 0,
    GEMM_F32_EINVAL = -1,   /* negative size, null pointer with work to do,
                               C overlapping A or B, unknown mode or flag   */
    GEMM_F32_EDEVICE = -2,  /* current device is not sm_103 (GB300), or a
                               CUDA query failed                           */
    GEMM_F32_ELAUNCH = -3,  /* the kernel launch (or the K == 0 memset) was
                               refused by the CUDA runtime                  */
    GEMM_F32_ETIMEOUT = -4, /* gemm_f32_status(): a bounded device-side wait
                               ran out; C of that call is undefined.  Later
                               calls are not affected: the split-tail
                               bookkeeping the call left half done is
                               ignored by the next call on its own          */
    GEMM_F32_ESCRATCH = -5  /* gemm_f32_noalloc(): the product would need
                               more scratch than the library's fixed array
                               (GEMM_F32_NOALLOC_SCRATCH_BYTES); nothing was
                               launched                                     */
};

/* Arithmetic modes of gemm_f32_ex. */
enum gemm_f32_mode {
    GEMM_F32_MODE_TC3X = 0, /* default.  Tensor cores (tcgen05.mma
                               kind::tf32): each operand is split into a
                               TF32 high part and a TF32 low part and three
                               products hi*hi + hi*lo + lo*hi are accumulated
                               in fp32 (four, lo*lo too, in tiles of 64
                               rows).  |C - exact| <= 1e-5 * (|A||B|)_ij.   */
    GEMM_F32_MODE_FFMA = 1, /* CUDA-core fp32 fused multiply-add, register
                               tiled.  Same 1e-5 bound.                     */
    GEMM_F32_MODE_TC1X = 2  /* opt-in: one TF32 product; B rounded to TF32
                               (nearest, ties away), A rounded the same way
                               or, where the tensor-memory accelerator reads
                               it, truncated by the tensor core (per-product
                               error below 1.5e-3).  Bound 2e-3.            */
};

/* Flags of gemm_f32_ex (bitwise OR).  None changes the result beyond the
 * mode's bound; they exist to select kernel variants for tests and tuning. */
#define GEMM_F32_FLAG_FORCE_STAGED 0x1u  /* tensor modes: load operands with
                                            per-thread masked loads even where
                                            the tensor-memory-accelerator path
                                            is possible                       */
#define GEMM_F32_FLAG_TILE64 0x10u       /* tensor modes: output tiles of 64,  */
#define GEMM_F32_FLAG_TILE128 0x20u      /*   128, 224 or 256 rows of C (by 128 */
#define GEMM_F32_FLAG_TILE224 0x80u      /*   columns; 224 with TMA-readable    */
#define GEMM_F32_FLAG_TILE256 0x40u      /*   operands only, else 256);         */
                                         /*   default: chosen by size           */
#define GEMM_F32_FLAG_ONE_TILE_PER_CTA 0x100u /* launch one CTA per output
                                            tile instead of the persistent grid */
#define GEMM_F32_FLAG_NO_SPLIT_K 0x200u  /* never split the last wave along K
                                            (no workspace)                    */
#define GEMM_F32_FLAG_CTA_PAIR 0x400u    /* tensor modes: compute 256 x 256
                                            tiles on pairs of SMs (cluster of
                                            two CTAs, one M = 256 MMA); the
                                            default with a wave of such tiles
                                            and a deep K (on TMA-readable
                                            operands K >= 3072 in tc3x, K >=
                                            6144 in tc1x)                     */
#define GEMM_F32_FLAG_SINGLE_CTA 0x800u  /* tensor modes: one CTA per tile    */
#define GEMM_F32_FLAG_TEST_DROP_COPY 0x1000u /* testing only, on the TMA
                                            path of every mode: CTA 0 never
                                            issues its first operand copy, so
                                            its bounded waits run out (about
                                            2 s) and gemm_f32_status() returns
                                            GEMM_F32_ETIMEOUT.  C is undefined
                                            after such a call.  Ignored where
                                            operands are copied per thread
                                            (no waits there).                 */

/* Small products: without flags, a product of at most 2^23 multiply-adds
 * with K <= 256 runs in every mode on a CUDA-core kernel (fp32 fused
 * multiply-adds, within every mode's bound): at these sizes launch and
 * pipeline set-up, not arithmetic, set the time.  Any flag keeps the mode's
 * own kernels. */

/* C = A * B in the default mode (GEMM_F32_MODE_TC3X).  The environment
 * variable GEMM_F32_MODE ("tc3x", "ffma" or "tc1x"), read once per process,
 * changes the default.  Returns 0 or a negative GEMM_F32_E* code. */
int gemm_f32(const float* A, const float* B, float* C, int M, int N, int K,
             gemm_f32_stream_t stream);

/* C = A * B in an explicit mode with variant flags.  Returns 0 or a negative
 * code; GEMM_F32_EINVAL for an unknown mode or flag.
 * gemm_f32, gemm_f32_ex and gemm_f32_general may be captured into a CUDA
 * graph on `stream` once a call of the same shape, mode and flags has run
 * on the device outside the capture (that first call may allocate the
 * split-tail workspace, which a capture must not); a replay computes with
 * the captured pointers and whatever values they then hold. */
int gemm_f32_ex(const float* A, const float* B, float* C, int M, int N, int K,
                int mode, unsigned flags, gemm_f32_stream_t stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns 0, GEMM_F32_ETIMEOUT if a kernel since the last call gave up
 * on a bounded wait, or GEMM_F32_ELAUNCH if the synchronisation itself
 * reported a CUDA error.  `site` (may be NULL) receives the code of the first
 * wait that gave up (0 if none). */
int gemm_f32_status(gemm_f32_stream_t stream, unsigned* site);

/* The clock record of the current device.  The first thread of CTA 0 of
 * every tc_pair_kernel and ffma_gemm_kernel launch adds that CTA's lifetime
 * to two running sums: SM clock cycles (clock64) and nanoseconds
 * (%globaltimer).  tc_gemm_kernel and the small and teaching kernels add
 * nothing.  The persistent grids keep CTA 0 for the
 * whole launch, so the difference of two readings taken around a run of
 * launches, cycles / ns, is the SM clock those launches ran at.  That is
 * the clock a compute roofline needs ("Lesson 10: shared-memory tiled
 * GEMM", hpc.payai.win, section 1: the peak is a rate per clock times the
 * clock).  It can sit well below the clock the driver reports under a
 * tensor-core load.  The call synchronises `stream` and copies the two sums
 * to *sm_cycles and *ns, which must not be NULL.  The sums count from the
 * library's set-up on the device.  Launches running on several streams at
 * once add to the same sums.  Returns 0, GEMM_F32_EINVAL (a NULL output),
 * GEMM_F32_EDEVICE or GEMM_F32_ELAUNCH (the synchronisation or the copy
 * failed). */
int gemm_f32_clock_record(gemm_f32_stream_t stream, unsigned long long* sm_cycles,
                          unsigned long long* ns);

/* Number of kernels the last successful call on this host thread launched
 * (0 for a no-op, 1 for a GEMM or for the K == 0 memset, plus one per launch
 * that copied operands for the tensor-memory accelerator). */
int gemm_f32_last_launches(void);

/* Name of the kernel the last successful call on this host thread launched:
 * "tc_pair_kernel" (tensor cores, 256 x 256 tiles on SM pairs),
 * "tc_gemm_kernel" (tensor cores, one SM per tile), "ffma_gemm_kernel",
 * "small_gemm_kernel" (small products), "memset" (K == 0),
 * "scale_window_kernel" (gemm_f32_general with
 * alpha == 0 or K == 0), "ladder_v0" .. "ladder_v4" (gemm_f32_ladder) or
 * "none" (nothing launched).  Static string. */
const char* gemm_f32_last_kernel(void);

/* C = A * B with A, B and C in HOST memory: copies A and B to the device,
 * computes in `mode` (as gemm_f32_ex, no flags) and copies C back, all
 * queued asynchronously.  For throughput, consecutive calls overlap: the
 * library keeps per device two device-side slots (A, B and C buffers, grown
 * on demand and freed by gemm_f32_release) used by alternate calls, and
 * three internal streams (copy in, product, copy out), so one call's copies
 * run while its neighbour's product does.  Events order every reuse of a
 * slot.  Contract:
 *   - A and B are read asynchronously, without waiting for work already
 *     queued on `stream`: the host must have finished writing them, and must
 *     not change them until `stream` has passed this call.
 *   - `stream` waits for the copy of C: C holds the product once the work
 *     queued on `stream` up to this call has completed (for example after
 *     cudaStreamSynchronize or gemm_f32_status on `stream`).
 *   - Pinned host memory (cudaMallocHost, cudaHostAlloc) gives asynchronous
 *     copies at full link speed; pageable memory works but the runtime then
 *     copies it through staging buffers, partly synchronously.
 *   - C must not overlap A or B.  Calls from several host threads are
 *     serialised per device.
 * Returns 0, GEMM_F32_EINVAL (as gemm_f32_ex), GEMM_F32_EDEVICE or
 * GEMM_F32_ELAUNCH (a copy, an event or an allocation failed).  The pages
 * have no counterpart (their benchmark times device buffers); it is the
 * host-to-host path a caller without device memory uses. */
int gemm_f32_host(const float* A, const float* B, float* C, int M, int N, int K, int mode,
                  gemm_f32_stream_t stream);

/* Frees the current device's workspaces (split-tail partials, the copies of
 * operands the tensor-memory accelerator cannot read — odd strides,
 * unaligned bases or stored transposes in products of at least 2^27
 * multiply-adds are copied once into aligned buffers first — and
 * gemm_f32_host's device slots) after synchronising the device.
 * Returns 0, or GEMM_F32_EDEVICE / GEMM_F32_ELAUNCH on a CUDA error. */
int gemm_f32_release(void);

/* Size of the scratch array compiled into the library for gemm_f32_noalloc
 * (32 MiB, held on every device that loads the library until exit). */
#define GEMM_F32_NOALLOC_SCRATCH_BYTES (32u << 20)

/* C = A * B in a tensor mode (GEMM_F32_MODE_TC3X or GEMM_F32_MODE_TC1X)
 * without allocating any device memory.  The pages have no counterpart: it
 * exists for callers that must not allocate -- code that runs where
 * cudaMalloc is not allowed or not safe, such as a host that has handed all
 * device memory to its own pool, a latency-critical path that cannot take
 * cudaMalloc's implicit device synchronisation, or an embedding that must
 * keep the library's memory footprint fixed after start-up.  gemm_f32_ex may
 * allocate its split-tail workspace or aligned copies of its operands on
 * first use; this call takes the split tail's scratch from a fixed array
 * inside the library instead and never calls cudaMalloc, cudaFree or any
 * allocating routine.
 *   - The caller still passes A, B and C (device pointers, as gemm_f32).
 *   - The array's device address is looked up when the library first sets
 *     up a device (the first call of any entry point there), which loads
 *     the library's module holding the array.  Make one library call on each
 *     device before the caller's pool takes the device memory and before
 *     any stream capture; if that lookup failed, this call retries it.
 *   - Every call on a device shares the one array, which keeps what the
 *     last call left in it: two such calls whose kernels overlap on the GPU
 *     (for example on two streams) race and give wrong results.  The array's
 *     split-tail counters need no clearing between calls: they carry a
 *     generation that each call moves on.
 *   - It always runs the single-CTA tensor kernel (tiles 128 columns wide,
 *     or 64 for N <= 64 with TMA-readable operands), never the CTA-pair
 *     kernel nor operand copies, so on large squares (the pair kernel's
 *     domain) and on operands TMA cannot read (per-thread loads) it is
 *     slower than gemm_f32_ex, and its summation order can differ: the
 *     result meets the same bound as gemm_f32_ex in that mode, but need not
 *     be bitwise equal to it.
 *   - Returns GEMM_F32_ESCRATCH, launching nothing, when the product's
 *     split tail would need more than GEMM_F32_NOALLOC_SCRATCH_BYTES; other
 *     errors as gemm_f32_ex (GEMM_F32_EINVAL for mode FFMA or a bad mode,
 *     GEMM_F32_EDEVICE if the array's address cannot be had). */
int gemm_f32_noalloc(const float* A, const float* B, float* C, int M, int N, int K,
                     int mode, gemm_f32_stream_t stream);

/* General form, row-major storage throughout:
 *     C = alpha * op(A) * op(B) + beta * C
 * the scaled, strided and transposable product of the cuBLAS call on
 * "LeetGPU problem 2: matrix multiplication" (yekq.top, section "cuBLAS
 * reference"), restated for row-major matrices.
 *   op(A) is M x K: trans_a = 0, A is stored M x K with row stride lda
 *     (lda >= max(1, K)); trans_a = 1, A is stored K x M (lda >= max(1, M))
 *     and op(A) is its transpose.
 *   op(B) is K x N: trans_b = 0, B is stored K x N (ldb >= max(1, N));
 *     trans_b = 1, B is stored N x K (ldb >= max(1, K)).
 *   C is the M x N window of a row-major array with row stride ldc
 *     (ldc >= max(1, N)); nothing outside the window is read or written.
 *   beta == 0: C is not read (whatever it holds, NaN included, is
 *     overwritten).  alpha == 0 or K == 0: A and B are not read and
 *     C = beta * C.
 *   mode: GEMM_F32_MODE_TC3X, _FFMA or _TC1X with the bounds of gemm_f32_ex,
 *     taken relative to |alpha| (|op(A)||op(B)|)_ij + |beta| |C_ij|.
 * Untransposed operands with row strides a multiple of 4 and 16-byte
 * aligned bases take the tensor-memory-accelerator path; any other layout
 * the per-thread staged loads (slower, same results).
 * Device pointers, caller-owned; asynchronous on `stream`.  Returns 0,
 * GEMM_F32_EINVAL (trans flag not 0/1, a negative size, a stride below its
 * minimum, alpha or beta not finite, a null or misaligned pointer that
 * would be used, or the C window overlapping a stored A or B window),
 * GEMM_F32_EDEVICE or GEMM_F32_ELAUNCH.  May allocate the split-tail
 * workspace as gemm_f32_ex does. */
int gemm_f32_general(int trans_a, int trans_b, int M, int N, int K, float alpha,
                     const float* A, int lda, const float* B, int ldb, float beta, float* C,
                     int ldc, int mode, gemm_f32_stream_t stream);

/* The pages' optimisation ladder for this GEMM ("LeetGPU problem 2: matrix
 * multiplication", yekq.top, sections v0 .. v4 and "benchmark summary"),
 * rebuilt for sm_103a so that each step can be timed on this GPU.  Teaching
 * kernels, not the product path: C = A * B in fp32 fused multiply-adds
 * (ascending k, bound 1e-5 * (|A||B|)_ij as GEMM_F32_MODE_FFMA) by
 *   step 0  one thread per output, threadIdx.x along the rows of C;
 *   step 1  one thread per output, threadIdx.x along the columns;
 *   step 2  16 x 16 shared-memory tiles, zero-filled at the edges;
 *   step 3  64 x 64 block tiles, 4 outputs of one row per thread;
 *   step 4  64 x 64 block tiles, 4 x 4 outputs per thread.
 * Arguments, layout, ownership and errors as gemm_f32_ex; GEMM_F32_EINVAL
 * also for a step outside 0 .. 4 or a grid beyond the launch limits (more
 * than 65535 blocks along y: N > 1048560 for step 0, M > 1048560 for steps 1
 * and 2, M > 4194240 for steps 3 and 4).  Allocates nothing. */
int gemm_f32_ladder(const float* A, const float* B, float* C, int M, int N, int K, int step,
                    gemm_f32_stream_t stream);

/* Per-SM arithmetic rates of the units the kernels run on, measured on the
 * current device: the compute peaks of the roofline ("Lesson 10:
 * shared-memory tiled GEMM", hpc.payai.win, section 1, which judges a
 * kernel against the peak of the unit doing its work).  Each figure is
 * FLOP per SM per SM clock cycle (2 per multiply-add), the median over the
 * SMs of kernels that do nothing else -- no loads, no stores in the timed
 * span -- counted with the SM's own cycle counter, so it holds at any clock:
 *   tf32_flop_per_clk_sm       tcgen05.mma kind::tf32, cta_group::1,
 *                              M = 128, N = 256, K = 8, back to back
 *   tf32_pair_flop_per_clk_sm  the same on SM pairs (cta_group::2, M = 256),
 *                              per SM
 *   ffma_flop_per_clk_sm       fma.rn.f32x2 chains, 16 warps per SM
 *   sm_mhz                     SM clock during the probes (cycles over
 *                              globaltimer nanoseconds), median
 *   num_sms                    multiprocessors of the device
 * A peak in FLOP/s is rate x num_sms x the clock the measured kernel ran at.
 * Synchronises the device, allocates and frees a small buffer, takes a few
 * milliseconds.  Returns 0, GEMM_F32_EINVAL (null pointer), GEMM_F32_EDEVICE
 * (not sm_103), GEMM_F32_ELAUNCH or GEMM_F32_ETIMEOUT (the bounded wait for
 * the MMAs ran out). */
typedef struct {
    double tf32_flop_per_clk_sm;
    double tf32_pair_flop_per_clk_sm;
    double ffma_flop_per_clk_sm;
    double sm_mhz;
    int num_sms;
} gemm_f32_unit_rates_t;

int gemm_f32_unit_rates(gemm_f32_unit_rates_t* rates);

/* Static version string, e.g. "gemm_f32 1.0 sm_103a"; the debug library
 * built with -DGEMM_BOUNDS_CHECK (libgemm_f32_checked.so) appends
 * " bounds-checked".  In that build every hand-indexed global load and store
 * is checked against its array's extent: an index outside records site
 * 16 (A), 17 (B), 18 (C), 19 (split-tail partials) or 20 (operand copies)
 * in the error word that gemm_f32_status() reads, and the access is
 * skipped, as out-of-range elements are in "Lesson 10: shared-memory tiled
 * GEMM" (hpc.payai.win, section 3). */
const char* gemm_f32_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F32_H */
