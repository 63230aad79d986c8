// C-ABI front end of libgemm_f32: argument checks, per-device set-up, the
// K == 0 case, mode selection and the device error word.  The operation and
// the contract of each entry point are documented in include/gemm_f32.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/gemm_f32.h"
#include "device_common.cuh"
#include "launch.h"

namespace {

// One block of device words per device.  Word 0 is the error word: 0, or
// the site code of the first bounded wait (or, in the checked build, the
// first out-of-range index) since the last gemm_f32_status() on that device.
// Words 4..7 are the clock record (two 64-bit sums, SM clocks and
// nanoseconds of CTA 0 of each pair and FFMA launch), read by
// gemm_f32_clock_record().
__device__ __align__(16) unsigned g_device_words[8];

constexpr int kMaxDevices = 64;

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  void* pack = nullptr;           // repacked operands for the TMA path
  size_t pack_bytes = 0;
};

struct DeviceState {
  std::once_flag once;
  int status = GEMM_F32_EDEVICE;  // GEMM_F32_OK once set up
  int num_sms = 0;
  unsigned* err = nullptr;        // device address of g_device_words
  std::mutex fixed_mu;
  void* fixed_scratch = nullptr;  // device address of gemm_f32_noalloc's array
  std::mutex ws_mu;
  std::unordered_map<cudaStream_t, Workspace> ws;  // one per stream
};

DeviceState g_devices[kMaxDevices];
thread_local int t_last_launches = 0;
thread_local const char* t_last_kernel = "none";

// Set-up runs once per device, with that device current: checks it is an
// sm_103 part, reads the SM count, takes the address of the error word and
// clears it, and looks up the address of gemm_f32_noalloc's fixed scratch
// array (which, under lazy module loading, loads the module that holds it:
// the array is placed here, at the library's first call on the device, not
// inside a later gemm_f32_noalloc call).
DeviceState* device_state(int* device_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return nullptr;
  }
  *device_out = dev;
  DeviceState& st = g_devices[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return;
    }
    if (major != 10 || minor != 3) return;  // the kernels are built for sm_103a only
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_words) != cudaSuccess) {
      (void)cudaGetLastError();
      return;
    }
    const unsigned zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (cudaMemcpy(p, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      (void)cudaGetLastError();
      return;
    }
    st.num_sms = sms;
    st.err = static_cast<unsigned*>(p);
    st.fixed_scratch = gemm_f32_impl::fixed_scratch_address();   // retried if null
    st.status = GEMM_F32_OK;
  });
  return &st;
}

// The fixed scratch array's device address on the current device, looked up
// again if the set-up could not get it (a failed lookup is not kept).
void* fixed_scratch(DeviceState* st) {
  std::lock_guard<std::mutex> lock(st->fixed_mu);
  if (!st->fixed_scratch) st->fixed_scratch = gemm_f32_impl::fixed_scratch_address();
  return st->fixed_scratch;
}

int default_mode() {
  static const int mode = [] {
    const char* s = std::getenv("GEMM_F32_MODE");
    if (s && std::strcmp(s, "ffma") == 0) return static_cast<int>(GEMM_F32_MODE_FFMA);
    if (s && std::strcmp(s, "tc1x") == 0) return static_cast<int>(GEMM_F32_MODE_TC1X);
    return static_cast<int>(GEMM_F32_MODE_TC3X);
  }();
  return mode;
}

bool overlaps(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a_bytes && b_bytes && a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

constexpr unsigned kKnownFlags = GEMM_F32_FLAG_FORCE_STAGED | GEMM_F32_FLAG_TILE64 |
                                 GEMM_F32_FLAG_TILE128 | GEMM_F32_FLAG_TILE224 |
                                 GEMM_F32_FLAG_TILE256 |
                                 GEMM_F32_FLAG_ONE_TILE_PER_CTA | GEMM_F32_FLAG_NO_SPLIT_K |
                                 GEMM_F32_FLAG_CTA_PAIR | GEMM_F32_FLAG_SINGLE_CTA |
                                 GEMM_F32_FLAG_TEST_DROP_COPY;

}  // namespace

void* gemm_f32_impl::acquire_workspace(int device, cudaStream_t stream, size_t bytes) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  DeviceState& st = g_devices[device];
  std::lock_guard<std::mutex> lock(st.ws_mu);
  Workspace& w = st.ws[stream];
  if (w.bytes < bytes) {
    if (w.ptr) {
      (void)cudaFree(w.ptr);   // synchronises the device: no kernel still uses it
      w.ptr = nullptr;
      w.bytes = 0;
    }
    const size_t want = (bytes + (1u << 20) - 1) & ~static_cast<size_t>((1u << 20) - 1);
    void* p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    if (cudaMemset(p, 0, want) != cudaSuccess) {
      (void)cudaGetLastError();
      (void)cudaFree(p);
      return nullptr;
    }
    w.ptr = p;
    w.bytes = want;
  }
  return w.ptr;
}

namespace {

// Checks of the operands shared by the entry points, before any CUDA call:
// GEMM_F32_EINVAL, or 1 when there is nothing to compute (M or N zero), or 0.
int check_operands(const float* A, const float* B, const float* C, int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return GEMM_F32_EINVAL;
  if (M == 0 || N == 0) return 1;
  const size_t c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
  const size_t a_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * sizeof(float);
  const size_t b_bytes = static_cast<size_t>(K) * static_cast<size_t>(N) * sizeof(float);
  if (C == nullptr) return GEMM_F32_EINVAL;
  if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_F32_EINVAL;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 3u)
    return GEMM_F32_EINVAL;
  if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)) return GEMM_F32_EINVAL;
  return 0;
}

// C = beta * C over an M x N window with row stride ldc (C = 0 when beta
// is 0, without reading C).  The general form's case of an empty or
// zero-weighted product.
__global__ void scale_window_kernel(float* C, int M, int N, int ldc, float beta, unsigned* err) {
  const long long total = static_cast<long long>(M) * N;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long at = (t / N) * static_cast<long long>(ldc) + t % N;
    if (!GEMM_IN_EXTENT(at, gemm_f32_dev::stored_extent(M, N, ldc), err,
                        gemm_f32_dev::kSiteBoundsC))
      continue;
    float* c = C + at;
    *c = beta != 0.0f ? beta * *c : 0.0f;
  }
}

int scale_window(float* C, int M, int N, int ldc, float beta, int num_sms, unsigned* err,
                 cudaStream_t stream) {
  const long long total = static_cast<long long>(M) * N;
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 4LL * num_sms ? want : 4LL * num_sms);
  scale_window_kernel<<<grid, 256, 0, stream>>>(C, M, N, ldc, beta, err);
  if (cudaGetLastError() != cudaSuccess) return GEMM_F32_ELAUNCH;
  t_last_launches = 1;
  t_last_kernel = "scale_window_kernel";
  return GEMM_F32_OK;
}

// K == 0: an empty sum, C = 0.
int zero_fill(float* C, int M, int N, cudaStream_t stream) {
  const size_t c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
  if (cudaMemsetAsync(C, 0, c_bytes, stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  t_last_launches = 1;
  t_last_kernel = "memset";
  return GEMM_F32_OK;
}

}  // namespace

void* gemm_f32_impl::acquire_pack_buffer(int device, cudaStream_t stream, size_t bytes) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  DeviceState& st = g_devices[device];
  std::lock_guard<std::mutex> lock(st.ws_mu);
  Workspace& w = st.ws[stream];
  if (w.pack_bytes < bytes) {
    if (w.pack) {
      (void)cudaFree(w.pack);   // synchronises the device: no kernel still uses it
      w.pack = nullptr;
      w.pack_bytes = 0;
    }
    const size_t want = (bytes + (1u << 20) - 1) & ~static_cast<size_t>((1u << 20) - 1);
    void* p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    w.pack = p;
    w.pack_bytes = want;
  }
  return w.pack;
}

extern "C" int gemm_f32_ex(const float* A, const float* B, float* C, int M, int N, int K, int mode,
                           unsigned flags, gemm_f32_stream_t stream_handle) {
  t_last_launches = 0;
  t_last_kernel = "none";
  // ---- host-only checks first: no CUDA call for a malformed request
  if (M < 0 || N < 0 || K < 0) return GEMM_F32_EINVAL;
  if (mode != GEMM_F32_MODE_TC3X && mode != GEMM_F32_MODE_FFMA && mode != GEMM_F32_MODE_TC1X)
    return GEMM_F32_EINVAL;
  if (flags & ~kKnownFlags) return GEMM_F32_EINVAL;
  const unsigned bn_flags = flags & (GEMM_F32_FLAG_TILE64 | GEMM_F32_FLAG_TILE128 |
                                     GEMM_F32_FLAG_TILE224 | GEMM_F32_FLAG_TILE256);
  if (bn_flags & (bn_flags - 1)) return GEMM_F32_EINVAL;  // at most one tile width
  if ((flags & GEMM_F32_FLAG_CTA_PAIR) && (flags & GEMM_F32_FLAG_SINGLE_CTA)) return GEMM_F32_EINVAL;
  const int chk = check_operands(A, B, C, M, N, K);
  if (chk != 0) return chk < 0 ? chk : GEMM_F32_OK;

  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);

  if (K == 0) return zero_fill(C, M, N, stream);

  gemm_f32_impl::GemmArgs g;
  g.A = A;
  g.B = B;
  g.C = C;
  g.M = M;
  g.N = N;
  g.K = K;
  g.lda = K;
  g.ldb = N;
  g.ldc = N;
  g.err = st->err;
  g.num_sms = st->num_sms;
  g.device = dev;
  g.flags = flags;
  int launches = 0;
  int rc;
  if (flags == 0 && gemm_f32_impl::small_suits(g))
    rc = gemm_f32_impl::launch_small(g, stream, &launches);
  else if (mode == GEMM_F32_MODE_FFMA)
    rc = gemm_f32_impl::launch_ffma(g, stream, &launches);
  else
    rc = gemm_f32_impl::launch_tc(g, mode == GEMM_F32_MODE_TC1X ? 1 : 3, stream, &launches);
  if (rc == GEMM_F32_OK) {
    t_last_launches = launches;
    t_last_kernel = g.kernel;
  }
  return rc;
}

extern "C" int gemm_f32(const float* A, const float* B, float* C, int M, int N, int K,
                        gemm_f32_stream_t stream) {
  return gemm_f32_ex(A, B, C, M, N, K, default_mode(), 0u, stream);
}

extern "C" int gemm_f32_ladder(const float* A, const float* B, float* C, int M, int N, int K,
                               int step, gemm_f32_stream_t stream_handle) {
  t_last_launches = 0;
  t_last_kernel = "none";
  if (step < 0 || step > 4) return GEMM_F32_EINVAL;
  const int chk = check_operands(A, B, C, M, N, K);
  if (chk != 0) return chk < 0 ? chk : GEMM_F32_OK;
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  if (K == 0) return zero_fill(C, M, N, stream);
  gemm_f32_impl::GemmArgs g;
  g.A = A;
  g.B = B;
  g.C = C;
  g.M = M;
  g.N = N;
  g.K = K;
  g.lda = K;
  g.ldb = N;
  g.ldc = N;
  g.err = st->err;
  g.num_sms = st->num_sms;
  g.device = dev;
  g.flags = 0;
  int launches = 0;
  const int rc = gemm_f32_impl::launch_ladder(g, step, stream, &launches);
  if (rc == GEMM_F32_OK) {
    t_last_launches = launches;
    t_last_kernel = g.kernel;
  }
  return rc;
}

extern "C" int gemm_f32_general(int trans_a, int trans_b, int M, int N, int K, float alpha,
                                const float* A, int lda, const float* B, int ldb, float beta,
                                float* C, int ldc, int mode, gemm_f32_stream_t stream_handle) {
  t_last_launches = 0;
  t_last_kernel = "none";
  // ---- host-only checks first
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return GEMM_F32_EINVAL;
  if (M < 0 || N < 0 || K < 0) return GEMM_F32_EINVAL;
  if (mode != GEMM_F32_MODE_TC3X && mode != GEMM_F32_MODE_FFMA && mode != GEMM_F32_MODE_TC1X)
    return GEMM_F32_EINVAL;
  const int a_rows = trans_a ? K : M, a_cols = trans_a ? M : K;
  const int b_rows = trans_b ? N : K, b_cols = trans_b ? K : N;
  if (lda < std::max(1, a_cols) || ldb < std::max(1, b_cols) || ldc < std::max(1, N))
    return GEMM_F32_EINVAL;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return GEMM_F32_EINVAL;
  if (M == 0 || N == 0) return GEMM_F32_OK;
  const bool use_ab = K > 0 && alpha != 0.0f;
  if (C == nullptr || (use_ab && (A == nullptr || B == nullptr))) return GEMM_F32_EINVAL;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 3u)
    return GEMM_F32_EINVAL;
  // byte extents of the stored windows (first to last element touched)
  auto extent = [](int rows, int cols, int ld) -> size_t {
    return rows > 0 && cols > 0
               ? (static_cast<size_t>(rows - 1) * static_cast<size_t>(ld) + cols) * sizeof(float)
               : 0;
  };
  const size_t c_bytes = extent(M, N, ldc);
  if (use_ab && (overlaps(C, c_bytes, A, extent(a_rows, a_cols, lda)) ||
                 overlaps(C, c_bytes, B, extent(b_rows, b_cols, ldb))))
    return GEMM_F32_EINVAL;

  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  if (!use_ab) return scale_window(C, M, N, ldc, beta, st->num_sms, st->err, stream);

  gemm_f32_impl::GemmArgs g;
  g.A = A;
  g.B = B;
  g.C = C;
  g.M = M;
  g.N = N;
  g.K = K;
  g.lda = lda;
  g.ldb = ldb;
  g.ldc = ldc;
  g.trans_a = trans_a;
  g.trans_b = trans_b;
  g.alpha = alpha;
  g.beta = beta;
  g.scale = (alpha != 1.0f || beta != 0.0f) ? 1 : 0;
  g.err = st->err;
  g.num_sms = st->num_sms;
  g.device = dev;
  g.flags = 0;
  int launches = 0;
  const int rc = mode == GEMM_F32_MODE_FFMA
                     ? gemm_f32_impl::launch_ffma(g, stream, &launches)
                     : gemm_f32_impl::launch_tc(g, mode == GEMM_F32_MODE_TC1X ? 1 : 3, stream,
                                                &launches);
  if (rc == GEMM_F32_OK) {
    t_last_launches = launches;
    t_last_kernel = g.kernel;
  }
  return rc;
}

// ---------------------------------------------------------------- host buffers
// gemm_f32_host: per device, three streams (copy in, product, copy out) and
// two device slots taken by alternate calls, so that the copies of one call
// overlap the product of its neighbour.  Events order every reuse of a slot:
// its A and B are overwritten only after the product that read them, its C
// only after the copy that drained it.
namespace {

struct HostSlot {
  float* A = nullptr;
  float* B = nullptr;
  float* C = nullptr;
  size_t a_cap = 0, b_cap = 0, c_cap = 0;   // bytes
  cudaEvent_t loaded = nullptr, computed = nullptr, drained = nullptr;
  bool used = false;
};

struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  HostSlot slot[2];
  int next = 0;
};

HostPipe g_pipes[kMaxDevices];

bool host_pipe_init(HostPipe& hp) {
  if (hp.ready) return true;
  for (cudaStream_t* s : {&hp.in, &hp.comp, &hp.out})
    if (cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) != cudaSuccess) return false;
  for (HostSlot& sl : hp.slot)
    for (cudaEvent_t* e : {&sl.loaded, &sl.computed, &sl.drained})
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
  hp.ready = true;
  return true;
}

// Device buffer of at least `need` bytes (1 MiB granules), reallocated only
// when it must grow; the caller has made sure no queued work still uses it.
bool host_slot_buffer(float** p, size_t* cap, size_t need) {
  if (*cap >= need) return true;
  if (*p) (void)cudaFree(*p);
  *p = nullptr;
  *cap = 0;
  const size_t want = (need + (1u << 20) - 1) & ~static_cast<size_t>((1u << 20) - 1);
  if (cudaMalloc(reinterpret_cast<void**>(p), want) != cudaSuccess) return false;
  *cap = want;
  return true;
}

void host_pipe_free(HostPipe& hp) {
  for (HostSlot& sl : hp.slot) {
    for (float** b : {&sl.A, &sl.B, &sl.C}) {
      if (*b) (void)cudaFree(*b);
      *b = nullptr;
    }
    sl.a_cap = sl.b_cap = sl.c_cap = 0;
    sl.used = false;
  }
}

}  // namespace

extern "C" int gemm_f32_host(const float* A, const float* B, float* C, int M, int N, int K,
                             int mode, gemm_f32_stream_t stream_handle) {
  t_last_launches = 0;
  t_last_kernel = "none";
  if (mode != GEMM_F32_MODE_TC3X && mode != GEMM_F32_MODE_FFMA && mode != GEMM_F32_MODE_TC1X)
    return GEMM_F32_EINVAL;
  const int chk = check_operands(A, B, C, M, N, K);
  if (chk != 0) return chk < 0 ? chk : GEMM_F32_OK;
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  const size_t a_bytes = static_cast<size_t>(M) * K * sizeof(float);
  const size_t b_bytes = static_cast<size_t>(K) * N * sizeof(float);
  const size_t c_bytes = static_cast<size_t>(M) * N * sizeof(float);

  HostPipe& hp = g_pipes[dev];
  std::lock_guard<std::mutex> lock(hp.mu);
  auto fail = [] {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  };
  if (!host_pipe_init(hp)) return fail();
  HostSlot& sl = hp.slot[hp.next];
  hp.next ^= 1;
  if (sl.a_cap < a_bytes || sl.b_cap < b_bytes || sl.c_cap < c_bytes) {
    if (sl.used && cudaEventSynchronize(sl.drained) != cudaSuccess) return fail();
    if (!host_slot_buffer(&sl.A, &sl.a_cap, a_bytes) ||
        !host_slot_buffer(&sl.B, &sl.b_cap, b_bytes) ||
        !host_slot_buffer(&sl.C, &sl.c_cap, c_bytes)) {
      host_pipe_free(hp);
      return fail();
    }
  }
  // copy in, once the product that last read this slot is done
  if (sl.used && cudaStreamWaitEvent(hp.in, sl.computed, 0) != cudaSuccess) return fail();
  if (a_bytes && cudaMemcpyAsync(sl.A, A, a_bytes, cudaMemcpyHostToDevice, hp.in) != cudaSuccess)
    return fail();
  if (b_bytes && cudaMemcpyAsync(sl.B, B, b_bytes, cudaMemcpyHostToDevice, hp.in) != cudaSuccess)
    return fail();
  if (cudaEventRecord(sl.loaded, hp.in) != cudaSuccess) return fail();
  // the product, once the operands are in and this slot's last C has drained
  if (cudaStreamWaitEvent(hp.comp, sl.loaded, 0) != cudaSuccess) return fail();
  if (sl.used && cudaStreamWaitEvent(hp.comp, sl.drained, 0) != cudaSuccess) return fail();
  const int rc = gemm_f32_ex(sl.A, sl.B, sl.C, M, N, K, mode, 0u,
                             reinterpret_cast<gemm_f32_stream_t>(hp.comp));
  if (rc != GEMM_F32_OK) return rc;
  const int launches = t_last_launches;
  const char* kernel = t_last_kernel;
  if (cudaEventRecord(sl.computed, hp.comp) != cudaSuccess) return fail();
  // copy out, then the caller's stream waits for it
  if (cudaStreamWaitEvent(hp.out, sl.computed, 0) != cudaSuccess) return fail();
  if (cudaMemcpyAsync(C, sl.C, c_bytes, cudaMemcpyDeviceToHost, hp.out) != cudaSuccess) return fail();
  if (cudaEventRecord(sl.drained, hp.out) != cudaSuccess) return fail();
  sl.used = true;
  if (cudaStreamWaitEvent(stream, sl.drained, 0) != cudaSuccess) return fail();
  t_last_launches = launches;
  t_last_kernel = kernel;
  return GEMM_F32_OK;
}

extern "C" int gemm_f32_noalloc(const float* A, const float* B, float* C, int M, int N, int K,
                                int mode, gemm_f32_stream_t stream_handle) {
  t_last_launches = 0;
  t_last_kernel = "none";
  if (M < 0 || N < 0 || K < 0) return GEMM_F32_EINVAL;
  if (mode != GEMM_F32_MODE_TC3X && mode != GEMM_F32_MODE_TC1X) return GEMM_F32_EINVAL;
  if (M == 0 || N == 0) return GEMM_F32_OK;
  const size_t c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
  const size_t a_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * sizeof(float);
  const size_t b_bytes = static_cast<size_t>(K) * static_cast<size_t>(N) * sizeof(float);
  if (C == nullptr) return GEMM_F32_EINVAL;
  if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_F32_EINVAL;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 3u)
    return GEMM_F32_EINVAL;
  if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)) return GEMM_F32_EINVAL;

  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  if (K == 0) {
    if (cudaMemsetAsync(C, 0, c_bytes, stream) != cudaSuccess) {
      (void)cudaGetLastError();
      return GEMM_F32_ELAUNCH;
    }
    t_last_launches = 1;
    t_last_kernel = "memset";
    return GEMM_F32_OK;
  }
  gemm_f32_impl::GemmArgs g;
  g.A = A;
  g.B = B;
  g.C = C;
  g.M = M;
  g.N = N;
  g.K = K;
  g.lda = K;
  g.ldb = N;
  g.ldc = N;
  g.err = st->err;
  g.num_sms = st->num_sms;
  g.device = dev;
  g.flags = 0;
  int launches = 0;
  const int rc = gemm_f32_impl::launch_tc_fixed_scratch(
      g, mode == GEMM_F32_MODE_TC1X ? 1 : 3, fixed_scratch(st), stream, &launches);
  if (rc == GEMM_F32_OK) {
    t_last_launches = launches;
    t_last_kernel = g.kernel;
  }
  return rc;
}

extern "C" int gemm_f32_status(gemm_f32_stream_t stream_handle, unsigned* site) {
  if (site) *site = 0;
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_handle)) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  unsigned word = 0;
  const unsigned zero = 0;
  if (cudaMemcpy(&word, st->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(st->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  if (site) *site = word;
  return word ? GEMM_F32_ETIMEOUT : GEMM_F32_OK;
}

extern "C" int gemm_f32_clock_record(gemm_f32_stream_t stream_handle,
                                     unsigned long long* sm_cycles, unsigned long long* ns) {
  if (sm_cycles) *sm_cycles = 0;
  if (ns) *ns = 0;
  if (!sm_cycles || !ns) return GEMM_F32_EINVAL;
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_handle)) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  unsigned long long rec[2] = {0, 0};
  if (cudaMemcpy(rec, st->err + 4, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess) {
    (void)cudaGetLastError();
    return GEMM_F32_ELAUNCH;
  }
  *sm_cycles = rec[0];
  *ns = rec[1];
  return GEMM_F32_OK;
}

extern "C" int gemm_f32_release(void) {
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (!st || st->status != GEMM_F32_OK) return GEMM_F32_EDEVICE;
  // same lock order as gemm_f32_host: its pipe, then the workspaces
  std::lock_guard<std::mutex> hlock(g_pipes[dev].mu);
  std::lock_guard<std::mutex> lock(st->ws_mu);
  int rc = GEMM_F32_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    (void)cudaGetLastError();
    rc = GEMM_F32_ELAUNCH;
  }
  for (auto& kv : st->ws) {
    if (kv.second.ptr) (void)cudaFree(kv.second.ptr);
    if (kv.second.pack) (void)cudaFree(kv.second.pack);
  }
  st->ws.clear();
  host_pipe_free(g_pipes[dev]);
  return rc;
}

extern "C" int gemm_f32_last_launches(void) { return t_last_launches; }

extern "C" const char* gemm_f32_last_kernel(void) { return t_last_kernel; }

extern "C" const char* gemm_f32_version(void) {
#ifdef GEMM_BOUNDS_CHECK
  return "gemm_f32 1.0 sm_103a bounds-checked";
#else
  return "gemm_f32 1.0 sm_103a";
#endif
}
