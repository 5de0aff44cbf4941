// noalloc.cu -- cider_w8a8_linear_noalloc: the W8A8 linear without any
// device-memory allocation.
//
// cider_w8a8_linear takes its scratch (the quantized activation codes and the
// per-token scales) from a stream-ordered memory pool.  Some callers must not
// allocate while they run: an inference engine that reserved nearly all of
// HBM for its weights and KV cache before serving starts, or a latency-bound
// decode loop that may not let the allocator grow its pool (which can fail
// under memory pressure or stall on the driver).  This entry point serves
// them from one fixed scratch array in device global memory instead.
//
// The array lives for as long as the library is loaded: every GPU on which it
// has been used keeps it until the process exits.  All calls share it, so
// two calls whose kernels overlap on the GPU (different streams without an
// ordering between them, or different host threads) race on its contents and
// give wrong results; calls on one stream are ordered and safe.  Each call
// overwrites every scratch byte it reads (the quantization kernel writes all
// codes and scales before the GEMM reads them), so nothing needs clearing
// between calls.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>

#include "cider.h"
#include "cider_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = CIDER_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (the host-side symbol is only a stand-in, not a device
// address).  0 = not looked up yet.
std::atomic<uintptr_t> g_scratch_addr[kMaxDevices];

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

cider_status_t scratch_for_current_device(void** out, int* num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CIDER_ERR_UNSUPPORTED_DEVICE;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return CIDER_ERR_UNSUPPORTED_DEVICE;
  }
  if (major != 10 || minor != 3) return CIDER_ERR_UNSUPPORTED_DEVICE;
  uintptr_t a = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (a == 0) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return CIDER_ERR_CUDA;
    }
    a = reinterpret_cast<uintptr_t>(p);
    g_scratch_addr[dev].store(a, std::memory_order_release);
  }
  *out = reinterpret_cast<void*>(a);
  *num_sms = sms;
  return CIDER_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Scratch bytes one call needs: for the tensor-core path the activation
// codes, per-token scales and per-token sums of |code|; none for small M.
size_t noalloc_scratch_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0) return 0;
  const size_t mk = static_cast<size_t>(M) * static_cast<size_t>(K);
  if (cider::gemv_fits(M, K)) return 0;  // the small-M kernel quantizes in shared memory
  return round256(2 * mk) + 2 * round256(4 * static_cast<size_t>(M));
}

}  // namespace

extern "C" cider_status_t cider_w8a8_linear_noalloc(const void* x, int64_t M, int64_t N, int64_t K,
                                                    const int8_t* qw, const float* sw,
                                                    int granularity, int group_size, void* y,
                                                    void* stream) {
  try {
    if (M == 0 || N == 0) return CIDER_OK;
    if (M < 0 || N < 0 || M > 2147483647 || N > 2147483647) return CIDER_ERR_INVALID_ARGUMENT;
    if (!x || !qw || !sw || !y) return CIDER_ERR_INVALID_ARGUMENT;
    if (K < 32 || K % 32 != 0 || K > 131072 || N % 8 != 0) return CIDER_ERR_INVALID_ARGUMENT;
    if (granularity == CIDER_PER_CHANNEL) {
      if (group_size != 0) return CIDER_ERR_INVALID_ARGUMENT;
    } else if (granularity == CIDER_PER_GROUP) {
      if (!((group_size == 64 || group_size == 128) && K % group_size == 0))
        return CIDER_ERR_INVALID_ARGUMENT;
    } else {
      return CIDER_ERR_INVALID_ARGUMENT;
    }
    if (noalloc_scratch_bytes(M, K) > kNoallocScratchBytes) return CIDER_ERR_INVALID_ARGUMENT;
    if (!aligned(x, 16) || !aligned(qw, 16) || !aligned(y, 16) || !aligned(sw, 4))
      return CIDER_ERR_MISALIGNED;
    const char* force = getenv("CIDER_FORCE_UNSUPPORTED");
    if (force && force[0] == '1') return CIDER_ERR_UNSUPPORTED_DEVICE;
    void* scratch = nullptr;
    int sms = 0;
    cider_status_t s = scratch_for_current_device(&scratch, &sms);
    if (s != CIDER_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* w = reinterpret_cast<const uint8_t*>(qw);
    __half* yh = static_cast<__half*>(y);
    uint8_t* base = static_cast<uint8_t*>(scratch);
    cudaError_t e;
    (void)base;
    if (cider::gemv_fits(M, K)) {
      e = cider::launch_gemv(static_cast<const __half*>(x), nullptr, nullptr, M, N, K, w, false, sw,
                             group_size, cider::kEpiY, yh, nullptr, /*no K split*/ nullptr, sms, st);
    } else {
      const size_t qbytes = round256(2 * static_cast<size_t>(M) * static_cast<size_t>(K));
      const size_t vbytes = round256(4 * static_cast<size_t>(M));
      __half* q16 = reinterpret_cast<__half*>(base);
      float* sa = reinterpret_cast<float*>(base + qbytes);
      int* row_l1 = reinterpret_cast<int*>(base + qbytes + vbytes);
      e = cider::launch_quant_act_f16(static_cast<const __half*>(x), M, K, q16, sa, row_l1,
                                      nullptr, 0, st);
      if (e == cudaSuccess)   // no workspace: every output tile is computed whole by one CTA pair
        e = cider::launch_gemm_tc(q16, sa, row_l1, M, N, K, w, false, sw, group_size, cider::kEpiY,
                                  yh, nullptr, nullptr, sms, st);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return CIDER_ERR_CUDA;
    }
    return CIDER_OK;
  } catch (...) {
    return CIDER_ERR_CUDA;
  }
}
