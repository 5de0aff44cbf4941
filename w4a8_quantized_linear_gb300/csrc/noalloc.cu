// noalloc.cu -- cider_w8a8_linear_noalloc: the W8A8 linear without any
// device-memory allocation.
//
// cider_w8a8_linear takes its scratch (the quantized activation codes and the
// per-token scales) from a stream-ordered memory pool.  Some callers must not
// allocate while they run: an inference engine that reserved nearly all of
// HBM for its weights and KV cache before serving starts, or a latency-bound
// decode loop that may not let the allocator grow its pool (which can fail
// under memory pressure or stall on the driver).  This entry point serves
// them from one fixed scratch array in device global memory instead, and
// otherwise runs exactly the dispatch and kernels of cider_w8a8_linear (the
// same argument and device checks, the same small-M and tensor-core paths);
// only the optional work-split buffers are left out when the array has no
// room for them beside the codes, which changes the speed, not the result.
//
// The array lives for as long as the library is loaded: every GPU on which it
// has been used keeps it until the process exits.  All calls share it, so
// two calls whose kernels overlap on the GPU (different streams without an
// ordering between them, or different host threads) race on its contents and
// give wrong results; calls on one stream are ordered and safe.  Each call
// writes every scratch byte it later reads (the quantization kernel writes
// all codes and scales, and clears the GEMM's work-split flags, before the
// GEMM reads them), so nothing left by an earlier call is ever used.
#include <cuda_runtime.h>
#include <stdint.h>

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

cider_status_t scratch_for_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return CIDER_ERR_UNSUPPORTED_DEVICE;
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
  return CIDER_OK;
}

}  // namespace

extern "C" cider_status_t cider_w8a8_linear_noalloc(const void* x, int64_t M, int64_t N, int64_t K,
                                                    const int8_t* qw, const float* sw,
                                                    int granularity, int group_size, void* y,
                                                    void* stream) {
  try {
    if (M == 0 || N == 0) return CIDER_OK;
    if (!x) return CIDER_ERR_INVALID_ARGUMENT;
    cider::LinearArgs a;
    a.x = x;
    a.M = M;
    a.N = N;
    a.K = K;
    a.w = qw;
    a.sw = sw;
    a.granularity = granularity;
    a.group_size = group_size;
    a.y = y;
    a.mode = cider::kEpiY;
    a.st = static_cast<cudaStream_t>(stream);
    cider_status_t s = cider::validate_linear(a);
    if (s != CIDER_OK) return s;
    // the codes and per-token values must fit; checked before the device is touched
    if (cider::linear_required_scratch(a) > kNoallocScratchBytes) return CIDER_ERR_INVALID_ARGUMENT;
    int dev = 0;
    s = cider::check_device(&dev, nullptr);
    if (s != CIDER_OK) return s;
    void* base = nullptr;
    s = scratch_for_device(dev, &base);
    if (s != CIDER_OK) return s;
    cider::ScratchSource scratch = cider::ScratchSource::fixed(base, kNoallocScratchBytes);
    return cider::run_linear(a, scratch);
  } catch (...) {
    return CIDER_ERR_CUDA;
  }
}
