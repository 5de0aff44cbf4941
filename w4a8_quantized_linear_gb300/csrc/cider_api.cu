// cider_api.cu -- the C ABI declared in include/cider.h: argument checks,
// device check, scratch memory from a per-device stream-ordered pool, and
// the dispatch by M between the small-M GEMV and the tensor-core GEMM.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "cider.h"
#include "cider_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxK = 131072;  // keeps |acc| <= 16129 * K below 2^31
constexpr int64_t kMaxDim = 2147483647;

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 supported, 2 unsupported
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};

bool force_unsupported() {
  const char* v = getenv("CIDER_FORCE_UNSUPPORTED");
  return v != nullptr && v[0] == '1';
}

cudaError_t get_pool(int dev, cudaMemPool_t* pool) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p;
    cudaError_t e = cudaMemPoolCreate(&p, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse by later calls
    e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(p);
      return e;
    }
    g_pool[dev] = p;
  }
  *pool = g_pool[dev];
  return cudaSuccess;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cider_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CIDER_OK;
  cudaGetLastError();  // clear a sticky launch error so later calls start clean
  return CIDER_ERR_CUDA;
}

bool valid_k(int64_t K) { return K >= 32 && K % 32 == 0 && K <= kMaxK; }

// Granularity / group size rules shared by the linears.
bool valid_grouping(int granularity, int group_size, int64_t K) {
  if (granularity == CIDER_PER_CHANNEL) return group_size == 0;
  if (granularity == CIDER_PER_GROUP)
    return (group_size == 64 || group_size == 128) && K % group_size == 0;
  return false;
}

// Per-thread kernel timing (cider_timing_begin / cider_timing_end).
struct KernelTimer {
  std::vector<cudaEvent_t> ev;  // pairs: 2 i (before), 2 i + 1 (after)
  int64_t used = 0;
  bool on = false;
};
thread_local KernelTimer t_timer;

void timer_release() {
  for (cudaEvent_t e : t_timer.ev) cudaEventDestroy(e);
  t_timer.ev.clear();
  t_timer.used = 0;
  t_timer.on = false;
}

// Record a timing event; inside a stream capture the record must become a
// graph node (an external record), or it would only mark a dependency.
cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

// Launch one GEMM kernel, bracketed by the next event pair when timing is on.
template <typename F>
cudaError_t timed_launch(cudaStream_t st, F&& launch) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (t_timer.on && 2 * (t_timer.used + 1) <= static_cast<int64_t>(t_timer.ev.size())) {
    e0 = t_timer.ev[2 * t_timer.used];
    e1 = t_timer.ev[2 * t_timer.used + 1];
  }
  if (e0) {
    cudaError_t e = record_timing_event(e0, st);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) return e;
  if (e1) {
    e = record_timing_event(e1, st);
    if (e != cudaSuccess) return e;
    ++t_timer.used;
  }
  return cudaSuccess;
}

template <typename F>
cider_status_t guarded(F&& f) {
  try {
    return f();
  } catch (...) {
    return CIDER_ERR_CUDA;
  }
}

// clip_percentile < 0: min-max scales; else percentile-clipped ones.
cider_status_t quantize_weight(const float* w, int64_t N, int64_t K, int group_size, void* q,
                               float* sw, bool int4, void* stream, double clip_percentile = -1.0) {
  if (N == 0) return CIDER_OK;
  if (N < 0 || N > kMaxDim || !w || !q || !sw || !valid_k(K)) return CIDER_ERR_INVALID_ARGUMENT;
  if (!(group_size == 0 || ((group_size == 64 || group_size == 128) && K % group_size == 0)))
    return CIDER_ERR_INVALID_ARGUMENT;
  if (!aligned(w, 16) || !aligned(q, 16)) return CIDER_ERR_MISALIGNED;
  if (!aligned(sw, 4)) return CIDER_ERR_MISALIGNED;
  cider_status_t s = cider::check_device(nullptr, nullptr);
  if (s != CIDER_OK) return s;
  if (clip_percentile >= 0.0)
    return cuda_status(cider::launch_quant_weight_clip(w, N, K, group_size, clip_percentile, int4,
                                                       static_cast<uint8_t*>(q), sw,
                                                       static_cast<cudaStream_t>(stream)));
  return cuda_status(cider::launch_quant_weight(w, N, K, group_size, int4,
                                                static_cast<uint8_t*>(q), sw,
                                                static_cast<cudaStream_t>(stream)));
}

bool valid_percentile(double p) { return p > 0.0 && p <= 100.0; }   // false for NaN

}  // namespace

namespace cider {

// Supported = compute capability 10.3 (GB300).  Caches the SM count.
cider_status_t check_device(int* dev_out, int* num_sms) {
  if (force_unsupported()) return CIDER_ERR_UNSUPPORTED_DEVICE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CIDER_ERR_UNSUPPORTED_DEVICE;
  }
  DeviceInfo& d = g_dev[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    if (!ok) cudaGetLastError();
    ok = ok && major == 10 && minor == 3 && sms > 0;
    d.num_sms = sms;
    st = ok ? 1 : 2;
    d.state.store(st, std::memory_order_release);
  }
  if (st != 1) return CIDER_ERR_UNSUPPORTED_DEVICE;
  if (dev_out) *dev_out = dev;
  if (num_sms) *num_sms = d.num_sms;
  return CIDER_OK;
}

ScratchSource::ScratchSource(ScratchSource&& o) noexcept
    : st_(o.st_), base_(o.base_), capacity_(o.capacity_), pool_ptr_(o.pool_ptr_) {
  o.pool_ptr_ = nullptr;
}

ScratchSource::~ScratchSource() {
  if (pool_ptr_) cudaFreeAsync(pool_ptr_, st_);
}

cider_status_t ScratchSource::get(size_t bytes, void** out) {
  if (base_ != nullptr) {
    if (bytes > capacity_) return CIDER_ERR_INVALID_ARGUMENT;
    *out = base_;
    return CIDER_OK;
  }
  if (pool_ptr_ != nullptr) return CIDER_ERR_INVALID_ARGUMENT;   // one request per call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_status(cudaErrorInvalidDevice);
  cudaMemPool_t pool;
  e = get_pool(dev, &pool);
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&pool_ptr_, bytes, pool, st_);
  if (e != cudaSuccess) {
    pool_ptr_ = nullptr;
    return cuda_status(e);
  }
  *out = pool_ptr_;
  return CIDER_OK;
}

cider_status_t validate_linear(const LinearArgs& a) {
  if (a.M < 0 || a.N < 0 || a.K < 0) return CIDER_ERR_INVALID_ARGUMENT;
  if (a.M > kMaxDim || a.N > kMaxDim) return CIDER_ERR_INVALID_ARGUMENT;
  const bool prequant = a.x == nullptr;
  if (prequant ? (!a.qa || (a.mode != kEpiAcc && !a.sa)) : false)
    return CIDER_ERR_INVALID_ARGUMENT;
  if (!a.w) return CIDER_ERR_INVALID_ARGUMENT;
  if (a.mode != kEpiAcc && (!a.sw || !a.y)) return CIDER_ERR_INVALID_ARGUMENT;
  if (a.mode == kEpiAcc && !a.acc) return CIDER_ERR_INVALID_ARGUMENT;
  if (!valid_k(a.K) || a.N % 8 != 0) return CIDER_ERR_INVALID_ARGUMENT;
  if (a.mode != kEpiAcc) {
    if (!valid_grouping(a.granularity, a.group_size, a.K)) return CIDER_ERR_INVALID_ARGUMENT;
  } else {
    if (!(a.group_size == 0 || ((a.group_size == 64 || a.group_size == 128) && a.K % a.group_size == 0)))
      return CIDER_ERR_INVALID_ARGUMENT;
  }
  if ((a.x && !aligned(a.x, 16)) || (a.qa && !aligned(a.qa, 16)) || !aligned(a.w, 16) ||
      (a.y && !aligned(a.y, 16)))
    return CIDER_ERR_MISALIGNED;
  if ((a.sa && !aligned(a.sa, 4)) || (a.sw && !aligned(a.sw, 4)) || (a.acc && !aligned(a.acc, 4)))
    return CIDER_ERR_MISALIGNED;
  return CIDER_OK;
}

size_t linear_required_scratch(const LinearArgs& a) {
  if (a.M <= 0 || a.N <= 0 || a.K <= 0) return 0;
  if (gemv_fits(a.M, a.K)) {
    const bool quantize_first =
        a.x && (a.x_bf16 || a.mode == kEpiYb || !gemv_quantizes_itself(a.M, a.K));
    return quantize_first ? round_up(static_cast<size_t>(a.M * a.K), 256) + round_up(4 * a.M, 256)
                          : 0;
  }
  return round_up(static_cast<size_t>(a.M * a.K) * 2, 256) + 2 * round_up(4 * a.M, 256);
}

cider_status_t run_linear(const LinearArgs& a, ScratchSource& scratch) {
  if (a.M == 0 || a.N == 0) return CIDER_OK;
  cider_status_t s = validate_linear(a);
  if (s != CIDER_OK) return s;
  int dev = 0, sms = 0;
  s = check_device(&dev, &sms);
  if (s != CIDER_OK) return s;
  const uint8_t* w = static_cast<const uint8_t*>(a.w);
  __half* y = static_cast<__half*>(a.y);
  const int gs = a.group_size;
  if (gemv_fits(a.M, a.K)) {
    // small M: for one token or short rows the GEMV quantizes the rows itself
    // (every CTA repeats that work, cheaper than a second launch for so few
    // values); otherwise one quantization kernel writes the int8 codes first.
    // bf16 rows, and problems whose K is split over several CTAs per row
    // block, always take the quantization kernel, as do bf16 outputs (the
    // kernel that quantizes its own rows writes fp16).  The K split's partial
    // sums are optional scratch: without room for them the row blocks stay
    // whole.
    const size_t qs_bytes = round_up(static_cast<size_t>(a.M * a.K), 256) + round_up(4 * a.M, 256);
    size_t pbytes = gemv_part_bytes(a.M, a.N, a.K, a.int4, gs, a.mode, sms);
    if (pbytes > 0 && !scratch.fits((a.x ? qs_bytes : 0) + round_up(pbytes, 256))) pbytes = 0;
    const __half* xg = static_cast<const __half*>(a.x);
    const int8_t* qa = a.qa;
    const float* sa = a.sa;
    void* part = nullptr;
    const bool quantize_first =
        a.x && (a.x_bf16 || a.mode == kEpiYb || pbytes > 0 || !gemv_quantizes_itself(a.M, a.K));
    const size_t qbytes = quantize_first ? round_up(static_cast<size_t>(a.M * a.K), 256) : 0;
    const size_t sbytes = quantize_first ? round_up(4 * a.M, 256) : 0;
    // the GEMV overlaps the quantization launch just before it, unless a
    // kernel-timing event is recorded between the two
    const bool overlap = quantize_first && !t_timer.on;
    if (qbytes + sbytes + pbytes > 0) {
      void* sp = nullptr;
      s = scratch.get(qbytes + sbytes + round_up(pbytes, 256), &sp);
      if (s != CIDER_OK) return s;
      uint8_t* base = static_cast<uint8_t*>(sp);
      if (pbytes > 0) part = base + qbytes + sbytes;
      if (quantize_first) {
        int8_t* qs = reinterpret_cast<int8_t*>(base);
        float* ss = reinterpret_cast<float*>(base + qbytes);
        cudaError_t e = a.x_bf16 ? launch_quant_act_s8_bf16(static_cast<const __nv_bfloat16*>(a.x),
                                                            a.M, a.K, qs, ss, a.st, overlap)
                                 : launch_quant_act_s8(xg, a.M, a.K, qs, ss, a.st, overlap);
        if (e != cudaSuccess) return cuda_status(e);
        xg = nullptr;
        qa = qs;
        sa = ss;
      }
    }
    return cuda_status(timed_launch(a.st, [&] {
      return launch_gemv(xg, qa, sa, a.M, a.N, a.K, w, a.int4, a.sw, gs, a.mode, y, a.acc, part,
                         sms, a.st, overlap);
    }));
  }
  // tensor-core path: activation codes as fp16 integers, scales, row sums of
  // |code|; the per-channel GEMM's K-piece workspace is optional scratch
  // (without it every output tile is computed whole by one CTA pair)
  const size_t qbytes = round_up(static_cast<size_t>(a.M * a.K) * 2, 256);
  const size_t vbytes = round_up(4 * a.M, 256);
  GemmScratch gsc = gemm_tc_scratch(a.M, a.N, a.K, gs);
  if (gsc.bytes > 0 && !scratch.fits(qbytes + 2 * vbytes + gsc.bytes)) gsc = GemmScratch{};
  void* sp = nullptr;
  s = scratch.get(qbytes + 2 * vbytes + gsc.bytes, &sp);
  if (s != CIDER_OK) return s;
  uint8_t* sbase = static_cast<uint8_t*>(sp);
  __half* q16 = reinterpret_cast<__half*>(sbase);
  int* row_l1 = reinterpret_cast<int*>(sbase + qbytes + vbytes);
  uint8_t* ws = gsc.bytes ? sbase + qbytes + 2 * vbytes : nullptr;
  int* zero = ws ? reinterpret_cast<int*>(ws + gsc.zero_offset) : nullptr;
  const float* sa = a.sa;
  // the GEMM overlaps its set-up with the quantization launch just before it,
  // unless a kernel-timing event is recorded between the two
  const bool overlap = !t_timer.on;
  cudaError_t e;
  if (a.x) {
    float* sscr = reinterpret_cast<float*>(sbase + qbytes);
    e = a.x_bf16 ? launch_quant_act_f16_from_bf16(static_cast<const __nv_bfloat16*>(a.x), a.M, a.K,
                                                  q16, sscr, row_l1, zero, gsc.zero_words, a.st,
                                                  overlap)
                 : launch_quant_act_f16(static_cast<const __half*>(a.x), a.M, a.K, q16, sscr,
                                        row_l1, zero, gsc.zero_words, a.st, overlap);
    sa = sscr;
  } else {
    e = launch_codes_s8_to_f16(a.qa, a.M, a.K, q16, row_l1, zero, gsc.zero_words, a.st);
  }
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(timed_launch(a.st, [&] {
    return launch_gemm_tc(q16, sa, row_l1, a.M, a.N, a.K, w, a.int4, a.sw, gs, a.mode, y, a.acc,
                          ws, sms, a.st, overlap);
  }));
}

}  // namespace cider

extern "C" {

int cider_version(void) { return 100; }

int cider_is_available(void) { return cider::check_device(nullptr, nullptr) == CIDER_OK ? 1 : 0; }

const char* cider_status_string(int status) {
  switch (status) {
    case CIDER_OK: return "CIDER_OK";
    case CIDER_ERR_INVALID_ARGUMENT: return "CIDER_ERR_INVALID_ARGUMENT: bad size, pointer or mode";
    case CIDER_ERR_MISALIGNED: return "CIDER_ERR_MISALIGNED: a pointer is not aligned as required";
    case CIDER_ERR_UNSUPPORTED_DEVICE: return "CIDER_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
    case CIDER_ERR_CUDA: return "CIDER_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case CIDER_ERR_TIMEOUT: return "CIDER_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    default: return "unknown cider status";
  }
}

static cider_status_t quantize_act_entry(const void* x, bool bf16, int64_t M, int64_t K, int8_t* qa,
                                         float* sa, void* stream) {
  return guarded([&]() -> cider_status_t {
    if (M == 0) return CIDER_OK;
    if (M < 0 || M > kMaxDim || !x || !qa || !sa || !valid_k(K)) return CIDER_ERR_INVALID_ARGUMENT;
    if (!aligned(x, 16) || !aligned(qa, 16)) return CIDER_ERR_MISALIGNED;
    if (!aligned(sa, 4)) return CIDER_ERR_MISALIGNED;
    cider_status_t s = cider::check_device(nullptr, nullptr);
    if (s != CIDER_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(bf16 ? cider::launch_quant_act_s8_bf16(static_cast<const __nv_bfloat16*>(x),
                                                              M, K, qa, sa, st)
                            : cider::launch_quant_act_s8(static_cast<const __half*>(x), M, K, qa,
                                                         sa, st));
  });
}

cider_status_t cider_quantize_act(const void* x, int64_t M, int64_t K, int8_t* qa, float* sa,
                                  void* stream) {
  return quantize_act_entry(x, false, M, K, qa, sa, stream);
}

cider_status_t cider_quantize_act_bf16(const void* x, int64_t M, int64_t K, int8_t* qa, float* sa,
                                       void* stream) {
  return quantize_act_entry(x, true, M, K, qa, sa, stream);
}

cider_status_t cider_int4_from_offset_binary(const uint8_t* src, uint8_t* dst, int64_t nbytes,
                                             void* stream) {
  return guarded([&]() -> cider_status_t {
    if (nbytes == 0) return CIDER_OK;
    if (nbytes < 0 || !src || !dst) return CIDER_ERR_INVALID_ARGUMENT;
    if (!aligned(src, 16) || !aligned(dst, 16)) return CIDER_ERR_MISALIGNED;
    cider_status_t s = cider::check_device(nullptr, nullptr);
    if (s != CIDER_OK) return s;
    return cuda_status(
        cider::launch_int4_from_offset(src, dst, nbytes, static_cast<cudaStream_t>(stream)));
  });
}

cider_status_t cider_quantize_weight_int8(const float* w, int64_t N, int64_t K, int group_size,
                                          int8_t* qw, float* sw, void* stream) {
  return guarded([&] { return quantize_weight(w, N, K, group_size, qw, sw, false, stream); });
}

cider_status_t cider_quantize_weight_int4(const float* w, int64_t N, int64_t K, int group_size,
                                          uint8_t* qw_packed, float* sw, void* stream) {
  return guarded([&] { return quantize_weight(w, N, K, group_size, qw_packed, sw, true, stream); });
}

cider_status_t cider_quantize_weight_int8_clip(const float* w, int64_t N, int64_t K,
                                               int group_size, double clip_percentile, int8_t* qw,
                                               float* sw, void* stream) {
  if (!valid_percentile(clip_percentile)) return CIDER_ERR_INVALID_ARGUMENT;
  return guarded(
      [&] { return quantize_weight(w, N, K, group_size, qw, sw, false, stream, clip_percentile); });
}

cider_status_t cider_quantize_weight_int4_clip(const float* w, int64_t N, int64_t K,
                                               int group_size, double clip_percentile,
                                               uint8_t* qw_packed, float* sw, void* stream) {
  if (!valid_percentile(clip_percentile)) return CIDER_ERR_INVALID_ARGUMENT;
  return guarded([&] {
    return quantize_weight(w, N, K, group_size, qw_packed, sw, true, stream, clip_percentile);
  });
}

static cider_status_t linear_entry(const void* x, const int8_t* qa, const float* sa, int64_t M,
                                   int64_t N, int64_t K, const void* w, bool int4, const float* sw,
                                   int granularity, int group_size, void* y, void* stream,
                                   bool x_bf16 = false, bool y_bf16 = false) {
  return guarded([&] {
    cider::LinearArgs a;
    a.x = x;
    a.x_bf16 = x_bf16;
    a.qa = qa;
    a.sa = sa;
    a.M = M;
    a.N = N;
    a.K = K;
    a.w = w;
    a.int4 = int4;
    a.sw = sw;
    a.granularity = granularity;
    a.group_size = group_size;
    a.y = y;
    a.mode = y_bf16 ? cider::kEpiYb : cider::kEpiY;
    a.st = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0) return CIDER_OK;
    if (!x && !qa) return CIDER_ERR_INVALID_ARGUMENT;
    cider::ScratchSource scratch = cider::ScratchSource::pooled(a.st);
    return cider::run_linear(a, scratch);
  });
}

cider_status_t cider_w8a8_linear(const void* x, int64_t M, int64_t N, int64_t K, const int8_t* qw,
                                 const float* sw, int granularity, int group_size, void* y,
                                 void* stream) {
  if (x == nullptr && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(x, nullptr, nullptr, M, N, K, qw, false, sw, granularity, group_size, y, stream);
}

cider_status_t cider_w4a8_linear(const void* x, int64_t M, int64_t N, int64_t K,
                                 const uint8_t* qw_packed, const float* sw, int granularity,
                                 int group_size, void* y, void* stream) {
  if (x == nullptr && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(x, nullptr, nullptr, M, N, K, qw_packed, true, sw, granularity, group_size, y,
                      stream);
}

cider_status_t cider_w8a8_linear_bf16(const void* x, int64_t M, int64_t N, int64_t K,
                                      const int8_t* qw, const float* sw, int granularity,
                                      int group_size, void* y, void* stream) {
  if (x == nullptr && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(x, nullptr, nullptr, M, N, K, qw, false, sw, granularity, group_size, y,
                      stream, true);
}

cider_status_t cider_w4a8_linear_bf16(const void* x, int64_t M, int64_t N, int64_t K,
                                      const uint8_t* qw_packed, const float* sw, int granularity,
                                      int group_size, void* y, void* stream) {
  if (x == nullptr && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(x, nullptr, nullptr, M, N, K, qw_packed, true, sw, granularity, group_size, y,
                      stream, true);
}

cider_status_t cider_w8a8_linear_ex(const void* x, int x_dtype, int64_t M, int64_t N, int64_t K,
                                    const int8_t* qw, const float* sw, int granularity,
                                    int group_size, void* y, int y_dtype, void* stream) {
  if (x == nullptr && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  if ((x_dtype != CIDER_F16 && x_dtype != CIDER_BF16) || (y_dtype != CIDER_F16 && y_dtype != CIDER_BF16))
    return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(x, nullptr, nullptr, M, N, K, qw, false, sw, granularity, group_size, y,
                      stream, x_dtype == CIDER_BF16, y_dtype == CIDER_BF16);
}

cider_status_t cider_w4a8_linear_ex(const void* x, int x_dtype, int64_t M, int64_t N, int64_t K,
                                    const uint8_t* qw_packed, const float* sw, int granularity,
                                    int group_size, void* y, int y_dtype, void* stream) {
  if (x == nullptr && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  if ((x_dtype != CIDER_F16 && x_dtype != CIDER_BF16) || (y_dtype != CIDER_F16 && y_dtype != CIDER_BF16))
    return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(x, nullptr, nullptr, M, N, K, qw_packed, true, sw, granularity, group_size,
                      y, stream, x_dtype == CIDER_BF16, y_dtype == CIDER_BF16);
}

cider_status_t cider_w8a8_linear_prequant(const int8_t* qa, const float* sa, int64_t M, int64_t N,
                                          int64_t K, const int8_t* qw, const float* sw,
                                          int granularity, int group_size, void* y, void* stream) {
  if ((qa == nullptr || sa == nullptr) && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(nullptr, qa, sa, M, N, K, qw, false, sw, granularity, group_size, y, stream);
}

cider_status_t cider_w4a8_linear_prequant(const int8_t* qa, const float* sa, int64_t M, int64_t N,
                                          int64_t K, const uint8_t* qw_packed, const float* sw,
                                          int granularity, int group_size, void* y, void* stream) {
  if ((qa == nullptr || sa == nullptr) && M != 0 && N != 0) return CIDER_ERR_INVALID_ARGUMENT;
  return linear_entry(nullptr, qa, sa, M, N, K, qw_packed, true, sw, granularity, group_size, y,
                      stream);
}

static cider_status_t acc_entry(const int8_t* qa, int64_t M, int64_t N, int64_t K, const void* w,
                                bool int4, int group_size, int32_t* acc, void* stream) {
  return guarded([&] {
    if (M != 0 && N != 0 && !qa) return CIDER_ERR_INVALID_ARGUMENT;
    cider::LinearArgs a;
    a.qa = qa;
    a.M = M;
    a.N = N;
    a.K = K;
    a.w = w;
    a.int4 = int4;
    a.group_size = group_size;
    a.acc = acc;
    a.mode = cider::kEpiAcc;
    a.st = static_cast<cudaStream_t>(stream);
    cider::ScratchSource scratch = cider::ScratchSource::pooled(a.st);
    return cider::run_linear(a, scratch);
  });
}

cider_status_t cider_w8a8_accumulators(const int8_t* qa, int64_t M, int64_t N, int64_t K,
                                       const int8_t* qw, int group_size, int32_t* acc,
                                       void* stream) {
  return acc_entry(qa, M, N, K, qw, false, group_size, acc, stream);
}

cider_status_t cider_w4a8_accumulators(const int8_t* qa, int64_t M, int64_t N, int64_t K,
                                       const uint8_t* qw_packed, int group_size, int32_t* acc,
                                       void* stream) {
  return acc_entry(qa, M, N, K, qw_packed, true, group_size, acc, stream);
}

cider_status_t cider_timing_begin(int64_t capacity) {
  return guarded([&]() -> cider_status_t {
    if (capacity < 1) return CIDER_ERR_INVALID_ARGUMENT;
    timer_release();
    t_timer.ev.resize(static_cast<size_t>(2 * capacity), nullptr);
    for (auto& e : t_timer.ev) {
      if (cudaEventCreate(&e) != cudaSuccess) {
        e = nullptr;
        timer_release();
        return cuda_status(cudaErrorUnknown);
      }
    }
    t_timer.on = true;
    return CIDER_OK;
  });
}

cider_status_t cider_timing_end(int64_t* count, double* total_ms) {
  return guarded([&]() -> cider_status_t {
    if (!count || !total_ms) return CIDER_ERR_INVALID_ARGUMENT;
    double sum = 0.0;
    cider_status_t st = CIDER_OK;
    for (int64_t i = 0; i < t_timer.used; ++i) {
      float ms = 0.0f;
      if (cudaEventSynchronize(t_timer.ev[2 * i + 1]) != cudaSuccess ||
          cudaEventElapsedTime(&ms, t_timer.ev[2 * i], t_timer.ev[2 * i + 1]) != cudaSuccess) {
        st = cuda_status(cudaErrorUnknown);
        break;
      }
      sum += ms;
    }
    *count = t_timer.used;
    *total_ms = sum;
    timer_release();
    return st;
  });
}

cider_status_t cider_trim_scratch_pool(int64_t keep_bytes, void* stream) {
  return guarded([&] {
    if (keep_bytes < 0) return CIDER_ERR_INVALID_ARGUMENT;
    int dev = 0;
    cider_status_t s = cider::check_device(&dev, nullptr);
    if (s != CIDER_OK) return s;
    cudaMemPool_t pool = nullptr;
    {
      std::lock_guard<std::mutex> lk(g_pool_mu);
      pool = g_pool[dev];
    }
    if (pool == nullptr) return CIDER_OK;   // nothing allocated on this device yet
    // blocks freed by calls still queued on `stream` return to the pool only
    // when those calls have run
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return cuda_status(cudaErrorUnknown);
    return cuda_status(cudaMemPoolTrimTo(pool, static_cast<size_t>(keep_bytes)));
  });
}

cider_status_t cider_check_device_error(void* stream) {
  return guarded([&] {
    cider_status_t s = cider::check_device(nullptr, nullptr);
    if (s != CIDER_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return cuda_status(cudaErrorUnknown);
    int v = 0;
    if (cider::read_and_clear_device_error(&v) != cudaSuccess) return cuda_status(cudaErrorUnknown);
    return v ? CIDER_ERR_TIMEOUT : CIDER_OK;
  });
}

cider_status_t cider_debug_wait_timeout(int64_t max_polls, void* stream) {
  return guarded([&] {
    if (max_polls < 1) return CIDER_ERR_INVALID_ARGUMENT;
    cider_status_t s = cider::check_device(nullptr, nullptr);
    if (s != CIDER_OK) return s;
    return cuda_status(cider::launch_debug_wait_timeout(max_polls, static_cast<cudaStream_t>(stream)));
  });
}

cider_status_t cider_debug_small_m_slices(int64_t M, int64_t N, int64_t K, int int4,
                                          int group_size, int num_sms, int32_t* slices) {
  return guarded([&] {
    if (M < 1 || M > 16 || N < 1 || K < 1 || num_sms < 1 || slices == nullptr)
      return CIDER_ERR_INVALID_ARGUMENT;
    *slices = cider::gemv_slices(M, N, K, int4 != 0, group_size, cider::kEpiY, num_sms);
    return CIDER_OK;
  });
}

cider_status_t cider_debug_small_m_launch(int64_t M, int64_t N, int64_t K, int int4,
                                          int group_size, int split_allowed, int num_sms,
                                          int32_t* info) {
  return guarded([&] {
    if (M < 1 || N < 1 || K < 1 || num_sms < 1 || info == nullptr || !cider::gemv_fits(M, K))
      return CIDER_ERR_INVALID_ARGUMENT;
    cider::gemv_launch_info(M, N, K, int4 != 0, group_size, split_allowed != 0, num_sms, info);
    return CIDER_OK;
  });
}

cider_status_t cider_debug_pair_schedule(int64_t M, int64_t N, int64_t K, int pairs,
                                         int64_t capacity, int32_t* units, int64_t* count,
                                         int32_t* info) {
  return guarded([&] {
    if (M < 1 || N < 1 || K < 1 || pairs < 1 || capacity < 0 || count == nullptr ||
        info == nullptr || (capacity > 0 && units == nullptr))
      return CIDER_ERR_INVALID_ARGUMENT;
    cider::pair_schedule(M, N, K, pairs, capacity, units, count, info);
    return CIDER_OK;
  });
}

}  // extern "C"
