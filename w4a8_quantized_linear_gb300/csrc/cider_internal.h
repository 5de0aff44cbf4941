// cider_internal.h -- launchers shared between the translation units of the
// library (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>

#include <atomic>

#include "cider.h"

namespace cider {

// 2D TMA tensor map over a row-major matrix: `inner` elements per row,
// `outer` rows, `row_bytes` between rows; box of box_inner x box_outer.
// Out-of-bounds elements of a box read as zero.  Returns false on failure.
bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle swz);

// Raise a kernel's dynamic shared memory limit once per device (bit d of
// `done` records device d).
inline cudaError_t ensure_max_dynamic_smem(const void* kern, int bytes,
                                           std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Epilogue kinds of the integer GEMM / GEMV main loops.
enum EpiMode : int {
  kEpiY = 0,    // dequantize and store fp16 y [M, N]
  kEpiAcc = 1,  // store the exact int32 accumulators [M, N, G]
  kEpiYb = 2,   // dequantize and store bf16 y [M, N]
};

// quant.cu.  release: the library's own GEMM or GEMV is launched next on the
// stream as a programmatic dependent, and may start as soon as every CTA of
// the quantization is running (false: later work waits for its completion).
cudaError_t launch_quant_act_s8(const __half* x, int64_t M, int64_t K, int8_t* q, float* sa,
                                cudaStream_t st, bool release = false);
// fp16 codes for the tensor-core path, plus row_l1[m] = sum_k |q[m,k]|; also
// clears `zero_words` int32 words at `zero` (the GEMM's flags) on the way.
cudaError_t launch_quant_act_f16(const __half* x, int64_t M, int64_t K, __half* q, float* sa,
                                 int* row_l1, int* zero, int zero_words, cudaStream_t st,
                                 bool release = false);
// The same two from bf16 activations.
cudaError_t launch_quant_act_s8_bf16(const __nv_bfloat16* x, int64_t M, int64_t K, int8_t* q,
                                     float* sa, cudaStream_t st, bool release = false);
cudaError_t launch_quant_act_f16_from_bf16(const __nv_bfloat16* x, int64_t M, int64_t K, __half* q,
                                           float* sa, int* row_l1, int* zero, int zero_words,
                                           cudaStream_t st, bool release = false);
cudaError_t launch_quant_weight(const float* w, int64_t N, int64_t K, int group_size, bool int4,
                                uint8_t* q, float* sw, cudaStream_t st);
// The same with percentile-clipped scales (clip_percentile in (0, 100]).
cudaError_t launch_quant_weight_clip(const float* w, int64_t N, int64_t K, int group_size,
                                     double clip_percentile, bool int4, uint8_t* q, float* sw,
                                     cudaStream_t st);
// Offset-binary INT4 bytes -> two's complement INT4 bytes (src may equal dst).
cudaError_t launch_int4_from_offset(const uint8_t* src, uint8_t* dst, int64_t nbytes,
                                    cudaStream_t st);
cudaError_t launch_codes_s8_to_f16(const int8_t* qa, int64_t M, int64_t K, __half* out,
                                   int* row_l1, int* zero, int zero_words, cudaStream_t st);

// gemv.cu: small-M weight-streaming path (M <= 16).  Activations either as
// fp16 x [M, K] (quantized inside the kernel; x != nullptr) or as codes
// qa int8 [M, K] with scales sa [M].  group_size 0 = per channel.  Exactly
// one of y / acc is used (by mode).
bool gemv_fits(int64_t M, int64_t K);
// Whether the linear entry points let the GEMV quantize the activation rows
// itself (every CTA repeats that work) rather than run a quantization kernel
// first: for one token, or while the rows are short (measured on GB300).
inline bool gemv_quantizes_itself(int64_t M, int64_t K) { return M == 1 || M * K <= 8192; }
// K split of the small-M path (few weight-row blocks, long rows): the bytes of
// partial sums it needs for this problem (0: no split); the split needs
// pre-quantized rows (qa, sa) and y output.
size_t gemv_part_bytes(int64_t M, int64_t N, int64_t K, bool int4, int group_size, int mode,
                       int num_sms);
// The number of K slices it uses (1: none).  Host arithmetic only.
int gemv_slices(int64_t M, int64_t N, int64_t K, bool int4, int group_size, int mode,
                int num_sms);
// Sizes of the GEMV launch for y output (host arithmetic only): info[0..9] =
// {padded token count, tensor-core form, K slices, weight tiles per slice,
// staged codes per token row, their row pitch in bytes, ring slots, dynamic
// shared memory bytes, the launch's cap on it, codes per weight tile row}.
// split_allowed: the rows come pre-quantized and scratch for partials exists.
void gemv_launch_info(int64_t M, int64_t N, int64_t K, bool int4, int group_size, bool split_allowed,
                      int num_sms, int32_t* info);
// after_quant: the launch just before on `st` is this library's activation
// quantization, which the GEMV may overlap (programmatic dependent launch).
cudaError_t launch_gemv(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                        int64_t K, const uint8_t* w, bool int4, const float* sw, int group_size,
                        int mode, __half* y, int32_t* acc, void* part, int num_sms, cudaStream_t st,
                        bool after_quant);

// gemm_tc.cu: tensor-core path.  qa16 holds the activation codes as fp16
// integers [M, K]; row_l1[m] = sum_k |code| (used by the per-channel kernel
// to decide per tile whether one fp32 accumulation over all of K is exact).
// Per channel (group_size 0) it runs the CTA-pair kernel of gemm_pair.cu,
// which shares the blocks of the last partial round of tiles among all CTA
// pairs when `workspace` (gemm_tc_scratch(...).bytes, or null to deal every
// tile whole) allows it.
struct GemmScratch {
  size_t bytes = 0;        // workspace size (0: none wanted)
  size_t zero_offset = 0;  // byte offset of int32 words that must be zero at launch
  int zero_words = 0;
};
GemmScratch gemm_tc_scratch(int64_t M, int64_t N, int64_t K, int group_size);
cudaError_t launch_gemm_tc(const __half* qa16, const float* sa, const int* row_l1, int64_t M,
                           int64_t N, int64_t K, const uint8_t* w, bool int4, const float* sw,
                           int group_size, int mode, __half* y, int32_t* acc, void* workspace,
                           int num_sms, cudaStream_t st, bool after_quant);
// gemm_pg.cu: per-group tensor-core path on CTA pairs (see launch_gemm_tc).
cudaError_t launch_gemm_pg(const __half* qa16, const float* sa, int64_t M, int64_t N, int64_t K,
                           const uint8_t* w, bool int4, const float* sw, int group_size, int mode,
                           __half* y, int32_t* acc, cudaStream_t st, bool after_quant);
// gemm_pair.cu: per-channel tensor-core path on CTA pairs (see launch_gemm_tc).
GemmScratch gemm_pair_scratch(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_pair(const __half* qa16, const float* sa, const int* row_l1, int64_t M,
                             int64_t N, int64_t K, const uint8_t* w, bool int4, const float* sw,
                             int mode, __half* y, int32_t* acc, void* workspace, cudaStream_t st,
                             bool after_quant);
// Host copy of the pair GEMM's work split (see cider_debug_pair_schedule).
void pair_schedule(int64_t M, int64_t N, int64_t K, int pairs, int64_t capacity, int32_t* units,
                   int64_t* count, int32_t* info);
cudaError_t read_and_clear_device_error(int* value);
// Device address of the library's error word on the current device.
cudaError_t device_error_word(int** ptr);
constexpr uint64_t kKernelWaitTimeoutNs = 2000000000ull;
cudaError_t launch_debug_wait_timeout(int64_t max_polls, cudaStream_t st);

// ---------------------------------------------------------------- cider_api.cu
// One linear / accumulator call, as the C entry points receive it.
struct LinearArgs {
  const void* x = nullptr;  // fp16 / bf16 activations (or null for the prequant forms)
  bool x_bf16 = false;
  const int8_t* qa = nullptr;
  const float* sa = nullptr;
  int64_t M = 0, N = 0, K = 0;
  const void* w = nullptr;
  bool int4 = false;
  const float* sw = nullptr;
  int granularity = 0, group_size = 0;
  void* y = nullptr;
  int32_t* acc = nullptr;
  int mode = kEpiY;
  cudaStream_t st = nullptr;
};

// Host argument checks shared by every linear entry point (the order the
// public header documents): sizes, pointers, K and N rules, grouping, alignment.
cider_status_t validate_linear(const LinearArgs& a);
// Current device is a supported sm_103 GPU (cached per device; honours
// CIDER_FORCE_UNSUPPORTED=1); writes its index and SM count.
cider_status_t check_device(int* dev_out, int* num_sms);

// Where a call's scratch memory comes from: the library's per-device
// stream-ordered pool (allocated and freed on the call's stream), or a fixed
// caller-provided region [base, base + capacity) that is carved up without
// any allocation.
class ScratchSource {
 public:
  static ScratchSource pooled(cudaStream_t st) { return ScratchSource(st, nullptr, 0); }
  static ScratchSource fixed(void* base, size_t capacity) {
    return ScratchSource(nullptr, base, capacity);
  }
  ScratchSource(ScratchSource&& o) noexcept;
  ScratchSource(const ScratchSource&) = delete;
  ScratchSource& operator=(const ScratchSource&) = delete;
  ~ScratchSource();
  // Whether `bytes` can be had (always, for the pool).
  bool fits(size_t bytes) const { return base_ == nullptr || bytes <= capacity_; }
  // `bytes` of scratch for this call (at most one request per call): a pool
  // allocation error maps to CIDER_ERR_CUDA, a fixed region too small to
  // CIDER_ERR_INVALID_ARGUMENT.
  cider_status_t get(size_t bytes, void** out);

 private:
  ScratchSource(cudaStream_t st, void* base, size_t cap) : st_(st), base_(base), capacity_(cap) {}
  cudaStream_t st_;
  void* base_;
  size_t capacity_;
  void* pool_ptr_ = nullptr;
};

// Scratch bytes a linear call cannot do without (activation codes and
// per-token values; the K-piece and K-slice workspaces are optional and left
// out when a fixed region has no room for them).
size_t linear_required_scratch(const LinearArgs& a);
// The M-bucket dispatch of every linear entry point: argument and device
// checks, then the small-M GEMV (M <= 16) or quantization + tensor-core GEMM.
cider_status_t run_linear(const LinearArgs& a, ScratchSource& scratch);

}  // namespace cider
