// gemm_tc.cu -- the tensor-core path's host dispatch (per channel: the
// CTA-pair kernel of gemm_pair.cu; per group: the CTA-pair kernel of
// gemm_pg.cu), the TMA tensor-map helper they share, and the library's
// device error word with its bounded-wait test kernel (Cider README, page
// "cider": "Architecture / Metal kernel pipeline", matmul_fused_dequant).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {

__device__ int g_device_error = 0;

namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

__global__ void debug_wait_kernel(int64_t max_polls) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, &g_device_error, kWaitTimeoutNs,
                      static_cast<uint64_t>(max_polls));
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle swz) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tc(const __half* qa16, const float* sa, const int* row_l1, int64_t M,
                           int64_t N, int64_t K, const uint8_t* w, bool int4, const float* sw,
                           int group_size, int mode, __half* y, int32_t* acc, void* workspace,
                           int num_sms, cudaStream_t st, bool after_quant) {
  (void)num_sms;
  if (group_size == 0)
    return launch_gemm_pair(qa16, sa, row_l1, M, N, K, w, int4, sw, mode, y, acc, workspace, st,
                            after_quant);
  return launch_gemm_pg(qa16, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, st, after_quant);
}

GemmScratch gemm_tc_scratch(int64_t M, int64_t N, int64_t K, int group_size) {
  return group_size == 0 ? gemm_pair_scratch(M, N, K) : GemmScratch{};
}

cudaError_t device_error_word(int** ptr) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_device_error);
  *ptr = static_cast<int*>(p);
  return e;
}

cudaError_t read_and_clear_device_error(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

cudaError_t launch_debug_wait_timeout(int64_t max_polls, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(max_polls);
  return cudaGetLastError();
}

}  // namespace cider
