// gemm_tc.cu -- tensor-core integer GEMM with fused per-group dequant for
// M > 16 (Cider README, page "cider": "Architecture / Metal kernel pipeline",
// matmul_fused_dequant: INT8 x INT8 -> INT32 -> FP16 with the scales applied
// in the store; per-group scales from "W8A8 quantization granularity"; W4A8
// unpacks INT4 ahead of the multiply, "Architecture" and "Limitations").
// Per-channel problems go to the CTA-pair kernel in gemm_pair.cu; this file
// also holds the library's device error word, the TMA descriptor helper and
// the dispatch between the two.
//
// sm_103a has no integer tcgen05 MMA kind, so the exact integer product runs
// on the fp16 tensor pipe (tcgen05.mma kind::f16, fp32 accumulation in
// tensor memory): every code in [-127, 127] is an exact fp16 value, every
// product an exact integer below 2^14, and the accumulator is drained after
// every group of 64 / 128 K-elements, so each partial sum stays below 2^21
// and is exact in fp32.
//
// Roles (one CTA per SM, persistent over 128 x 128 output tiles):
//   warp 0      TMA producer: weight tile (int8 [128 n][64 k], 64-byte
//               swizzle; INT4: packed [128 n][32 B], 32-byte swizzle) and
//               activation-code tile (fp16 [128 m][64 k], 128-byte swizzle)
//               into an 8-stage shared-memory ring.
//   warps 2-5   converters: each thread owns one weight row, reads its 64
//               codes of the stage from shared memory, converts them to fp16
//               in registers (INT4: nibble unpack) and stores them into its
//               tensor-memory lane: this is the MMA's A operand.
//   warp 1      MMA issuer (one thread): D[128 n x 128 m] += A[tmem] * B[smem]^T,
//               K = 16 per instruction, into one of two accumulators.
//   warps 6-13  epilogue: drain the accumulator after every group, keep the
//               fp32 per-group sums (or exact int32 accumulators) in
//               registers, dequantize and store fp16 y (or raw int32).
// Tensor memory (512 columns): accumulators at columns [0,128) and [128,256),
// the 8 A-operand slots of 32 columns each at [256, 512).
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

constexpr int kTileN = 128;  // weight rows per tile: MMA M, tensor-memory lanes
constexpr int kTileM = 128;  // tokens per tile: MMA N
constexpr int kBK = 64;      // K per pipeline stage
constexpr int kStages = 8;
constexpr int kUmmaK = 16;
constexpr int kAccCols = kTileM;
constexpr int kASlotCols = kBK / 2;  // fp16 pairs per 32-bit column
constexpr int kACol0 = 2 * kAccCols;
constexpr int kTmemCols = 512;
constexpr int kPcChunkKB = 8;  // per-channel drain interval: 8 stages = 512 K
constexpr int kThreads = 448;
constexpr int kEpiWarp0 = 6;
constexpr int kBStageBytes = kTileM * kBK * 2;  // 16 KiB
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

static_assert(kACol0 + kStages * kASlotCols <= kTmemCols, "tensor memory budget");

template <bool INT4>
struct Cfg {
  static constexpr int kAStageBytes = INT4 ? kTileN * kBK / 2 : kTileN * kBK;
  static constexpr int kStageBytes = kBStageBytes + kAStageBytes;
  static constexpr int kBarOffset = kStages * kStageBytes;
  // full, empty, conv per stage; acc_full, acc_empty x2; tmem slot; abort
  static constexpr int kSmemBytes = kBarOffset + (3 * kStages + 4) * 8 + 16 + 1024;
};

struct GemmArgs {
  int M, N, K;
  int gs;  // 0 = per channel
  int G;
  int num_m_tiles, num_tiles;
  const float* sa;
  const float* sw;
  __half* y;
  int32_t* acc;
};

template <bool INT4, bool PG, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs p) {
  using C = Cfg<INT4>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sB = [&](int s) { return base + s * C::kStageBytes; };
  auto sA = [&](int s) { return base + s * C::kStageBytes + kBStageBytes; };
  const uint32_t bars = base + C::kBarOffset;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto conv_bar = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (3 * kStages + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (3 * kStages + 2 + b); };
  const uint32_t tmem_slot = bars + 8u * (3 * kStages + 4);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * (3 * kStages + 4) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(conv_bar(s), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 8);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset +
                                                              8 * (3 * kStages + 4));

  const int nkb = (p.K + kBK - 1) / kBK;
  const int kbpc = PG ? p.gs / kBK : kPcChunkKB;  // stages per drained chunk
  const int nchunks = (nkb + kbpc - 1) / kbpc;
  int* err = &g_device_error;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
        const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kWaitTimeoutNs)) goto done;
          mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
          tma_load_2d(sB(s), &tmB, full_bar(s), kb * kBK, mt * kTileM);
          tma_load_2d(sA(s), &tmA, full_bar(s), INT4 ? kb * (kBK / 2) : kb * kBK, nt * kTileN);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kTileN, kTileM);
      int it = 0, ch = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const bool cstart = (kb % kbpc) == 0;
          const int b = ch & 1;
          if (cstart) {
            if (!mbar_wait_bounded(acce_bar(b), ((ch >> 1) & 1) ^ 1u, abort_flag, err,
                                   kWaitTimeoutNs))
              goto done;
            tc_fence_after();
          }
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait_bounded(full_bar(s), ph, abort_flag, err, kWaitTimeoutNs)) goto done;
          if (!mbar_wait_bounded(conv_bar(s), ph, abort_flag, err, kWaitTimeoutNs)) goto done;
          tc_fence_after();
          const uint32_t d_tmem = tmem + b * kAccCols;
          const uint32_t a_tmem = tmem + kACol0 + s * kASlotCols;
          const uint64_t bdesc = smem_desc_k_sw128(sB(s));
#pragma unroll
          for (int j = 0; j < kBK / kUmmaK; ++j)
            tc_mma_ts(d_tmem, a_tmem + j * (kUmmaK / 2), bdesc + static_cast<uint64_t>(j * 2),
                      idesc, (cstart && j == 0) ? 0u : 1u);
          tc_commit(empty_bar(s));
          if ((kb % kbpc) == kbpc - 1 || kb == nkb - 1) {
            tc_commit(accf_bar(b));
            ++ch;
          }
        }
      }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;                // tensor-memory lane quadrant
    const int row = q * 32 + lane;         // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(s), ph, abort_flag, err,
                                                       kWaitTimeoutNs)))
          goto done;
        tc_fence_after();
        uint32_t h[32];
        const uint8_t* arow = gbase + (sA(s) - base);
        if (!INT4) {
          // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                arow + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
            s8x4_to_h2x2(v.x, h[8 * c + 0], h[8 * c + 1]);
            s8x4_to_h2x2(v.y, h[8 * c + 2], h[8 * c + 3]);
            s8x4_to_h2x2(v.z, h[8 * c + 4], h[8 * c + 5]);
            s8x4_to_h2x2(v.w, h[8 * c + 6], h[8 * c + 7]);
          }
        } else {
          // 32-byte swizzle: chunk c of row r sits at chunk c ^ ((r >> 2) & 1)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                arow + row * 32 + ((c ^ ((row >> 2) & 1)) << 4));
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t t[4];
              s4x8_to_h2x4(vw[j], t);
              h[16 * c + 4 * j + 0] = t[0];
              h[16 * c + 4 * j + 1] = t[1];
              h[16 * c + 4 * j + 2] = t[2];
              h[16 * c + 4 * j + 3] = t[3];
            }
          }
        }
        tmem_st32(tmem + lane_base + kACol0 + s * kASlotCols, h);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(conv_bar(s));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;   // 0..7
    const int q = warp & 3;           // lane quadrant
    const int colh = e >> 2;          // which 64 accumulator columns
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int ch = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int n = nt * kTileN + row;
      const bool nvalid = n < p.N;
      const int m0 = mt * kTileM + colh * 64;
      int isum[64];
      float fsum[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        isum[j] = 0;
        fsum[j] = 0.0f;
      }
      // per group: the weight scale of the next group is loaded while this
      // group's accumulator is still being filled (a cache round trip after
      // the wait would sit on every group's critical path)
      const bool load_sw = PG && EPI == kEpiY && nvalid;
      const float* swrow = p.sw + static_cast<int64_t>(n) * p.G;
      float sw_next = load_sw ? __ldg(swrow) : 0.0f;
      for (int c = 0; c < nchunks; ++c, ++ch) {
        const int b = ch & 1;
        const float swg = sw_next;
        if (load_sw && c + 1 < nchunks) sw_next = __ldg(swrow + c + 1);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                       err, kWaitTimeoutNs)))
          goto done;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + b * kAccCols + colh * 64 + hh * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float f = __uint_as_float(v[j]);
            if (!PG) {
              isum[hh * 32 + j] += __float2int_rn(f);
            } else if (EPI == kEpiY) {
              fsum[hh * 32 + j] = fmaf(swg, f, fsum[hh * 32 + j]);
            } else {
              const int m = m0 + hh * 32 + j;
              if (nvalid && m < p.M)
                p.acc[(static_cast<int64_t>(m) * p.N + n) * p.G + c] = __float2int_rn(f);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(b));
      }
      if (PG && EPI == kEpiAcc) continue;
      // the 64 token scales of this warp's columns: two per lane, handed out
      // by shuffles (the whole warp takes part, also lanes past N)
      float sa_lo = 0.0f, sa_hi = 0.0f;
      if (EPI == kEpiY) {
        if (m0 + lane < p.M) sa_lo = __ldg(p.sa + m0 + lane);
        if (m0 + 32 + lane < p.M) sa_hi = __ldg(p.sa + m0 + 32 + lane);
      }
      const float swn = (!PG && EPI == kEpiY && nvalid) ? __ldg(p.sw + n) : 0.0f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int m = m0 + j;
        const float sam = EPI == kEpiY ? __shfl_sync(0xffffffffu, j < 32 ? sa_lo : sa_hi, j & 31) : 0.0f;
        if (nvalid && m < p.M) {
          const int64_t off = static_cast<int64_t>(m) * p.N + n;
          if (EPI == kEpiAcc) {
            p.acc[off] = isum[j];
          } else if (!PG) {
            const float v = __fmul_rn(__fmul_rn(__int2float_rn(isum[j]), sam), swn);
            p.y[off] = __float2half_rn(v);
          } else {
            p.y[off] = __float2half_rn(__fmul_rn(fsum[j], sam));
          }
        }
      }
    }
  }
done:
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


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

namespace {

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swz) {
  return make_tensor_map_2d(map, dt, ptr, inner, outer, row_bytes, box_inner, box_outer, swz);
}

template <bool INT4, bool PG, int EPI>
cudaError_t launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                      int num_sms, cudaStream_t st) {
  auto kern = gemm_tc_kernel<INT4, PG, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                          Cfg<INT4>::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = a.num_tiles < num_sms ? a.num_tiles : num_sms;
  kern<<<grid, kThreads, Cfg<INT4>::kSmemBytes, st>>>(tmA, tmB, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(const __half* qa16, const float* sa, const int* row_l1, int64_t M,
                           int64_t N, int64_t K, const uint8_t* w, bool int4, const float* sw,
                           int group_size, int mode, __half* y, int32_t* acc, void* workspace,
                           int num_sms, cudaStream_t st) {
  if (group_size == 0)
    return launch_gemm_pair(qa16, sa, row_l1, M, N, K, w, int4, sw, mode, y, acc, workspace, st);
  // 128-element groups: the CTA-pair kernel of gemm_pg.cu; 64-element groups
  // (twice the drains per K) run faster on this file's single-CTA kernel
  if (group_size == 128)
    return launch_gemm_pg(qa16, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, st);
  CUtensorMap tmA, tmB;
  if (!make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qa16, K, M, K * 2, kBK, kTileM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t wbytes = int4 ? K / 2 : K;
  if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, N, wbytes,
                   int4 ? kBK / 2 : kBK, kTileN,
                   int4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  GemmArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.gs = group_size;
  a.G = static_cast<int>(K / group_size);
  a.num_m_tiles = static_cast<int>((M + kTileM - 1) / kTileM);
  a.num_tiles = a.num_m_tiles * static_cast<int>((N + kTileN - 1) / kTileN);
  a.sa = sa;
  a.sw = sw;
  a.y = y;
  a.acc = acc;
  if (int4)
    return mode == kEpiY ? launch_tc<true, true, kEpiY>(tmA, tmB, a, num_sms, st)
                         : launch_tc<true, true, kEpiAcc>(tmA, tmB, a, num_sms, st);
  return mode == kEpiY ? launch_tc<false, true, kEpiY>(tmA, tmB, a, num_sms, st)
                       : launch_tc<false, true, kEpiAcc>(tmA, tmB, a, num_sms, st);
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
