// gemm_tc.cu -- tensor-core integer GEMM with fused dequant for M > 16
// (Cider README, page "cider": "Architecture / Metal kernel pipeline",
// matmul_fused_dequant: INT8 x INT8 -> INT32 -> FP16 with the scales applied
// in the store; per-group scales from "W8A8 quantization granularity"; W4A8
// unpacks INT4 ahead of the multiply, "Architecture" and "Limitations").
//
// sm_103a has no integer tcgen05 MMA kind, so the exact integer product runs
// on the fp16 tensor pipe (tcgen05.mma kind::f16, fp32 accumulation in
// tensor memory): every code in [-127, 127] is an exact fp16 value, every
// product an exact integer below 2^14, and the accumulator is drained after
// at most 512 K-elements (per group: after every group of 64 / 128), so each
// partial sum stays below 2^23 and is exact in fp32.  Drained chunks are
// summed in int32 registers, which makes the per-channel accumulator exact
// for any K (|acc| <= 16129 K < 2^31 for K < 133144).
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
//   warps 6-13  epilogue: drain the accumulator per chunk / group, keep the
//               exact int32 (per channel) or fp32 per-group sums in
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
      for (int c = 0; c < nchunks; ++c, ++ch) {
        const int b = ch & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                       err, kWaitTimeoutNs)))
          goto done;
        tc_fence_after();
        const float swg = (PG && EPI == kEpiY && nvalid) ? __ldg(p.sw + static_cast<int64_t>(n) * p.G + c) : 0.0f;
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
      if (!nvalid || (PG && EPI == kEpiAcc)) continue;
      const float swn = (!PG && EPI == kEpiY) ? __ldg(p.sw + n) : 0.0f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int m = m0 + j;
        if (m < p.M) {
          const int64_t off = static_cast<int64_t>(m) * p.N + n;
          if (EPI == kEpiAcc) {
            p.acc[off] = isum[j];
          } else if (!PG) {
            const float v = __fmul_rn(__fmul_rn(__int2float_rn(isum[j]), __ldg(p.sa + m)), swn);
            p.y[off] = __float2half_rn(v);
          } else {
            p.y[off] = __float2half_rn(__fmul_rn(fsum[j], __ldg(p.sa + m)));
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


// ============================================================================
// Per-channel kernel, wide tiles: 128 weight rows x 256 tokens.
//
// Each 64-wide K stage feeds four 128x256x16 MMAs (512 tensor-pipe cycles), and
// the MMA thread synchronizes with the converter warps once per stage pair, so
// the fixed cost of a barrier handshake (a few hundred cycles per wait) stays
// below the tensor work it guards.  One 256-column fp32 accumulator.
//
// Exactness per tile: every partial sum of a row m is bounded by
// qmax_w * sum_k |q_a[m,k]| (qmax_w = 127 for INT8, 8 for INT4).  When that
// bound is <= 2^23 for all 256 rows of the tile ("fast" tile, the normal case
// for real activations: sum |q_a| is a few thousand per 1000 K), the whole K
// accumulates in fp32 exactly and the accumulator is drained once.  Otherwise
// ("slow" tile) the tile runs as two 128-token passes whose accumulators
// alternate between the two 128-column halves and are drained every 512 K into
// exact int32 register sums, as in the per-group kernel.
// ============================================================================
constexpr int kWTileM = 256;
constexpr int kWStages = 5;
constexpr int kWBStageBytes = kWTileM * kBK * 2;  // 32 KiB
constexpr int kWChunkKB = 8;                       // slow tiles: drain every 512 K
constexpr int64_t kLongK = 4096;                   // K above which the TS kernel is used

static_assert(kACol0 + kWStages * kASlotCols <= kTmemCols, "tensor memory budget (wide)");

template <bool INT4>
struct WCfg {
  static constexpr int kAStageBytes = INT4 ? kTileN * kBK / 2 : kTileN * kBK;
  static constexpr int kStageBytes = kWBStageBytes + kAStageBytes;
  static constexpr int kBarOffset = kWStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOffset + (3 * kWStages + 4) * 8 + 16 + 1024;
};
static_assert(WCfg<false>::kStageBytes % 1024 == 0 && WCfg<true>::kStageBytes % 1024 == 0,
              "stages must keep 1024-byte alignment for the 128-byte swizzle");

struct WideArgs {
  GemmArgs g;
  const int* row_l1;
  int l1_limit;  // a tile is fast when max row_l1 over its rows <= l1_limit
};

// Whole warp: is every row of token tile mt within the exactness bound?
__device__ __forceinline__ bool wide_tile_fast(const WideArgs& a, int mt, int lane) {
  int mx = 0;
#pragma unroll
  for (int i = 0; i < kWTileM / 32; ++i) {
    const int m = mt * kWTileM + i * 32 + lane;
    if (m < a.g.M) mx = max(mx, __ldg(a.row_l1 + m));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  return mx <= a.l1_limit;
}

template <bool INT4, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_wide_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const WideArgs a) {
  using C = WCfg<INT4>;
  const GemmArgs& p = a.g;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sB = [&](int s) { return base + s * C::kStageBytes; };
  auto sA = [&](int s) { return base + s * C::kStageBytes + kWBStageBytes; };
  const uint32_t bars = base + C::kBarOffset;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kWStages + s); };
  auto conv_bar = [&](int s) { return bars + 8u * (2 * kWStages + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (3 * kWStages + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (3 * kWStages + 2 + b); };
  const uint32_t tmem_slot = bars + 8u * (3 * kWStages + 4);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * (3 * kWStages + 4) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
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
                                                              8 * (3 * kWStages + 4));
  const int nkb = (p.K + kBK - 1) / kBK;
  const int nch = (nkb + kWChunkKB - 1) / kWChunkKB;  // chunks per pass of a slow tile
  int* err = &g_device_error;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int passes = wide_tile_fast(a, mt, lane) ? 1 : 2;
      if (lane == 0) {
        for (int pass = 0; pass < passes; ++pass)
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = it % kWStages;
            const uint32_t ph = (it / kWStages) & 1;
            if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kWaitTimeoutNs)) break;
            mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
            tma_load_2d(sB(s), &tmB, full_bar(s), kb * kBK, mt * kWTileM);
            tma_load_2d(sA(s), &tmA, full_bar(s), INT4 ? kb * (kBK / 2) : kb * kBK, nt * kTileN);
          }
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_w = idesc_f16_f32(kTileN, kWTileM);
    constexpr uint32_t idesc_n = idesc_f16_f32(kTileN, kTileM);
    int it = 0, ch = 0;
    int last_use[2] = {-1, -1};  // last chunk written into each accumulator half
    // Wait until chunk c has been drained by the epilogue.
    auto drained = [&](int c) -> bool {
      if (c < 0) return true;
      return mbar_wait_bounded(acce_bar(c & 1), (c >> 1) & 1, abort_flag, err, kWaitTimeoutNs);
    };
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles;
      const bool fast = wide_tile_fast(a, mt, lane);
      if (lane == 0) {
        const int passes = fast ? 1 : 2;
        bool ok = true;
        for (int pass = 0; pass < passes && ok; ++pass) {
          int pending = -1;  // stage whose MMAs wait for the next conv wait
          for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
            const bool cstart = fast ? (kb == 0) : (kb % kWChunkKB) == 0;
            const bool cend = fast ? (kb == nkb - 1) : ((kb % kWChunkKB) == kWChunkKB - 1 || kb == nkb - 1);
            const int b = ch & 1;
            if (cstart) {
              if (fast) {
                ok = drained(last_use[0]) && drained(last_use[1]);
                last_use[0] = last_use[1] = ch;
              } else {
                ok = drained(last_use[b]);
                last_use[b] = ch;
              }
              if (!ok) break;
            }
            const int s = it % kWStages;
            // issue after odd stages and at chunk ends: one conv wait covers the pair
            if ((kb & 1) == 0 && !cend) {
              pending = it;
              continue;
            }
            const uint32_t ph = (it / kWStages) & 1;
            if (!mbar_wait_bounded(conv_bar(s), ph, abort_flag, err, kWaitTimeoutNs)) { ok = false; break; }
            tc_fence_after();
            for (int q = (pending >= 0 ? 0 : 1); q < 2; ++q) {
              const int its = q == 0 ? pending : it;
              const int ss = its % kWStages;
              const int kbs = kb - (q == 0 ? 1 : 0);
              const bool first = fast ? (kbs == 0) : (kbs % kWChunkKB) == 0;
              const uint32_t a_tmem = tmem + kACol0 + ss * kASlotCols;
              if (fast) {
                const uint64_t bdesc = smem_desc_k_sw128(sB(ss));
#pragma unroll
                for (int j = 0; j < kBK / kUmmaK; ++j)
                  tc_mma_ts(tmem, a_tmem + j * (kUmmaK / 2), bdesc + static_cast<uint64_t>(j * 2),
                            idesc_w, (first && j == 0) ? 0u : 1u);
              } else {
                const uint64_t bdesc = smem_desc_k_sw128(sB(ss) + pass * (kTileM * 128));
#pragma unroll
                for (int j = 0; j < kBK / kUmmaK; ++j)
                  tc_mma_ts(tmem + b * kAccCols, a_tmem + j * (kUmmaK / 2),
                            bdesc + static_cast<uint64_t>(j * 2), idesc_n,
                            (first && j == 0) ? 0u : 1u);
              }
              tc_commit(empty_bar(ss));
            }
            pending = -1;
            if (cend) {
              tc_commit(accf_bar(b));
              ++ch;
            }
          }
        }
        if (!ok) *abort_flag = 1u;
      }
      __syncwarp();
      ch = __shfl_sync(0xffffffffu, ch, 0);
      it = __shfl_sync(0xffffffffu, it, 0);
      if (*abort_flag) break;
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles;
      const int passes = wide_tile_fast(a, mt, lane) ? 1 : 2;
      for (int pass = 0; pass < passes; ++pass) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kWStages;
          const uint32_t ph = (it / kWStages) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(s), ph, abort_flag, err,
                                                         kWaitTimeoutNs)))
            goto done;
          tc_fence_after();
          uint32_t h[32];
          const uint8_t* arow = gbase + (sA(s) - base);
          if (!INT4) {
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
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;  // 0..7
    const int q = warp & 3;
    const int colh = e >> 2;         // fast: 128-column half; slow: 64-column half
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int ch = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const bool fast = wide_tile_fast(a, mt, lane);
      const int n = nt * kTileN + row;
      const bool nvalid = n < p.N;
      const float swn = (EPI == kEpiY && nvalid) ? __ldg(p.sw + n) : 0.0f;
      if (fast) {
        const int b = ch & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                       err, kWaitTimeoutNs)))
          goto done;
        tc_fence_after();
        const int m0 = mt * kWTileM + colh * 128;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + colh * 128 + c4 * 32, v);
          tmem_wait_ld();
          if (c4 == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(b));
          }
          if (nvalid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + c4 * 32 + j;
              if (m < p.M) {
                const int64_t off = static_cast<int64_t>(m) * p.N + n;
                const float f = __uint_as_float(v[j]);  // an exact integer
                if (EPI == kEpiAcc)
                  p.acc[off] = __float2int_rn(f);
                else
                  p.y[off] = __float2half_rn(__fmul_rn(__fmul_rn(f, __ldg(p.sa + m)), swn));
              }
            }
          }
        }
        ++ch;
      } else {
        for (int pass = 0; pass < 2; ++pass) {
          int isum[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) isum[j] = 0;
          for (int c = 0; c < nch; ++c, ++ch) {
            const int b = ch & 1;
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
              for (int j = 0; j < 32; ++j) isum[hh * 32 + j] += __float2int_rn(__uint_as_float(v[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(b));
          }
          if (!nvalid) continue;
          const int m0 = mt * kWTileM + pass * kTileM + colh * 64;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int m = m0 + j;
            if (m < p.M) {
              const int64_t off = static_cast<int64_t>(m) * p.N + n;
              if (EPI == kEpiAcc)
                p.acc[off] = isum[j];
              else
                p.y[off] = __float2half_rn(
                    __fmul_rn(__fmul_rn(__int2float_rn(isum[j]), __ldg(p.sa + m)), swn));
            }
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


// ============================================================================
// Per-channel kernel, wide tiles, both MMA operands in shared memory and two
// 256-column accumulators in tensor memory (all 512 columns), so the epilogue
// drains one tile while the tensor pipe already works on the next.
//
// The converter warps read the TMA-staged weight codes, convert them to fp16
// and write them back to shared memory in the canonical K-major 128-byte
// swizzled layout the MMA descriptor expects (16-byte chunk c of row r at
// r * 128 + ((c ^ (r & 7)) << 4)), then fence the generic-proxy writes for
// the tensor core.  Stage layout: activation codes fp16 [256][64] (32 KiB) |
// weights fp16 [128][64] (16 KiB) | weight codes as loaded (8 KiB INT8 /
// 4 KiB INT4).  Exactness per tile exactly as in the kernel above.
// ============================================================================
constexpr int kSStages = 4;

template <bool INT4>
struct SCfg {
  static constexpr int kA8Bytes = INT4 ? kTileN * kBK / 2 : kTileN * kBK;
  static constexpr int kA16Bytes = kTileN * kBK * 2;
  static constexpr int kStageBytes = kWBStageBytes + kA16Bytes + kA8Bytes;
  static constexpr int kTmaBytes = kWBStageBytes + kA8Bytes;
  static constexpr int kBarOffset = kSStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOffset + (3 * kSStages + 4) * 8 + 16 + 1024;
};
static_assert(SCfg<false>::kStageBytes % 1024 == 0 && SCfg<true>::kStageBytes % 1024 == 0,
              "stages must keep 1024-byte alignment");
static_assert(SCfg<false>::kSmemBytes <= 232448, "shared memory budget");

template <bool INT4, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_wss_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const WideArgs a) {
  using C = SCfg<INT4>;
  const GemmArgs& p = a.g;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sB = [&](int s) { return base + s * C::kStageBytes; };
  auto sA16 = [&](int s) { return base + s * C::kStageBytes + kWBStageBytes; };
  auto sA8 = [&](int s) { return base + s * C::kStageBytes + kWBStageBytes + C::kA16Bytes; };
  const uint32_t bars = base + C::kBarOffset;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kSStages + s); };
  auto conv_bar = [&](int s) { return bars + 8u * (2 * kSStages + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (3 * kSStages + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (3 * kSStages + 2 + b); };
  const uint32_t tmem_slot = bars + 8u * (3 * kSStages + 4);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * (3 * kSStages + 4) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSStages; ++s) {
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
                                                              8 * (3 * kSStages + 4));
  const int nkb = (p.K + kBK - 1) / kBK;
  const int nch = (nkb + kWChunkKB - 1) / kWChunkKB;
  int* err = &g_device_error;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int passes = wide_tile_fast(a, mt, lane) ? 1 : 2;
      if (lane == 0) {
        for (int pass = 0; pass < passes; ++pass)
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = it % kSStages;
            const uint32_t ph = (it / kSStages) & 1;
            if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kWaitTimeoutNs)) break;
            mbar_arrive_expect_tx(full_bar(s), C::kTmaBytes);
            tma_load_2d(sB(s), &tmB, full_bar(s), kb * kBK, mt * kWTileM);
            tma_load_2d(sA8(s), &tmA, full_bar(s), INT4 ? kb * (kBK / 2) : kb * kBK, nt * kTileN);
          }
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_w = idesc_f16_f32(kTileN, kWTileM);
    constexpr uint32_t idesc_n = idesc_f16_f32(kTileN, kTileM);
    int it = 0, ch = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles;
      const bool fast = wide_tile_fast(a, mt, lane);
      if (lane == 0) {
        const int passes = fast ? 1 : 2;
        bool ok = true;
        for (int pass = 0; pass < passes && ok; ++pass) {
          int pending = -1;
          for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
            const bool cstart = fast ? (kb == 0) : (kb % kWChunkKB) == 0;
            const bool cend = fast ? (kb == nkb - 1) : ((kb % kWChunkKB) == kWChunkKB - 1 || kb == nkb - 1);
            const int b = ch & 1;
            if (cstart && ch >= 2) {
              // accumulator b was last used by chunk ch - 2: wait until it is drained
              ok = mbar_wait_bounded(acce_bar(b), ((ch - 2) >> 1) & 1, abort_flag, err, kWaitTimeoutNs);
              if (!ok) break;
              tc_fence_after();
            }
            const int s = it % kSStages;
            if ((kb & 1) == 0 && !cend) {
              pending = it;
              continue;
            }
            const uint32_t ph = (it / kSStages) & 1;
            if (!mbar_wait_bounded(conv_bar(s), ph, abort_flag, err, kWaitTimeoutNs)) { ok = false; break; }
            tc_fence_after();
            for (int q = (pending >= 0 ? 0 : 1); q < 2; ++q) {
              const int its = q == 0 ? pending : it;
              const int ss = its % kSStages;
              const int kbs = kb - (q == 0 ? 1 : 0);
              const bool first = fast ? (kbs == 0) : (kbs % kWChunkKB) == 0;
              const uint64_t adesc = smem_desc_k_sw128(sA16(ss));
              const uint64_t bdesc = smem_desc_k_sw128(sB(ss) + (fast ? 0 : pass * (kTileM * 128)));
#pragma unroll
              for (int j = 0; j < kBK / kUmmaK; ++j)
                tc_mma_ss(tmem + b * kWTileM, adesc + static_cast<uint64_t>(j * 2),
                          bdesc + static_cast<uint64_t>(j * 2), fast ? idesc_w : idesc_n,
                          (first && j == 0) ? 0u : 1u);
              tc_commit(empty_bar(ss));
            }
            pending = -1;
            if (cend) {
              tc_commit(accf_bar(b));
              ++ch;
            }
          }
        }
        if (!ok) *abort_flag = 1u;
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ converters
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles;
      const int passes = wide_tile_fast(a, mt, lane) ? 1 : 2;
      for (int pass = 0; pass < passes; ++pass) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kSStages;
          const uint32_t ph = (it / kSStages) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(s), ph, abort_flag, err,
                                                         kWaitTimeoutNs)))
            goto done;
          uint32_t h[32];
          const uint8_t* arow = gbase + (sA8(s) - base);
          if (!INT4) {
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
          uint8_t* drow = gbase + (sA16(s) - base) + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(drow + ((c ^ (row & 7)) << 4)) =
                make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(conv_bar(s));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;
    const int q = warp & 3;
    const int colh = e >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int ch = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const bool fast = wide_tile_fast(a, mt, lane);
      const int n = nt * kTileN + row;
      const bool nvalid = n < p.N;
      const float swn = (EPI == kEpiY && nvalid) ? __ldg(p.sw + n) : 0.0f;
      if (fast) {
        const int b = ch & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                       err, kWaitTimeoutNs)))
          goto done;
        tc_fence_after();
        const int m0 = mt * kWTileM + colh * 128;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + b * kWTileM + colh * 128 + c4 * 32, v);
          tmem_wait_ld();
          if (nvalid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + c4 * 32 + j;
              if (m < p.M) {
                const int64_t off = static_cast<int64_t>(m) * p.N + n;
                const float f = __uint_as_float(v[j]);  // an exact integer
                if (EPI == kEpiAcc)
                  p.acc[off] = __float2int_rn(f);
                else
                  p.y[off] = __float2half_rn(__fmul_rn(__fmul_rn(f, __ldg(p.sa + m)), swn));
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(b));
        ++ch;
      } else {
        for (int pass = 0; pass < 2; ++pass) {
          int isum[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) isum[j] = 0;
          for (int c = 0; c < nch; ++c, ++ch) {
            const int b = ch & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                           err, kWaitTimeoutNs)))
              goto done;
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t v[32];
              tmem_ld32(tmem + lane_base + b * kWTileM + colh * 64 + hh * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) isum[hh * 32 + j] += __float2int_rn(__uint_as_float(v[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(b));
          }
          if (!nvalid) continue;
          const int m0 = mt * kWTileM + pass * kTileM + colh * 64;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int m = m0 + j;
            if (m < p.M) {
              const int64_t off = static_cast<int64_t>(m) * p.N + n;
              if (EPI == kEpiAcc)
                p.acc[off] = isum[j];
              else
                p.y[off] = __float2half_rn(
                    __fmul_rn(__fmul_rn(__int2float_rn(isum[j]), __ldg(p.sa + m)), swn));
            }
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

// Test hook: wait on a barrier that no one completes, bounded by max_polls.
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

template <bool INT4, int EPI>
cudaError_t launch_wide(const CUtensorMap& tmA, const CUtensorMap& tmB, const WideArgs& a,
                        int num_sms, cudaStream_t st) {
  auto kern = gemm_wide_kernel<INT4, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                          WCfg<INT4>::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = a.g.num_tiles < num_sms ? a.g.num_tiles : num_sms;
  kern<<<grid, kThreads, WCfg<INT4>::kSmemBytes, st>>>(tmA, tmB, a);
  return cudaGetLastError();
}

template <bool INT4, int EPI>
cudaError_t launch_wss(const CUtensorMap& tmA, const CUtensorMap& tmB, const WideArgs& a,
                       int num_sms, cudaStream_t st) {
  auto kern = gemm_wss_kernel<INT4, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                          SCfg<INT4>::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = a.g.num_tiles < num_sms ? a.g.num_tiles : num_sms;
  kern<<<grid, kThreads, SCfg<INT4>::kSmemBytes, st>>>(tmA, tmB, a);
  return cudaGetLastError();
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
                           int group_size, int mode, __half* y, int32_t* acc, int num_sms,
                           cudaStream_t st) {
  if (group_size == 0 && row_l1 != nullptr)
    return launch_gemm_pair(qa16, sa, row_l1, M, N, K, w, int4, sw, mode, y, acc, st);
  CUtensorMap tmA, tmB;
  const bool wide = false;
  if (!make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qa16, K, M, K * 2, kBK,
                   wide ? kWTileM : kTileM, CU_TENSOR_MAP_SWIZZLE_128B))
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
  a.G = group_size > 0 ? static_cast<int>(K / group_size) : 1;
  a.num_m_tiles = static_cast<int>((M + kTileM - 1) / kTileM);
  a.num_tiles = a.num_m_tiles * static_cast<int>((N + kTileN - 1) / kTileN);
  a.sa = sa;
  a.sw = sw;
  a.y = y;
  a.acc = acc;
  if (wide) {
    WideArgs wa;
    wa.g = a;
    wa.g.num_m_tiles = static_cast<int>((M + kWTileM - 1) / kWTileM);
    wa.g.num_tiles = wa.g.num_m_tiles * static_cast<int>((N + kTileN - 1) / kTileN);
    wa.row_l1 = row_l1;
    wa.l1_limit = (1 << 23) / (int4 ? 8 : 127);
    // Up to K = 4096 the tile-boundary drain is a large share of a tile, so
    // the double-buffered kernel (weights through shared memory) wins; for
    // longer K the single-accumulator kernel with the weight operand in
    // tensor memory is faster (less shared-memory traffic per stage).
    // Measured crossover on GB300: equal at K = 4096.
    if (K > kLongK) {
      if (int4)
        return mode == kEpiY ? launch_wide<true, kEpiY>(tmA, tmB, wa, num_sms, st)
                             : launch_wide<true, kEpiAcc>(tmA, tmB, wa, num_sms, st);
      return mode == kEpiY ? launch_wide<false, kEpiY>(tmA, tmB, wa, num_sms, st)
                           : launch_wide<false, kEpiAcc>(tmA, tmB, wa, num_sms, st);
    }
    if (int4)
      return mode == kEpiY ? launch_wss<true, kEpiY>(tmA, tmB, wa, num_sms, st)
                           : launch_wss<true, kEpiAcc>(tmA, tmB, wa, num_sms, st);
    return mode == kEpiY ? launch_wss<false, kEpiY>(tmA, tmB, wa, num_sms, st)
                         : launch_wss<false, kEpiAcc>(tmA, tmB, wa, num_sms, st);
  }
  const bool pg = group_size > 0;
#define CIDER_TC_CASE(I4, P, E) \
  if (int4 == I4 && pg == P && mode == E) return launch_tc<I4, P, E>(tmA, tmB, a, num_sms, st);
  CIDER_TC_CASE(false, false, kEpiY)
  CIDER_TC_CASE(false, true, kEpiY)
  CIDER_TC_CASE(false, false, kEpiAcc)
  CIDER_TC_CASE(false, true, kEpiAcc)
  CIDER_TC_CASE(true, false, kEpiY)
  CIDER_TC_CASE(true, true, kEpiY)
  CIDER_TC_CASE(true, false, kEpiAcc)
  CIDER_TC_CASE(true, true, kEpiAcc)
#undef CIDER_TC_CASE
  return cudaErrorInvalidValue;
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
