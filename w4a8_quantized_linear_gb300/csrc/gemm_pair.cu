// gemm_pair.cu -- per-channel tensor-core GEMM with fused dequant on CTA
// pairs (Cider README, page "cider": "Architecture / Metal kernel pipeline",
// matmul_fused_dequant: INT8 x INT8 -> INT32 -> FP16 with the scales applied
// in the store; W4A8 unpacks INT4 ahead of the multiply, "Modes").
//
// The exact integer product runs on the fp16 tensor pipe (sm_103a has no
// integer tcgen05 kind): codes are exact fp16 values and products exact
// integers; the fp32 accumulation is exact while every partial sum stays
// below 2^24 (see the per-tile bound below).
//
// A cluster of two CTAs (on two SMs) computes a 256 x 256 output tile,
// 256 weight rows (n) x 256 tokens (m), with tcgen05.mma.cta_group::2:
// CTA r of the pair holds weight rows [128 r, 128 r + 128) of the tile (the
// MMA's A operand, M = 256 split over the pair) and tokens [128 r, 128 r + 128)
// (its half of the B operand, N = 256); each CTA's tensor memory receives its
// own 128 weight rows x all 256 tokens.  Per SM this halves the activation
// bytes read from L2 and shared memory per multiply-add compared with a
// 128 x 256 tile on one SM, which is what lets the tensor pipe run at its
// full rate.
//
// Roles in each CTA (one CTA per SM, persistent over tiles):
//   warp 0      activation producer: TMA of the CTA's fp16 codes [128 m][64 k]
//               (128-byte swizzle) into the 6-stage operand ring; the copies
//               of both CTAs complete on the even CTA's "ready" barrier.
//   warp 14     weight producer: TMA of int8 codes [128 n][64 k] (64-byte
//               swizzle; INT4: packed [128 n][32 B], 32-byte swizzle) into a
//               separate 4-slot ring, running ahead of the conversion.
//   warps 2-9   converters, two groups of 4 warps taking alternate stages:
//               each thread owns one weight row, converts its 64 codes of the
//               stage to fp16 and writes them into the stage's A operand in
//               the canonical K-major 128-byte-swizzled layout as soon as the
//               stage is free, then reports to the even CTA's "ready" barrier.
//               (One group alone is latency-bound at ~450 ns per stage, the
//               MMAs of a stage take ~250 ns.)
//   warp 1      even CTA only, one thread: waits until both CTAs' stages are
//               ready, issues 4 MMAs (K = 16 each) into one of two 256-column
//               accumulators, and commits to both CTAs' barriers (stage free;
//               accumulator full).  Both CTAs' warp 1 allocate tensor memory.
//   warps 10-13 epilogue, one per tensor-memory lane quarter: drain the
//               accumulator (tcgen05.ld), dequantize, store fp16 y (or int32
//               accumulators), release it.
// Keeping the int8 weights out of the operand ring leaves room for six
// 32 KiB stages: enough work in flight to cover the ~2 us it takes to refill
// a stage (commit, TMA from L2, conversion, cross-CTA signal).
//
// Exactness per tile: every partial sum of token m is bounded by
// qmax_w * sum_k |q_a[m,k]| (qmax_w = 127 INT8, 8 INT4).  When that bound is
// <= 2^23 for all 256 tokens of the tile ("fast" tile, the normal case) all of
// K accumulates in fp32 exactly and the accumulator is drained once.  Else
// ("slow" tile) the tile runs as four passes of 64 tokens (N = 64 MMAs, 32
// tokens from each CTA) whose accumulators are drained every 512 K into exact
// int32 register sums.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kPTileN = 256;          // weight rows per pair tile (MMA M)
constexpr int kPTileM = 256;          // tokens per pair tile (MMA N)
constexpr int kPHalf = 128;           // rows of each operand per CTA
constexpr int kPBK = 64;              // K per pipeline stage
constexpr int kPUmmaK = 16;
constexpr int kPStages = 6;           // operand ring (activations + converted weights)
constexpr int kP8Slots = 4;           // int8 / int4 weight ring
constexpr int kPChunkKB = 8;          // slow tiles: drain every 512 K
constexpr int kPThreads = 480;
constexpr int kPConvWarp0 = 2;        // two groups of 4 converter warps
constexpr int kPEpiWarp0 = 10;
constexpr int kPSlowPasses = 4;       // slow tiles: 64 tokens per pass
constexpr int kPW8Warp = 14;
constexpr int kPAccCols = 256;
constexpr int kPTmemCols = 512;
constexpr int kPBBytes = kPHalf * kPBK * 2;    // 16 KiB activation codes
constexpr int kPA16Bytes = kPHalf * kPBK * 2;  // 16 KiB converted weights
constexpr int kPStageBytes = kPBBytes + kPA16Bytes;
constexpr uint64_t kPWaitNs = 2000000000ull;

template <bool INT4>
struct PCfg {
  static constexpr int kA8Bytes = INT4 ? kPHalf * kPBK / 2 : kPHalf * kPBK;
  static constexpr int kA8Offset = kPStages * kPStageBytes;
  static constexpr int kBarOffset = kA8Offset + kP8Slots * 8192;
  // ready, empty per stage; full8, empty8 per weight slot; accf x2, acce x2,
  // mma_done; tmem slot; abort
  static constexpr int kNumBars = 2 * kPStages + 2 * kP8Slots + 5;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;
};
static_assert(kPStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for the swizzle");
static_assert(PCfg<false>::kSmemBytes <= 232448, "shared memory budget");

struct PairArgs {
  int M, N, K;
  int num_m_tiles, num_tiles;
  const float* sa;
  const float* sw;
  __half* y;
  int32_t* acc;
  const int* row_l1;
  int l1_limit;
  int* err;
};

// Whole warp: is every token of token tile mt within the exactness bound?
__device__ __forceinline__ bool pair_tile_fast(const PairArgs& a, int mt, int lane) {
  int mx = 0;
#pragma unroll
  for (int i = 0; i < kPTileM / 32; ++i) {
    const int m = mt * kPTileM + i * 32 + lane;
    if (m < a.M) mx = max(mx, __ldg(a.row_l1 + m));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  return mx <= a.l1_limit;
}

template <bool INT4, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const PairArgs p) {
  using C = PCfg<INT4>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sB = [&](int s) { return base + s * kPStageBytes; };
  auto sA16 = [&](int s) { return base + s * kPStageBytes + kPBBytes; };
  auto sA8 = [&](int j) { return base + C::kA8Offset + j * 8192; };
  const uint32_t bars = base + C::kBarOffset;
  auto ready_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kPStages + s); };
  auto full8_bar = [&](int j) { return bars + 8u * (2 * kPStages + j); };
  auto empty8_bar = [&](int j) { return bars + 8u * (2 * kPStages + kP8Slots + j); };
  constexpr int kBar2 = 2 * kPStages + 2 * kP8Slots;
  auto accf_bar = [&](int b) { return bars + 8u * (kBar2 + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (kBar2 + 2 + b); };
  const uint32_t done_bar = bars + 8u * (kBar2 + 4);
  const uint32_t tmem_slot = bars + 8u * (kBar2 + 5);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * (kBar2 + 5) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  int* err = p.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      // the even CTA's producer arrival (with the byte count of both CTAs'
      // activation copies) + 4 converter warps x 2 CTAs
      mbar_init(ready_bar(s), 9);
      mbar_init(empty_bar(s), 1);
    }
    for (int j = 0; j < kP8Slots; ++j) {
      mbar_init(full8_bar(j), 1);
      mbar_init(empty8_bar(j), 4);     // the 4 warps of the converter group of this use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 8);       // 4 epilogue warps x 2 CTAs
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tmB);
  if (warp == kPW8Warp && lane == 0) prefetch_tensormap(&tmA);
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // barriers of both CTAs initialised, tensor memory held
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset +
                                                              8 * (kBar2 + 5));
  const int nkb = (p.K + kPBK - 1) / kPBK;
  const int nch = (nkb + kPChunkKB - 1) / kPChunkKB;

  if (warp == 0) {
    // ------------------------------------------------------------ activation producer
    const uint32_t ready_leader0 = mapa_shared(ready_bar(0), 0);
    int it = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      const int mt = tile % p.num_m_tiles;
      const int passes = pair_tile_fast(p, mt, lane) ? 1 : kPSlowPasses;
      if (lane == 0) {
        for (int pass = 0; pass < passes; ++pass)
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = it % kPStages;
            const uint32_t ph = (it / kPStages) & 1;
            if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kPWaitNs)) break;
            if (rank == 0) mbar_arrive_expect_tx(ready_bar(s), 2 * kPBBytes);
            tma_load_2d_pair(sB(s), &tmB, ready_leader0 + 8u * s, kb * kPBK,
                             mt * kPTileM + rank * kPHalf);
          }
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else if (warp == kPW8Warp) {
    // ------------------------------------------------------------ weight producer
    int it = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int passes = pair_tile_fast(p, mt, lane) ? 1 : kPSlowPasses;
      if (lane == 0) {
        for (int pass = 0; pass < passes; ++pass)
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int j = it % kP8Slots;
            const uint32_t ph = (it / kP8Slots) & 1;
            if (!mbar_wait_bounded(empty8_bar(j), ph ^ 1u, abort_flag, err, kPWaitNs)) break;
            mbar_arrive_expect_tx(full8_bar(j), C::kA8Bytes);
            tma_load_2d(sA8(j), &tmA, full8_bar(j), INT4 ? kb * (kPBK / 2) : kb * kPBK,
                        nt * kPTileN + rank * kPHalf);
          }
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0) {
      constexpr uint32_t idesc_fast = idesc_f16_f32(kPTileN, kPTileM);
      constexpr uint32_t idesc_slow = idesc_f16_f32(kPTileN, kPTileM / kPSlowPasses);
      int it = 0, ch = 0;
      for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
        const int mt = tile % p.num_m_tiles;
        const bool fast = pair_tile_fast(p, mt, lane);
        if (lane == 0) {
          const int passes = fast ? 1 : kPSlowPasses;
          bool ok = true;
          for (int pass = 0; pass < passes && ok; ++pass) {
            for (int kb = 0; kb < nkb; ++kb, ++it) {
              const bool cstart = fast ? (kb == 0) : (kb % kPChunkKB) == 0;
              const bool cend =
                  fast ? (kb == nkb - 1) : ((kb % kPChunkKB) == kPChunkKB - 1 || kb == nkb - 1);
              const int b = ch & 1;
              if (cstart && ch >= 2) {
                // accumulator b was last used by chunk ch - 2: wait until both CTAs drained it
                ok = mbar_wait_bounded(acce_bar(b), ((ch - 2) >> 1) & 1, abort_flag, err, kPWaitNs);
                if (!ok) break;
                tc_fence_after();
              }
              const int s = it % kPStages;
              const uint32_t ph = (it / kPStages) & 1;
              if (!mbar_wait_bounded(ready_bar(s), ph, abort_flag, err, kPWaitNs)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t adesc = smem_desc_k_sw128(sA16(s));
              // slow pass p uses rows [32 p, 32 p + 32) of each CTA's 128 tokens
              const uint64_t bdesc = smem_desc_k_sw128(sB(s) + (fast ? 0 : pass * (32 * 128)));
#pragma unroll
              for (int j = 0; j < kPBK / kPUmmaK; ++j)
                tc_mma_ss_pair(tmem + b * kPAccCols, adesc + static_cast<uint64_t>(j * 2),
                               bdesc + static_cast<uint64_t>(j * 2), fast ? idesc_fast : idesc_slow,
                               (cstart && j == 0) ? 0u : 1u);
              tc_commit_pair_mc(empty_bar(s), 0x3);
              if (cend) {
                tc_commit_pair_mc(accf_bar(b), 0x3);
                ++ch;
              }
            }
          }
          if (!ok) *abort_flag = 1u;
        }
        __syncwarp();
        if (*abort_flag) break;
      }
      // every MMA issued so far completes before either CTA frees tensor memory
      if (lane == 0) tc_commit_pair_mc(done_bar, 0x3);
      __syncwarp();
    }
  } else if (warp < kPEpiWarp0) {
    // ------------------------------------------------------------ converters
    const int group = (warp - kPConvWarp0) >> 2;   // takes the uses with it % 2 == group
    const int row = (warp & 3) * 32 + lane;
    const uint32_t ready_leader0 = mapa_shared(ready_bar(0), 0);
    int it = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      const int mt = tile % p.num_m_tiles;
      const int passes = pair_tile_fast(p, mt, lane) ? 1 : kPSlowPasses;
      for (int pass = 0; pass < passes; ++pass) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          if ((it & 1) != group) continue;
          const int j8 = it % kP8Slots;
          const uint32_t ph8 = (it / kP8Slots) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(full8_bar(j8), ph8, abort_flag, err,
                                                         kPWaitNs)))
            goto done;
          uint32_t h[32];
          const uint8_t* arow = gbase + (sA8(j8) - base);
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
              for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t t[4];
                s4x8_to_h2x4(vw[q4], t);
                h[16 * c + 4 * q4 + 0] = t[0];
                h[16 * c + 4 * q4 + 1] = t[1];
                h[16 * c + 4 * q4 + 2] = t[2];
                h[16 * c + 4 * q4 + 3] = t[3];
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty8_bar(j8));   // weight slot consumed (in registers)
          // the stage's A operand is free once the MMAs of its previous use completed
          const int s = it % kPStages;
          const uint32_t ph = (it / kPStages) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err,
                                                         kPWaitNs)))
            goto done;
          uint8_t* drow = gbase + (sA16(s) - base) + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(drow + ((c ^ (row & 7)) << 4)) =
                make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(ready_leader0 + 8u * s);
        }
      }
    }
  } else if (warp < kPW8Warp) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // tensor-memory lane quarter of this warp
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    int ch = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const bool fast = pair_tile_fast(p, mt, lane);
      const int n = nt * kPTileN + static_cast<int>(rank) * kPHalf + row;
      const bool nvalid = n < p.N;
      const float swn = (EPI == kEpiY && nvalid) ? __ldg(p.sw + n) : 0.0f;
      if (fast) {
        const int b = ch & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag, err,
                                                       kPWaitNs)))
          goto done;
        tc_fence_after();
        // column j of the accumulator is token mt * 256 + j
        const int m0 = mt * kPTileM;
#pragma unroll 1
        for (int c8 = 0; c8 < kPAccCols / 32; ++c8) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + b * kPAccCols + c8 * 32, v);
          tmem_wait_ld();
          if (nvalid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + c8 * 32 + j;
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
        if (lane == 0) mbar_arrive_remote(acce_leader0 + 8u * b);
        ++ch;
      } else {
        for (int pass = 0; pass < kPSlowPasses; ++pass) {
          int isum[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) isum[j] = 0;
          for (int c = 0; c < nch; ++c, ++ch) {
            const int b = ch & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                           err, kPWaitNs)))
              goto done;
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t v[32];
              tmem_ld32(tmem + lane_base + b * kPAccCols + hh * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) isum[hh * 32 + j] += __float2int_rn(__uint_as_float(v[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acce_leader0 + 8u * b);
          }
          if (!nvalid) continue;
          // N = 64 pass: column j is row 32 pass + (j % 32) of the tokens of CTA j / 32
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int m = mt * kPTileM + (j >> 5) * kPHalf + pass * 32 + (j & 31);
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
  if (warp == 1) {
    // the even CTA's last commit reaches both CTAs; wait for it (bounded, and
    // also after an abort) so no MMA is in flight when the pair frees its
    // tensor memory
    if (lane == 0) {
      volatile uint32_t keep_waiting = 0u;
      mbar_wait_bounded(done_bar, 0, &keep_waiting, err, kPWaitNs);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // neither CTA leaves while the other may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPTmemCols);
  }
}

template <bool INT4, int EPI>
cudaError_t launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const PairArgs& a,
                        cudaStream_t st) {
  auto kern = gemm_pair_kernel<INT4, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                          PCfg<INT4>::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  // clusters that fit on the GPU at once (one CTA per SM), cached per device
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int nc = dev < 64 ? max_clusters[dev].load(std::memory_order_relaxed) : 0;
  if (nc <= 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = PCfg<INT4>::kSmemBytes;
    int q = 0;
    if (cudaOccupancyMaxActiveClusters(&q, reinterpret_cast<const void*>(kern), &cfg) !=
            cudaSuccess ||
        q <= 0) {
      (void)cudaGetLastError();
      q = sms / 2;
    }
    nc = q;
    if (dev < 64) max_clusters[dev].store(nc, std::memory_order_relaxed);
  }
  const int clusters = a.num_tiles < nc ? a.num_tiles : nc;
  kern<<<2 * clusters, kPThreads, PCfg<INT4>::kSmemBytes, st>>>(tmA, tmB, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_pair(const __half* qa16, const float* sa, const int* row_l1, int64_t M,
                             int64_t N, int64_t K, const uint8_t* w, bool int4, const float* sw,
                             int mode, __half* y, int32_t* acc, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  if (!make_tensor_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qa16, K, M, K * 2, kPBK, kPHalf,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t wbytes = int4 ? K / 2 : K;
  if (!make_tensor_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, N, wbytes,
                          int4 ? kPBK / 2 : kPBK, kPHalf,
                          int4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  PairArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.num_m_tiles = static_cast<int>((M + kPTileM - 1) / kPTileM);
  a.num_tiles = a.num_m_tiles * static_cast<int>((N + kPTileN - 1) / kPTileN);
  a.sa = sa;
  a.sw = sw;
  a.y = y;
  a.acc = acc;
  a.row_l1 = row_l1;
  a.l1_limit = (1 << 23) / (int4 ? 8 : 127);
  cudaError_t e = device_error_word(&a.err);
  if (e != cudaSuccess) return e;
  if (int4)
    return mode == kEpiY ? launch_pair<true, kEpiY>(tmA, tmB, a, st)
                         : launch_pair<true, kEpiAcc>(tmA, tmB, a, st);
  return mode == kEpiY ? launch_pair<false, kEpiY>(tmA, tmB, a, st)
                       : launch_pair<false, kEpiAcc>(tmA, tmB, a, st);
}

}  // namespace cider
