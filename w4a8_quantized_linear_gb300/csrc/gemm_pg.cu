// gemm_pg.cu -- per-group tensor-core GEMM with fused dequant on CTA pairs
// (Cider README, page "cider": "Architecture / Metal kernel pipeline",
// matmul_fused_dequant; per-group weight scales, one per 64 or 128 K
// elements, from "W8A8 quantization granularity"; W4A8 unpacks INT4 ahead of
// the multiply, "Modes").
//
// y[m,n] = fp16(s_a[m] * sum over groups g, increasing, of s_w[n,g] * acc_g),
// acc_g the exact integer dot product over group g's K range (a
// reassociation of (s_a * s_w) * acc_g summed in fp32, within a few fp32
// ulps of it).
//
// As in the per-channel kernel, the exact integer products run on the fp16
// tensor pipe: codes are exact fp16 values, every product an exact integer,
// and a group's sum (|acc_g| <= 127 * 127 * 128 < 2^21) is exact in fp32, so
// the accumulator is drained once per group.
//
// A cluster of two CTAs computes a 256-token x 128-weight-row tile with
// tcgen05.mma.cta_group::2 (M = 256 tokens, N = 128 weight rows, K = 16):
// CTA r holds tokens [128 r, 128 r + 128) (its half of the A operand, fp16
// codes by TMA) and weight rows [64 r, 64 r + 64) (its half of B, converted
// to fp16 by converter warps); each CTA's tensor memory receives its 128
// tokens (one per lane) x the tile's 128 weight rows.  Four 128-column
// accumulators let the MMA run up to three groups ahead of the drain.  (A
// 256-wide tile would need 256 running sums per token row, more than the
// register file holds beside the pipeline.)
//
// Roles in each CTA (one CTA per SM, persistent over tiles):
//   warp 0      producer: TMA of the CTA's activation codes, two [128 m][64 k]
//               sub-tiles per 128-K stage, both CTAs' copies completing on the
//               even CTA's "ready" barrier.
//   warps 1, 7  even CTA only, one thread each, alternate stages: per stage
//               and group, waits for a free accumulator, issues the group's
//               MMAs (8 per 128-K group, 4 per 64-K group) and commits
//               "accumulator full" to both CTAs; commits "stage free" after
//               the stage.
//   warps 2-5   converters, two groups of two warps taking alternate stages:
//               thread = weight row, its 128 codes of the stage -> fp16 in the
//               K-major 128-byte-swizzled operand layout; report to the even
//               CTA's "ready" barrier.
//   warp 6      weight-code producer: TMA of the int8 codes [64 n][64 k]
//               (INT4: packed [64 n][32 B]) into a 4-slot ring.
//   warps 8-23  epilogue, four per tensor-memory lane quarter (32 columns
//               each): per group, tcgen05.ld of its 32 columns, fp32 running
//               sums += s_w[n,g] * acc_g, the group's 32 weight scales read as
//               shared-memory broadcasts; at the tile's end y = fp16(s_a * sum)
//               with 16-byte stores.  Each warp streams its weight scales into
//               a 4-group ring in shared memory with asynchronous copies issued
//               three groups ahead: the scales of one row sit G * 4 bytes apart
//               in global memory, and a cache round trip per group on the
//               drain's critical path held earlier per-group kernels to a third
//               of the tensor rate.  In accumulator mode each group's exact
//               int32 values are stored instead.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kGTileM = 256;           // tokens per pair tile (MMA M)
constexpr int kGTileN = 128;           // weight rows per pair tile (MMA N)
constexpr int kGHalfM = 128;           // tokens per CTA
constexpr int kGHalfN = 64;            // weight rows per CTA
constexpr int kGSubK = 64;             // K per swizzled sub-tile (128 bytes of fp16)
constexpr int kGSub = 2;               // sub-tiles per stage
constexpr int kGBK = kGSub * kGSubK;   // K per stage
constexpr int kGUmmaK = 16;
constexpr int kGAccCols = kGTileN;
constexpr int kGAccBufs = 4;
constexpr int kGTmemCols = kGAccCols * kGAccBufs;            // 512
constexpr int kGASubBytes = kGHalfM * kGSubK * 2;            // 16 KiB
constexpr int kGBSubBytes = kGHalfN * kGSubK * 2;            // 8 KiB
constexpr int kGAOpBytes = kGSub * kGASubBytes;              // 32 KiB
constexpr int kGBOpBytes = kGSub * kGBSubBytes;              // 16 KiB
constexpr int kGStageBytes = kGAOpBytes + kGBOpBytes;        // 48 KiB
constexpr int kGStages = 4;
constexpr int kG8Slots = 4;
constexpr int kG8SlotBytes = kGHalfN * kGSubK;               // 4 KiB (int8 sub-tile)
constexpr int kGConvWarp0 = 2;
constexpr int kGW8Warp = 6;
constexpr int kGMma2Warp = 7;                                // second MMA issuer
constexpr int kGEpiWarp0 = 8;
constexpr int kGEpiWarps = 16;                               // 4 per lane quarter, 32 columns each
constexpr int kGThreads = 32 * (kGEpiWarp0 + kGEpiWarps);    // 768
// the even CTA's producer arrival (with both CTAs' activation bytes) + the
// two converter warps of the stage's group in each CTA
constexpr int kGReadyCount = 1 + 2 * 2;
constexpr uint32_t kGReadyBytes = 2 * kGAOpBytes;
constexpr int kGSwRing = 4;                                  // groups of weight scales in flight
constexpr int kGSwBytes = kGEpiWarps * kGSwRing * 32 * 4;     // per warp: ring of 32-scale vectors
constexpr uint64_t kGWaitNs = 2000000000ull;

static_assert(kGASubBytes % 1024 == 0 && kGBSubBytes % 1024 == 0,
              "sub-tiles keep 1024-byte alignment for the swizzle");
static_assert(kGTmemCols == 512, "tensor memory: four 128-column accumulators");

template <bool INT4>
struct GCfg {
  static constexpr int kA8Bytes = INT4 ? kGHalfN * kGSubK / 2 : kGHalfN * kGSubK;
  static constexpr int kA8Offset = kGStages * kGStageBytes;
  static constexpr int kSwOffset = kA8Offset + kG8Slots * kG8SlotBytes;
  static constexpr int kBarOffset = kSwOffset + kGSwBytes;
  // ready, empty per stage; full8, empty8 per weight slot; accf, acce per
  // accumulator; mma_done; then the tensor-memory slot and the abort flag
  static constexpr int kBar8 = 2 * kGStages;
  static constexpr int kBarAcc = kBar8 + 2 * kG8Slots;
  static constexpr int kNumBars = kBarAcc + 2 * kGAccBufs + 1;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct PgArgs {
  int M, N, K;
  int gs, G;          // group size (64 or 128), groups per row
  int num_m_tiles, num_tiles;
  int nkb;            // 128-K stages per tile
  const float* sa;
  const float* sw;    // [N, G]
  __half* y;
  int32_t* acc;       // [M, N, G] (accumulator mode)
  int* err;
};

template <bool INT4, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGThreads, 1)
    gemm_pg_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const PgArgs p) {
  using C = GCfg<INT4>;
  constexpr int S = kGStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sA = [&](int s) { return base + s * kGStageBytes; };               // activation codes
  auto sB = [&](int s) { return base + s * kGStageBytes + kGAOpBytes; };  // fp16 weights
  auto sW8 = [&](int j) { return base + C::kA8Offset + j * kG8SlotBytes; };
  const uint32_t bars = base + C::kBarOffset;
  auto ready_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto full8_bar = [&](int j) { return bars + 8u * (C::kBar8 + j); };
  auto empty8_bar = [&](int j) { return bars + 8u * (C::kBar8 + kG8Slots + j); };
  auto accf_bar = [&](int b) { return bars + 8u * (C::kBarAcc + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (C::kBarAcc + kGAccBufs + b); };
  const uint32_t done_bar = bars + 8u * (C::kBarAcc + 2 * kGAccBufs);
  const uint32_t tmem_slot = bars + 8u * C::kNumBars;
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * C::kNumBars + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int gpk = kGBK / p.gs;   // groups per 128-K stage: 1 or 2
  int* err = p.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(ready_bar(s), kGReadyCount);
      mbar_init(empty_bar(s), 1);
    }
    for (int j = 0; j < kG8Slots; ++j) {
      mbar_init(full8_bar(j), 1);
      mbar_init(empty8_bar(j), 2);     // the 2 warps of the converter group of this use
    }
    for (int b = 0; b < kGAccBufs; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * kGEpiWarps);   // 16 epilogue warps x 2 CTAs
    }
    mbar_init(done_bar, 2);            // the last commit of each of the two MMA issuers
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kGTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // barriers of both CTAs initialised, tensor memory held
  tc_fence_after();
  const uint32_t tmem =
      *reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * C::kNumBars);

  if (warp == 0) {
    // ------------------------------------------------------------ activation producer
    if (lane == 0) {
      const uint32_t ready_leader0 = mapa_shared(ready_bar(0), 0);
      int it = 0;
      for (int tile = cid; tile < p.num_tiles && !*abort_flag; tile += nclusters) {
        const int mt = tile % p.num_m_tiles;
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!mbar_sleep_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kGWaitNs)) break;
          if (rank == 0) mbar_arrive_expect_tx(ready_bar(s), kGReadyBytes);
          for (int t = 0; t < kGSub; ++t)
            tma_load_2d_pair(sA(s) + t * kGASubBytes, &tmX, ready_leader0 + 8u * s,
                             kb * kGBK + t * kGSubK, mt * kGTileM + rank * kGHalfM);
        }
      }
    }
  } else if (warp == 1 || warp == kGMma2Warp) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    // Two issuing threads on different SM sub-partitions take alternate
    // stages: issuing one tcgen05.mma with its bookkeeping costs a thread
    // about as long as the tensor core takes to execute a 256 x 128 x 16
    // product, so one issuer alone would leave the tensor pipe idle half the
    // time.  Each stage's groups use their own accumulators, and each issuer
    // commits only its own MMAs, so the two never wait on each other.
    const int who = warp == 1 ? 0 : 1;
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kGTileM, kGTileN);
      const int mmas_per_group = p.gs / kGUmmaK;
      int it = 0, ti = 0;
      bool ok = true;
      for (int tile = cid; tile < p.num_tiles && ok; tile += nclusters, ++ti) {
        for (int kb = 0; kb < p.nkb && ok; ++kb, ++it) {
          if ((it & 1) != who) continue;
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!mbar_wait_bounded(ready_bar(s), ph, abort_flag, err, kGWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_k_sw128(sA(s));
          const uint64_t bdesc = smem_desc_k_sw128(sB(s));
          // groups of this stage (the last stage of a K = 64 (mod 128) row has one)
          const int ng = min(gpk, p.G - kb * gpk);
          for (int t = 0; t < ng; ++t) {
            const int ch = ti * p.G + kb * gpk + t;   // group number in this pair's sequence
            const int b = ch % kGAccBufs;
            if (ch >= kGAccBufs) {
              // accumulator b was last used by group ch - 4: wait until both CTAs drained it
              if (!mbar_wait_bounded(acce_bar(b), ((ch - kGAccBufs) / kGAccBufs) & 1, abort_flag,
                                     err, kGWaitNs)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d = tmem + b * kGAccCols;
            if (mmas_per_group == 8) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                tc_mma_ss_pair(d, adesc + static_cast<uint64_t>((j >> 2) * (kGASubBytes >> 4) + (j & 3) * 2),
                               bdesc + static_cast<uint64_t>((j >> 2) * (kGBSubBytes >> 4) + (j & 3) * 2),
                               idesc, j == 0 ? 0u : 1u);
            } else {
              // 64-K group: sub-tile t of the stage
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tc_mma_ss_pair(d, adesc + static_cast<uint64_t>(t * (kGASubBytes >> 4) + j * 2),
                               bdesc + static_cast<uint64_t>(t * (kGBSubBytes >> 4) + j * 2),
                               idesc, j == 0 ? 0u : 1u);
            }
            tc_commit_pair_mc(accf_bar(b), 0x3);
          }
          if (!ok) break;
          tc_commit_pair_mc(empty_bar(s), 0x3);
        }
      }
      if (!ok) *abort_flag = 1u;
      // every MMA this thread issued completes before either CTA frees tensor memory
      tc_commit_pair_mc(done_bar, 0x3);
    }
    __syncwarp();
  } else if (warp < kGConvWarp0 + 4) {
    // ------------------------------------------------------------ converters
    const int group = (warp - kGConvWarp0) >> 1;   // takes the stages with it % 2 == group
    const int row = (warp & 1) * 32 + lane;        // weight row within the CTA's 64
    const uint32_t ready_leader0 = mapa_shared(ready_bar(0), 0);
    int it = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      for (int kb = 0; kb < p.nkb; ++kb, ++it) {
        if ((it & 1) != group) continue;
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        uint8_t* drow = gbase + (sB(s) - base) + row * 128;
#pragma unroll 1
        for (int t = 0; t < kGSub; ++t) {
          const int v8 = it * kGSub + t;   // weight sub-tile index
          const int j8 = v8 % kG8Slots;
          const uint32_t ph8 = (v8 / kG8Slots) & 1;
          if (!__all_sync(0xffffffffu,
                          mbar_sleep_bounded(full8_bar(j8), ph8, abort_flag, err, kGWaitNs)))
            goto done;
          uint32_t h[32];
          const uint8_t* arow = gbase + (sW8(j8) - base);
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
              for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t tt[4];
                s4x8_to_h2x4(vw[q4], tt);
                h[16 * c + 4 * q4 + 0] = tt[0];
                h[16 * c + 4 * q4 + 1] = tt[1];
                h[16 * c + 4 * q4 + 2] = tt[2];
                h[16 * c + 4 * q4 + 3] = tt[3];
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty8_bar(j8));   // weight slot consumed (in registers)
          // the stage's weight operand is free once the MMAs of its previous use completed
          if (t == 0 && !__all_sync(0xffffffffu, mbar_sleep_bounded(empty_bar(s), ph ^ 1u,
                                                                   abort_flag, err, kGWaitNs)))
            goto done;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(drow + t * kGBSubBytes + ((c ^ (row & 7)) << 4)) =
                make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(ready_leader0 + 8u * s);
      }
    }
  } else if (warp == kGW8Warp) {
    // ------------------------------------------------------------ weight-code producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = cid; tile < p.num_tiles && ok; tile += nclusters) {
        const int nt = tile / p.num_m_tiles;
        for (int kb = 0; kb < p.nkb && ok; ++kb)
          for (int t = 0; t < kGSub; ++t, ++it) {
            const int j = it % kG8Slots;
            const uint32_t ph = (it / kG8Slots) & 1;
            if (!mbar_sleep_bounded(empty8_bar(j), ph ^ 1u, abort_flag, err, kGWaitNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full8_bar(j), C::kA8Bytes);
            const int k0 = kb * kGBK + t * kGSubK;
            tma_load_2d(sW8(j), &tmW, full8_bar(j), INT4 ? k0 / 2 : k0,
                        nt * kGTileN + rank * kGHalfN);
          }
      }
    }
  } else if (warp >= kGEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kGEpiWarp0;          // 0..15
    const int q = warp & 3;                   // tensor-memory lane quarter of this warp
    const int c4 = e >> 2;                    // accumulator columns [32 c4, 32 c4 + 32)
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    // this warp's ring of weight-scale vectors: slot r holds the 32 scales of one group
    const uint32_t sw_ring = base + C::kSwOffset + e * (kGSwRing * 32 * 4);
    const float* sw_ring_g = reinterpret_cast<const float*>(gbase + C::kSwOffset) + e * (kGSwRing * 32);
    const int row = q * 32 + lane;            // token of this thread within the CTA's 128
    // scales of the f-th (tile, group) of this pair, in the order the drain
    // uses them: lane l copies row 32 c4 + l of that tile's weight rows
    auto fetch_scales = [&](int f) {
      const int tile = cid + (f / p.G) * nclusters;
      if (EPI == kEpiY && tile < p.num_tiles) {
        const int g = f % p.G;
        const int n = (tile / p.num_m_tiles) * kGTileN + c4 * 32 + lane;
        cp_async4(sw_ring + (f % kGSwRing) * 128 + lane * 4,
                  p.sw + (n < p.N ? static_cast<int64_t>(n) * p.G + g : 0), n < p.N);
      }
      cp_async_commit();   // one commit group per (tile, group), possibly empty
    };
#pragma unroll 1
    for (int f = 0; f < kGSwRing - 1; ++f) fetch_scales(f);
    int ch = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int m = mt * kGTileM + static_cast<int>(rank) * kGHalfM + row;
      const bool mvalid = m < p.M;
      // column j of the accumulator is weight row n0 + j - 32 c4 of the tile
      const int n0 = nt * kGTileN + c4 * 32;
      float fsum[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) fsum[j] = 0.0f;
      for (int g = 0; g < p.G; ++g, ++ch) {
        const int b = ch % kGAccBufs;
        // ch counts this pair's (tile, group) units, the order of the scale stream
        __syncwarp();                         // every lane is done with the slot refilled next
        fetch_scales(ch + kGSwRing - 1);
        cp_async_wait<kGSwRing - 1>();        // this group's scales have landed (own copies)
        __syncwarp();                         // ... and every lane's
        if (!__all_sync(0xffffffffu, mbar_sleep_bounded(accf_bar(b), (ch / kGAccBufs) & 1,
                                                       abort_flag, err, kGWaitNs)))
          goto done;
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + b * kGAccCols + c4 * 32, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acce_leader0 + 8u * b);   // accumulator is in registers
        if (EPI == kEpiY) {
          const float4* w4 = reinterpret_cast<const float4*>(sw_ring_g + (ch % kGSwRing) * 32);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 w = w4[j4];
            fsum[4 * j4 + 0] = fmaf(w.x, __uint_as_float(v[4 * j4 + 0]), fsum[4 * j4 + 0]);
            fsum[4 * j4 + 1] = fmaf(w.y, __uint_as_float(v[4 * j4 + 1]), fsum[4 * j4 + 1]);
            fsum[4 * j4 + 2] = fmaf(w.z, __uint_as_float(v[4 * j4 + 2]), fsum[4 * j4 + 2]);
            fsum[4 * j4 + 3] = fmaf(w.w, __uint_as_float(v[4 * j4 + 3]), fsum[4 * j4 + 3]);
          }
        } else if (mvalid) {
          // exact int32 accumulators [M, N, G]
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = n0 + j;
            if (n < p.N)
              p.acc[(static_cast<int64_t>(m) * p.N + n) * p.G + g] = __float2int_rn(__uint_as_float(v[j]));
          }
        }
      }
      if (EPI == kEpiY && mvalid) {
        const float sam = __ldg(p.sa + m);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int n = n0 + 8 * c;
          if (n < p.N) {   // N % 8 == 0: a group of 8 is all in or all out
            uint32_t hw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half lo = __float2half_rn(__fmul_rn(fsum[8 * c + 2 * i], sam));
              const __half hi = __float2half_rn(__fmul_rn(fsum[8 * c + 2 * i + 1], sam));
              hw[i] = static_cast<uint32_t>(__half_as_ushort(lo)) |
                      (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
            }
            *reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(m) * p.N + n) =
                make_uint4(hw[0], hw[1], hw[2], hw[3]);
          }
        }
      }
    }
  }
done:
  __syncwarp();
  cp_async_wait<0>();   // also after an abort: no copy into shared memory outlives the CTA
  if (warp == 1) {
    // the even CTA's last commit reaches both CTAs; wait for it (bounded, and
    // also after an abort) so no MMA is in flight when the pair frees its
    // tensor memory
    if (lane == 0) {
      volatile uint32_t keep_waiting = 0u;
      mbar_wait_bounded(done_bar, 0, &keep_waiting, err, kGWaitNs);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // neither CTA leaves while the other may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kGTmemCols);
  }
}

// CTA pairs of this kernel that fit on the current device at once, cached per
// device (all instantiations use the same shared memory and threads).
cudaError_t pg_max_clusters(int* out) {
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int nc = dev < 64 ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (nc <= 0) {
    auto kern = gemm_pg_kernel<false, kEpiY>;
    static std::atomic<uint64_t> attr_done{0};
    e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), GCfg<false>::kSmemBytes,
                                attr_done);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(kGThreads, 1, 1);
    cfg.dynamicSmemBytes = GCfg<false>::kSmemBytes;
    int q = 0;
    if (cudaOccupancyMaxActiveClusters(&q, reinterpret_cast<const void*>(kern), &cfg) !=
            cudaSuccess ||
        q <= 0) {
      (void)cudaGetLastError();
      q = sms / 2;
    }
    nc = q;
    if (dev < 64) cached[dev].store(nc, std::memory_order_relaxed);
  }
  *out = nc;
  return cudaSuccess;
}

template <bool INT4, int EPI>
cudaError_t launch_pg(const CUtensorMap& tmX, const CUtensorMap& tmW, const PgArgs& a, int clusters,
                      cudaStream_t st) {
  using C = GCfg<INT4>;
  auto kern = gemm_pg_kernel<INT4, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::kSmemBytes,
                                          attr_done);
  if (e != cudaSuccess) return e;
  kern<<<2 * clusters, kGThreads, C::kSmemBytes, st>>>(tmX, tmW, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_pg(const __half* qa16, const float* sa, int64_t M, int64_t N, int64_t K,
                           const uint8_t* w, bool int4, const float* sw, int group_size, int mode,
                           __half* y, int32_t* acc, cudaStream_t st) {
  if (group_size != 64 && group_size != 128) return cudaErrorInvalidValue;
  CUtensorMap tmX, tmW;
  if (!make_tensor_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qa16, K, M, K * 2, kGSubK,
                          kGHalfM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t wbytes = int4 ? K / 2 : K;
  if (!make_tensor_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, N, wbytes,
                          int4 ? kGSubK / 2 : kGSubK, kGHalfN,
                          int4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  int nc = 0;
  cudaError_t e = pg_max_clusters(&nc);
  if (e != cudaSuccess) return e;
  PgArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.gs = group_size;
  a.G = static_cast<int>(K / group_size);
  a.num_m_tiles = static_cast<int>((M + kGTileM - 1) / kGTileM);
  a.num_tiles = a.num_m_tiles * static_cast<int>((N + kGTileN - 1) / kGTileN);
  a.nkb = static_cast<int>((K + kGBK - 1) / kGBK);
  a.sa = sa;
  a.sw = sw;
  a.y = y;
  a.acc = acc;
  e = device_error_word(&a.err);
  if (e != cudaSuccess) return e;
  const int clusters = a.num_tiles < nc ? a.num_tiles : nc;
  if (int4)
    return mode == kEpiY ? launch_pg<true, kEpiY>(tmX, tmW, a, clusters, st)
                         : launch_pg<true, kEpiAcc>(tmX, tmW, a, clusters, st);
  return mode == kEpiY ? launch_pg<false, kEpiY>(tmX, tmW, a, clusters, st)
                       : launch_pg<false, kEpiAcc>(tmX, tmW, a, clusters, st);
}

}  // namespace cider
