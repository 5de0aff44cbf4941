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
// each accumulator holds one group.
//
// A cluster of two CTAs computes a 256-token x 256-weight-row tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), the per-channel
// kernel's shape: CTA r holds tokens [128 r, 128 r + 128) (A operand, fp16
// codes by TMA) and weight rows [128 r, 128 r + 128) (its half of B,
// converted to fp16 in shared memory).  On GB300 these GEMMs are bound by
// operand delivery from L2 (~10 TB/s measured for plain loads): a 256 x 256
// tile moves 1.5x fewer operand bytes per multiply-add than a 256 x 128 one,
// which measured no faster than a third of the tensor rate whatever its
// epilogue did.
//
// The cost is the drain: every group adds s_w[n,g] * acc_g into a running
// sum per output, 128 tokens x 256 weight rows = 32768 fp32 values per CTA,
// which live in the registers of eight epilogue warps (128 each per thread).
// The register file is split with setmaxnreg: the producer / issuer and
// converter warps give registers up, the epilogue warps take them (the host
// checks the kernel's launch register count covers the split, so the
// increase can never wait).  Two 256-column accumulators alternate between
// consecutive groups: the MMA fills one while the epilogue drains the other.
//
// Roles (16 warps, one CTA per SM, persistent over tiles):
//   warp 0      activation producer: TMA of the CTA's fp16 codes, two
//               [128 m][64 k] sub-tiles per 128-K stage into a 3-stage ring,
//               both CTAs' copies completing on the even CTA's "ready" barrier.
//   warp 1      even CTA only, one thread: per group, waits for a drained
//               accumulator, issues the group's MMAs (8 per 128-K group, 4 per
//               64-K group), commits "accumulator full" to both CTAs; commits
//               "stage free" after each stage.
//   warp 2      weight-code producer: TMA of int8 codes [128 n][64 k] (INT4:
//               packed [128 n][32 B]) into a 3-slot ring.
//   warp 3      weight-scale loader: per group, the tile's 256 scales
//               s_w[n0 .. n0 + 255, g] by cp.async into a 4-group ring (a
//               row's scales sit G * 4 bytes apart in global memory).
//   warps 4-7   converters: thread = weight row, its 128 codes of each stage
//               -> fp16 in the K-major 128-byte-swizzled operand layout, one
//               16-byte chunk at a time; report to the even CTA's "ready"
//               barrier.
//   warps 8-15  epilogue, two per tensor-memory lane quarter (columns 0-127
//               and 128-255): per group, tcgen05.ld of 32 columns at a time,
//               fp32 running sums += s_w * acc_g; at the tile's end
//               y = fp16(s_a * sum) goes out by TMA: the epilogue writes the
//               CTA's 128 x 256 outputs into the tile's last pipeline stage
//               (64 KiB, free once the tile's last MMAs completed; the issuer
//               leaves its "stage free" commit to the epilogue), as four
//               [128 rows][64 columns] boxes with the 128-byte swizzle, one
//               thread stores them with tiled TMA stores and hands the stage
//               back once the stores have read it.  The epilogue then drains
//               the next tile at once: storing y from registers (a warp's
//               store touching 32 rows) had held the running sums, and with
//               them the next tile's third group, for ~9000 cycles per tile.
//               In accumulator mode each group's exact int32 values are
//               stored instead.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kGTile = 256;            // tokens and weight rows per pair tile (MMA M and N)
constexpr int kGHalf = 128;            // rows of each operand per CTA
constexpr int kGSubK = 64;             // K per swizzled sub-tile (128 bytes of fp16)
constexpr int kGSub = 2;               // sub-tiles per stage
constexpr int kGBK = kGSub * kGSubK;   // K per stage
constexpr int kGAccCols = kGTile;
constexpr int kGTmemCols = 2 * kGAccCols;                    // two accumulators
constexpr int kGSubBytes = kGHalf * kGSubK * 2;              // 16 KiB
constexpr int kGOpBytes = kGSub * kGSubBytes;                // 32 KiB
constexpr int kGStageBytes = 2 * kGOpBytes;                  // activations | weights
constexpr int kGStages = 3;
constexpr int kG8Slots = 3;
constexpr int kG8SlotBytes = kGHalf * kGSubK;                // 8 KiB (int8 sub-tile)
constexpr int kGSwSlots = 4;                                 // groups of weight scales in flight
constexpr int kGSwSlotBytes = kGTile * 4;
constexpr int kGMmaWarp = 1;
constexpr int kGW8Warp = 2;
constexpr int kGConvWarp0 = 4;
constexpr int kGEpiWarp0 = 8;
constexpr int kGEpiWarps = 8;
constexpr int kGThreads = 32 * (kGEpiWarp0 + kGEpiWarps);    // 512
// register split per warpgroup (setmaxnreg): producers / issuer / loader and
// converters give registers up, the two epilogue warpgroups take them.  The
// converters convert one 16-byte chunk of codes at a time: a version that
// held a whole 64-code row in registers measured corrupted operands under an
// 80- or 96-register share (and was correct at 128).
constexpr int kGRegsLaunch = 128;
constexpr int kGRegsLow = 56;
constexpr int kGRegsConv = 80;
constexpr int kGRegsEpi = 184;
constexpr int kGRegsNeeded = 128 * kGRegsLow + 128 * kGRegsConv + 256 * kGRegsEpi;
// the even CTA's producer arrival (with both CTAs' activation bytes) + the
// four converter warps of each CTA
constexpr int kGReadyCount = 1 + 4 * 2;
constexpr uint32_t kGReadyBytes = 2 * kGOpBytes;
constexpr uint64_t kGWaitNs = 2000000000ull;

static_assert(kGSubBytes % 1024 == 0, "sub-tiles keep 1024-byte alignment for the swizzle");
static_assert(kGRegsNeeded <= kGThreads * kGRegsLaunch, "register split exceeds the launch's registers");

template <bool INT4>
struct GCfg {
  static constexpr int kA8Bytes = INT4 ? kGHalf * kGSubK / 2 : kGHalf * kGSubK;
  static constexpr int kA8Offset = kGStages * kGStageBytes;
  static constexpr int kSwOffset = kA8Offset + kG8Slots * kG8SlotBytes;
  static constexpr int kBarOffset = kSwOffset + kGSwSlots * kGSwSlotBytes;
  // ready, empty per stage; full8, empty8 per weight slot; swf, swe per
  // scale slot; accf, acce per accumulator; mma_done; y staged; then the
  // tensor-memory slot and the abort flag
  static constexpr int kBar8 = 2 * kGStages;
  static constexpr int kBarSw = kBar8 + 2 * kG8Slots;
  static constexpr int kBarAcc = kBarSw + 2 * kGSwSlots;
  static constexpr int kBarY = kBarAcc + 5;
  static constexpr int kNumBars = kBarY + 1;
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

template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

// Arrive on `bar` once all of this thread's earlier cp.async copies have
// landed (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns (see tmem_ld32).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// BATCH: the converters load a sub-tile's code chunks before converting them
// (their load latencies overlap); measured faster at gs 128 and slower at gs 64
// (where the two drains per stage pace the kernel), so it is chosen by group size.
template <bool INT4, int EPI, bool BATCH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGThreads, 1)
    gemm_pg_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmY, const PgArgs p) {
  using C = GCfg<INT4>;
  constexpr int S = kGStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sA = [&](int s) { return base + s * kGStageBytes; };               // activation codes
  auto sB = [&](int s) { return base + s * kGStageBytes + kGOpBytes; };   // fp16 weights
  auto sW8 = [&](int j) { return base + C::kA8Offset + j * kG8SlotBytes; };
  auto sSw = [&](int j) { return base + C::kSwOffset + j * kGSwSlotBytes; };
  const uint32_t bars = base + C::kBarOffset;
  auto ready_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto full8_bar = [&](int j) { return bars + 8u * (C::kBar8 + j); };
  auto empty8_bar = [&](int j) { return bars + 8u * (C::kBar8 + kG8Slots + j); };
  auto swf_bar = [&](int j) { return bars + 8u * (C::kBarSw + j); };
  auto swe_bar = [&](int j) { return bars + 8u * (C::kBarSw + kGSwSlots + j); };
  auto accf_bar = [&](int b) { return bars + 8u * (C::kBarAcc + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (C::kBarAcc + 2 + b); };
  const uint32_t done_bar = bars + 8u * (C::kBarAcc + 4);
  // a tile's y is staged in shared memory: one arrival per epilogue warp
  const uint32_t ystg_bar = bars + 8u * C::kBarY;
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
      mbar_init(empty8_bar(j), 4);     // the four converter warps
    }
    for (int j = 0; j < kGSwSlots; ++j) {
      mbar_init(swf_bar(j), 32);       // every lane of the loader, once its copies landed
      mbar_init(swe_bar(j), kGEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * kGEpiWarps);   // 8 epilogue warps x 2 CTAs
    }
    mbar_init(done_bar, 1);
    mbar_init(ystg_bar, kGEpiWarps);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  if (warp == kGMmaWarp) {
    tmem_alloc_pair(tmem_slot, kGTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // barriers of both CTAs initialised, tensor memory held
  pdl_wait();   // codes and scales come from the quantization launch just before
  tc_fence_after();
  const uint32_t tmem =
      *reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * C::kNumBars);

  if (warp < kGConvWarp0) {
    regs_dec<kGRegsLow>();
    if (warp == 0) {
      // ---------------------------------------------------------- activation producer
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
              tma_load_2d_pair(sA(s) + t * kGSubBytes, &tmX, ready_leader0 + 8u * s,
                               kb * kGBK + t * kGSubK, mt * kGTile + rank * kGHalf);
          }
        }
      }
    } else if (warp == kGMmaWarp) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      if (rank == 0 && lane == 0) {
        constexpr uint32_t idesc = idesc_f16_f32(kGTile, kGTile);
        int it = 0, ch = 0;
        bool ok = true;
        for (int tile = cid; tile < p.num_tiles && ok; tile += nclusters) {
          for (int kb = 0; kb < p.nkb && ok; ++kb, ++it) {
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
            for (int t = 0; t < ng; ++t, ++ch) {
              const int b = ch & 1;
              if (ch >= 2) {
                // accumulator b was last used by group ch - 2: wait until both CTAs drained it
                if (!mbar_wait_bounded(acce_bar(b), ((ch - 2) >> 1) & 1, abort_flag, err,
                                       kGWaitNs)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              const uint32_t d = tmem + b * kGAccCols;
              if (gpk == 1) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const uint64_t off =
                      static_cast<uint64_t>((j >> 2) * (kGSubBytes >> 4) + (j & 3) * 2);
                  tc_mma_ss_pair(d, adesc + off, bdesc + off, idesc, j == 0 ? 0u : 1u);
                }
              } else {
                // a 64-K group: sub-tile t of the stage
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint64_t off = static_cast<uint64_t>(t * (kGSubBytes >> 4) + j * 2);
                  tc_mma_ss_pair(d, adesc + off, bdesc + off, idesc, j == 0 ? 0u : 1u);
                }
              }
              tc_commit_pair_mc(accf_bar(b), 0x3);
            }
            if (!ok) break;
            // a tile's last stage is handed back by the epilogue, which stages y in it
            if (EPI == kEpiAcc || kb != p.nkb - 1) tc_commit_pair_mc(empty_bar(s), 0x3);
          }
        }
        if (!ok) *abort_flag = 1u;
        // every MMA issued so far completes before either CTA frees tensor memory
        tc_commit_pair_mc(done_bar, 0x3);
      }
      __syncwarp();
    } else if (warp == kGW8Warp) {
      // ---------------------------------------------------------- weight-code producer
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
                          nt * kGTile + rank * kGHalf);
            }
        }
      }
    } else if (EPI != kEpiAcc) {
      // ---------------------------------------------------------- weight-scale loader
      int f = 0;   // (tile, group) units of this pair, in drain order
      for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
        const int n0 = (tile / p.num_m_tiles) * kGTile;
        for (int g = 0; g < p.G; ++g, ++f) {
          const int j = f % kGSwSlots;
          const uint32_t ph = (f / kGSwSlots) & 1;
          if (!__all_sync(0xffffffffu, mbar_sleep_bounded(swe_bar(j), ph ^ 1u, abort_flag, err,
                                                           kGWaitNs)))
            goto done;
#pragma unroll
          for (int i = 0; i < kGTile / 32; ++i) {
            const int n = n0 + i * 32 + lane;
            cp_async4(sSw(j) + (i * 32 + lane) * 4,
                      p.sw + (n < p.N ? static_cast<int64_t>(n) * p.G + g : 0), n < p.N);
          }
          cp_async_arrive_noinc(swf_bar(j));
        }
      }
    }
  } else if (warp < kGEpiWarp0) {
    regs_dec<kGRegsConv>();
    // ------------------------------------------------------------ converters
    const int row = (warp - kGConvWarp0) * 32 + lane;   // weight row within the CTA's 128
    const uint32_t ready_leader0 = mapa_shared(ready_bar(0), 0);
    int it = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters) {
      for (int kb = 0; kb < p.nkb; ++kb, ++it) {
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
          const uint8_t* arow = gbase + (sW8(j8) - base);
          // the stage's weight operand is free once the MMAs of its previous use completed
          if (t == 0 && !__all_sync(0xffffffffu, mbar_sleep_bounded(empty_bar(s), ph ^ 1u,
                                                                   abort_flag, err, kGWaitNs)))
            goto done;
          if (!INT4) {
            // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3);
            // its 16 codes become fp16 chunks 2c and 2c + 1 of the 128-byte row
            uint4 vin[4];
            if (BATCH) {
#pragma unroll
              for (int c = 0; c < 4; ++c)
                vin[c] = *reinterpret_cast<const uint4*>(arow + row * 64 +
                                                         ((c ^ ((row >> 1) & 3)) << 4));
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 v = BATCH ? vin[c]
                                    : *reinterpret_cast<const uint4*>(
                                          arow + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
              uint32_t h[8];
              s8x4_to_h2x2(v.x, h[0], h[1]);
              s8x4_to_h2x2(v.y, h[2], h[3]);
              s8x4_to_h2x2(v.z, h[4], h[5]);
              s8x4_to_h2x2(v.w, h[6], h[7]);
              *reinterpret_cast<uint4*>(drow + t * kGSubBytes + (((2 * c) ^ (row & 7)) << 4)) =
                  make_uint4(h[0], h[1], h[2], h[3]);
              *reinterpret_cast<uint4*>(drow + t * kGSubBytes + (((2 * c + 1) ^ (row & 7)) << 4)) =
                  make_uint4(h[4], h[5], h[6], h[7]);
            }
          } else {
            // 32-byte swizzle: chunk c of row r sits at chunk c ^ ((r >> 2) & 1); its 32
            // codes become fp16 chunks 4c .. 4c + 3
            uint4 vin[2];
            if (BATCH) {
#pragma unroll
              for (int c = 0; c < 2; ++c)
                vin[c] = *reinterpret_cast<const uint4*>(arow + row * 32 +
                                                         ((c ^ ((row >> 2) & 1)) << 4));
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint4 v = BATCH ? vin[c]
                                    : *reinterpret_cast<const uint4*>(
                                          arow + row * 32 + ((c ^ ((row >> 2) & 1)) << 4));
              const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t tt[4];
                s4x8_to_h2x4(vw[q4], tt);
                *reinterpret_cast<uint4*>(drow + t * kGSubBytes + (((4 * c + q4) ^ (row & 7)) << 4)) =
                    make_uint4(tt[0], tt[1], tt[2], tt[3]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty8_bar(j8));   // weight slot consumed
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(ready_leader0 + 8u * s);
      }
    }
  } else {
    regs_inc<kGRegsEpi>();
    // ------------------------------------------------------------ epilogue
    const int e = warp - kGEpiWarp0;          // 0..7
    const int q = warp & 3;                   // tensor-memory lane quarter of this warp
    const int hcol = e >> 2;                  // accumulator columns [128 hcol, 128 hcol + 128)
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const int row = q * 32 + lane;            // token of this thread within the CTA's 128
    int ch = 0, tcount = 0;
    for (int tile = cid; tile < p.num_tiles; tile += nclusters, ++tcount) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int m = mt * kGTile + static_cast<int>(rank) * kGHalf + row;
      const bool mvalid = m < p.M;
      // column j of this warp's 128 is weight row n0 + j of the tile
      const int n0 = nt * kGTile + hcol * 128;
      float fsum[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) fsum[j] = 0.0f;
      for (int g = 0; g < p.G; ++g, ++ch) {
        const int b = ch & 1;
        const int js = ch % kGSwSlots;
        if (EPI != kEpiAcc && !__all_sync(0xffffffffu, mbar_sleep_bounded(
                                                         swf_bar(js), (ch / kGSwSlots) & 1,
                                                         abort_flag, err, kGWaitNs)))
          goto done;
        if (!__all_sync(0xffffffffu, mbar_sleep_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag,
                                                       err, kGWaitNs)))
          goto done;
        tc_fence_after();
        const uint32_t tsrc = tmem + lane_base + b * kGAccCols + hcol * 128;
        const float4* w4 =
            reinterpret_cast<const float4*>(gbase + C::kSwOffset + js * kGSwSlotBytes) + hcol * 32;
        // 32 columns per round: two 16-column loads, then their wait, before
        // any use (tcgen05.ld writes its registers asynchronously; nothing may
        // touch them until tcgen05.wait::ld)
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
          uint32_t v[2][16];
          tmem_ld16(tsrc + c2 * 32, v[0]);
          tmem_ld16(tsrc + c2 * 32 + 16, v[1]);
          tmem_wait_ld();
          if (c2 == 3) {
            // the last columns are in registers: the accumulator is free for group ch + 2
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acce_leader0 + 8u * b);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int c = 2 * c2 + hh;   // 16-column chunk of the warp's 128
            if (EPI != kEpiAcc) {
#pragma unroll
              for (int j4 = 0; j4 < 4; ++j4) {
                const float4 w = w4[c * 4 + j4];
                const uint32_t* vv = v[hh] + 4 * j4;
                float* fs = fsum + c * 16 + 4 * j4;
                fs[0] = fmaf(w.x, __uint_as_float(vv[0]), fs[0]);
                fs[1] = fmaf(w.y, __uint_as_float(vv[1]), fs[1]);
                fs[2] = fmaf(w.z, __uint_as_float(vv[2]), fs[2]);
                fs[3] = fmaf(w.w, __uint_as_float(vv[3]), fs[3]);
              }
            } else if (mvalid) {
              // exact int32 accumulators [M, N, G]
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = n0 + c * 16 + j;
                if (n < p.N)
                  p.acc[(static_cast<int64_t>(m) * p.N + n) * p.G + g] =
                      __float2int_rn(__uint_as_float(v[hh][j]));
              }
            }
          }
        }
        if (EPI != kEpiAcc) {
          __syncwarp();
          if (lane == 0) mbar_arrive(swe_bar(js));   // this warp is done with the slot's scales
        }
      }
      if (EPI != kEpiAcc) {
        // y of this CTA's 128 tokens x the tile's 256 columns, staged in the
        // tile's last pipeline stage: block j (columns [64 j, 64 j + 64)) is
        // [128 rows][128 bytes] at 16 KiB j, 16-byte chunk c of row r at chunk
        // c ^ (r & 7) (the TMA 128-byte swizzle)
        const int s_last = (tcount * p.nkb + p.nkb - 1) % S;
        const uint32_t ybuf = sA(s_last);
        const float sam = mvalid ? __ldg(p.sa + m) : 0.0f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {   // outputs 128 hcol + 8 c ... + 7 of the tile
          uint32_t hw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            hw[i] = y_bits2<EPI == kEpiYb>(__fmul_rn(fsum[8 * c + 2 * i], sam),
                                           __fmul_rn(fsum[8 * c + 2 * i + 1], sam));
          const int blk = 2 * hcol + (c >> 3), cc = c & 7;
          st_shared_v4(ybuf + blk * 16384 + row * 128 + ((cc ^ (row & 7)) << 4), hw);
        }
        fence_proxy_async_smem();   // the TMA engine reads what these threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(ystg_bar);
        // the first epilogue warp waits for all eight warps' parts and one of
        // its threads stores them; the other warps go on to the next tile
        if (e == 0) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(ystg_bar, tcount & 1, abort_flag, err,
                                                          kGWaitNs)))
            goto done;
          if (lane == 0) {
            const int m0 = mt * kGTile + static_cast<int>(rank) * kGHalf;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_store_2d(&tmY, ybuf + j * 16384, nt * kGTile + 64 * j, m0);
            bulk_commit_group();
            bulk_wait_group_read<0>();   // the stage may be refilled once the stores have read it
            mbar_arrive(empty_bar(s_last));
          }
          __syncwarp();
        }
      }
    }
  }
done:
  __syncwarp();
  cp_async_wait<0>();   // also after an abort: no copy into shared memory outlives the CTA
  if (EPI != kEpiAcc && warp == kGEpiWarp0 && lane == 0) bulk_wait_group<0>();   // y stores written
  if (warp == kGMmaWarp) {
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
  if (warp == kGMmaWarp) {
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
    auto kern = gemm_pg_kernel<false, kEpiY, true>;
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

// after_quant: may start before this library's quantization launch just
// before it ends (programmatic dependent launch; the kernel waits for it).
template <bool INT4, int EPI, bool BATCH>
cudaError_t launch_pg(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmY,
                      const PgArgs& a, int clusters, cudaStream_t st, bool after_quant) {
  using C = GCfg<INT4>;
  auto kern = gemm_pg_kernel<INT4, EPI, BATCH>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::kSmemBytes,
                                          attr_done);
  if (e != cudaSuccess) return e;
  // The warps' register increase (setmaxnreg) draws on the registers the CTA
  // was launched with; refuse a build whose launch count cannot cover the
  // split rather than launch a kernel whose increase would wait forever.
  static std::atomic<int> regs_ok{0};
  if (regs_ok.load(std::memory_order_relaxed) == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
    regs_ok.store(fa.numRegs * kGThreads >= kGRegsNeeded ? 1 : -1, std::memory_order_relaxed);
  }
  if (regs_ok.load(std::memory_order_relaxed) < 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kGThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_quant ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, tmY, a);
}

}  // namespace

cudaError_t launch_gemm_pg(const __half* qa16, const float* sa, int64_t M, int64_t N, int64_t K,
                           const uint8_t* w, bool int4, const float* sw, int group_size, int mode,
                           __half* y, int32_t* acc, cudaStream_t st, bool after_quant) {
  if (group_size != 64 && group_size != 128) return cudaErrorInvalidValue;
  CUtensorMap tmX, tmW;
  if (!make_tensor_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qa16, K, M, K * 2, kGSubK, kGHalf,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t wbytes = int4 ? K / 2 : K;
  if (!make_tensor_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, N, wbytes,
                          int4 ? kGSubK / 2 : kGSubK, kGHalf,
                          int4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  // y [M, N] of 2-byte outputs (fp16 or bf16 bits), stored in [128 rows][64 columns] boxes; in
  // accumulator mode the map is not used (a valid one over the weights is passed instead)
  CUtensorMap tmY;
  if (mode != kEpiAcc ? !make_tensor_map_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_UINT16, y, N, M, N * 2, 64,
                                            kGHalf, CU_TENSOR_MAP_SWIZZLE_128B)
                      : !make_tensor_map_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, N, wbytes,
                                            16, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
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
  a.num_m_tiles = static_cast<int>((M + kGTile - 1) / kGTile);
  a.num_tiles = a.num_m_tiles * static_cast<int>((N + kGTile - 1) / kGTile);
  a.nkb = static_cast<int>((K + kGBK - 1) / kGBK);
  a.sa = sa;
  a.sw = sw;
  a.y = y;
  a.acc = acc;
  e = device_error_word(&a.err);
  if (e != cudaSuccess) return e;
  const int clusters = a.num_tiles < nc ? a.num_tiles : nc;
#define CIDER_PG_LAUNCH(I4, B)                                                               \
  return mode == kEpiY    ? launch_pg<I4, kEpiY, B>(tmX, tmW, tmY, a, clusters, st, after_quant)          \
         : mode == kEpiYb ? launch_pg<I4, kEpiYb, B>(tmX, tmW, tmY, a, clusters, st, after_quant)         \
                          : launch_pg<I4, kEpiAcc, B>(tmX, tmW, tmY, a, clusters, st, after_quant);
  if (int4) {
    if (group_size == 128) CIDER_PG_LAUNCH(true, true)
    CIDER_PG_LAUNCH(true, false)
  }
  if (group_size == 128) CIDER_PG_LAUNCH(false, true)
  CIDER_PG_LAUNCH(false, false)
#undef CIDER_PG_LAUNCH
}

}  // namespace cider
