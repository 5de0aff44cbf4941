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
// 256 tokens (m) x 256 weight rows (n), with tcgen05.mma.cta_group::2:
// CTA r of the pair holds tokens [128 r, 128 r + 128) of the tile (the MMA's
// A operand, M = 256 split over the pair) and weight rows [128 r, 128 r + 128)
// (its half of the B operand, N = 256); each CTA's tensor memory receives its
// own 128 tokens (one per lane) x all 256 weight rows.  Per SM this halves
// the operand bytes read per multiply-add compared with a 128 x 256 tile on
// one SM, which is what lets the tensor pipe run at its full rate.
//
// The weight operand (fp16, K-major, 128-byte swizzle) is made in shared
// memory by converter warps from the int8 / int4 codes of each stage.
// (Converting all weights to fp16 in global memory first and feeding both
// operands by TMA makes the GEMM itself ~4 % faster on GB300, but the extra
// streaming pass costs more than that at every measured shape.)
//
// Roles in each CTA (one CTA per SM, persistent over tiles):
//   warp 0      producer: TMA of the CTA's activation codes (fp16, two
//               [128 m][64 k] sub-tiles per 128-K stage) into the 3-stage
//               operand ring; the copies of both CTAs complete on the even
//               CTA's "ready" barrier.
//   warps 1, 15 the two MMA issuers, even CTA only, one thread each, taking
//               alternate stages: wait until both CTAs' stage is ready, issue
//               8 MMAs (K = 16 each) into one of two 256-column accumulators
//               and commit to both CTAs' barriers (stage free; accumulator
//               full).  A token passed between them keeps the MMAs in stage
//               order.  One thread alone needed ~1300 cycles per stage for its
//               chain of waits, fences, commits and MMA issues (~75 cycles
//               each), more than the stage's 1024 cycles of MMAs.  Both CTAs'
//               warp 1 allocate tensor memory.  128-K stages halve the
//               per-stage synchronisation cost, which with 64-K stages kept
//               the tensor pipe ~30 % idle.
//   warps 10-13 epilogue, one per tensor-memory lane quarter: drain the
//               accumulator (tcgen05.ld: a thread holds 32 consecutive weight
//               rows of its token), release it once the last columns are in
//               registers, dequantize, store fp16 y (32-byte stores when rows
//               start 32-byte aligned, else 16-byte ones; a warp's store
//               touches 32 rows) or int32 accumulators.
//   converters  two groups of 4 warps (warps 2-9) taking alternate stages:
//               each thread converts its weight row's 128 codes of the stage
//               (two 64-K sub-tiles) and writes them in the canonical K-major
//               swizzled layout, then reports to the even CTA's "ready"
//               barrier.
//   warp 14     weight-code producer: TMA of the int8 codes [128 n][64 k] (INT4:
//               packed [128 n][32 B]) into a separate 4-slot ring, one
//               sub-tile per slot, running ahead of the conversion.
//
// Work split: with P pairs, whole tiles are dealt round-robin for
// floor(tiles / P) rounds.  When the remaining r tiles would leave most pairs
// idle in a last round, each of them is cut along K into s = floor(P / r)
// equal pieces (at least four 128-K blocks each) on s pairs: 640 tiles on 76
// pairs run as 8 whole rounds plus 32 tiles in 2 halves on 64 pairs, instead
// of 9 rounds.  A piece's accumulator is an exact integer (the per-tile bound
// below holds for any part of K).  Each pair stores it as int32 into its own
// workspace slot, in a layout where the 32 lanes of a warp touch 512
// consecutive bytes, and raises its slot's flag; it then waits for the flags
// of the tile's other pieces, adds up all s partials for its own 1/s of the
// tile's weight rows (exact int32) and dequantizes and stores that part of
// y.  Every pair writes before it waits, so the waits cannot cycle; the
// pieces of a tile run at the same time on co-resident pairs: such a launch
// is cooperative (all pairs resident at once, or the launch fails) and never
// exceeds the pairs the GPU holds at once.  The flags are zeroed by the
// activation-quantization kernel that precedes every launch.  The exchange
// pairs CTAs of equal rank, so a CTA whose 128 token rows all lie past M
// (the second CTA of every pair at M <= 128) skips it, as do its peers.
// The launch is a programmatic dependent of that quantization kernel: it
// sets up barriers and tensor memory, then waits for the kernel's results.
//
// Exactness per tile: every partial sum of token m is bounded by
// qmax_w * sum_k |q_a[m,k]| (qmax_w = 127 INT8, 8 INT4).  When that bound is
// <= 2^23 for all 256 tokens of the tile ("fast" tile, the normal case) all of
// K accumulates in fp32 exactly and the accumulator is drained once.  Else
// ("slow" tile) the tile runs as four passes of 64 weight rows (N = 64 MMAs,
// 32 rows from each CTA) whose accumulators are drained every 512 K into
// exact int32 register sums.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kPTileM = 256;          // tokens per pair tile (MMA M, tensor-memory lanes)
constexpr int kPTileN = 256;          // weight rows per pair tile (MMA N)
constexpr int kPHalf = 128;           // rows of each operand per CTA
constexpr int kPSubK = 64;            // K per swizzled sub-tile (128 bytes of fp16)
constexpr int kPSub = 2;              // sub-tiles per pipeline stage
constexpr int kPBK = kPSub * kPSubK;  // K per pipeline stage: 8 MMAs
constexpr int kPUmmaK = 16;
constexpr int kPChunkKB = 4;          // slow tiles: drain every 512 K
constexpr int kPSlowPasses = 4;       // slow tiles: 64 weight rows per pass
constexpr int kPAccCols = 256;
constexpr int kPTmemCols = 512;
constexpr int kPSubBytes = kPHalf * kPSubK * 2;  // 16 KiB: one operand sub-tile, fp16
constexpr int kPOpBytes = kPSub * kPSubBytes;    // 32 KiB: one operand of a stage
constexpr int kPStageBytes = 2 * kPOpBytes;      // activations | weights
constexpr int kP8Slots = 4;                      // int8 / int4 weight ring, one sub-tile per slot
constexpr int kPStages = 3;
constexpr int kPConvWarp0 = 2;                   // two groups of 4 converter warps
constexpr int kPEpiWarp0 = 10;
constexpr int kPW8Warp = 14;
constexpr int kPMma2Warp = 15;                   // the second MMA issuer
constexpr int kPThreads = 32 * (kPMma2Warp + 1);
// the even CTA's producer arrival (with both CTAs' activation bytes) + 4
// converter warps x 2 CTAs
constexpr int kPReadyCount = 9;
constexpr uint32_t kPReadyBytes = 2 * kPOpBytes;
constexpr uint64_t kPWaitNs = 2000000000ull;

template <bool INT4>
struct PCfg {
  static constexpr int kA8Bytes = INT4 ? kPHalf * kPSubK / 2 : kPHalf * kPSubK;
  static constexpr int kA8Offset = kPStages * kPStageBytes;
  static constexpr int kBarOffset = kA8Offset + kP8Slots * 8192;
  // ready, empty per stage; full8, empty8 per weight slot; accf x2, acce x2,
  // mma_done; the issuers' turn tokens; the pieces' partials copied in; then
  // the tensor-memory slot and the abort flag
  static constexpr int kBar8 = 2 * kPStages;
  static constexpr int kBar2 = kBar8 + 2 * kP8Slots;
  static constexpr int kBarTok = kBar2 + 5;       // the issuers' turn tokens
  static constexpr int kBarRed = kBarTok + 2;     // a cut tile's partials are in shared memory
  static constexpr int kNumBars = kBarRed + 1;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};
static_assert(kPSubBytes % 1024 == 0, "sub-tiles must keep 1024-byte alignment for the swizzle");

struct PairArgs {
  int M, N, K;
  int num_m_tiles, num_tiles;
  int nkb;          // 128-K blocks per tile
  int full_tiles;   // tiles [0, full_tiles) are dealt whole, round-robin over the pairs
  int sk_tiles;     // tiles [full_tiles, full_tiles + sk_tiles) are cut into pieces
  int sk_split;     // s: pieces per cut tile; pair c < sk_tiles * s takes piece c % s of tile c / s
  int4* part;       // partials [pair][2 CTAs][64 x 16-byte column groups][128 tokens]
  int* flags;       // [pair][2 CTAs][4 lane quarters], zero at launch
  const float* sa;
  const float* sw;
  __half* y;
  int32_t* acc;
  const int* row_l1;
  int l1_limit;
  int* err;
};

// One unit of a pair's work: blocks [kb0, kb1) of a tile.
enum : int {
  kUnitWhole = 0,   // the whole tile: dequantize and store
  kUnitPiece = 1,   // piece kb0..kb1 of a cut tile: store the partial, then reduce a 1/s slice
};
struct PUnit {
  int tile, kb0, kb1, kind;
};

__host__ __device__ __forceinline__ int pair_whole_units(const PairArgs& p, int c, int P) {
  return c < p.full_tiles ? (p.full_tiles - 1 - c) / P + 1 : 0;
}

// Number of units of pair c (of P), and the i-th of them.  Every role of
// both CTAs walks the same sequence.
__host__ __device__ __forceinline__ int pair_num_units(const PairArgs& p, int c, int P) {
  return pair_whole_units(p, c, P) + (c < p.sk_tiles * p.sk_split ? 1 : 0);
}

__host__ __device__ __forceinline__ PUnit pair_unit(const PairArgs& p, int c, int P, int i) {
  if (i < pair_whole_units(p, c, P)) return PUnit{c + i * P, 0, p.nkb, kUnitWhole};
  const int k = c % p.sk_split;
  return PUnit{p.full_tiles + c / p.sk_split, k * p.nkb / p.sk_split, (k + 1) * p.nkb / p.sk_split,
               kUnitPiece};
}

// 16-byte column groups [j0, j1) of the tile (4 weight rows each, in pairs so
// that groups of 8 outputs stay whole) that piece k of s reduces and stores.
__host__ __device__ __forceinline__ void piece_slice(int k, int s, int* j0, int* j1) {
  *j0 = 2 * ((32 * k) / s);
  *j1 = 2 * ((32 * (k + 1)) / s);
}

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

// y[m, n0 .. n0 + 7] = round((acc * s_a[m]) * s_w[n]) to fp16 (or bf16) from
// eight exact accumulator values and the eight weight scales, one 16-byte store.
template <bool BF16>
__device__ __forceinline__ void store8_y(const PairArgs& p, int m, float sam, int n0, const float* f,
                                         const float (&w)[8]) {
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    h[i] = y_bits2<BF16>(__fmul_rn(__fmul_rn(f[2 * i], sam), w[2 * i]),
                         __fmul_rn(__fmul_rn(f[2 * i + 1], sam), w[2 * i + 1]));
  *reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(m) * p.N + n0) =
      make_uint4(h[0], h[1], h[2], h[3]);
}

// The same for sixteen outputs n0 .. n0 + 15 with one 32-byte store (the
// address must be 32-byte aligned).  A lane's stores go to its own token's
// row, so a warp's store touches 32 rows: wider stores halve the requests.
template <bool BF16>
__device__ __forceinline__ void store16_y(const PairArgs& p, int m, float sam, int n0,
                                          const float (&f)[16], const float (&w)[16]) {
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    h[i] = y_bits2<BF16>(__fmul_rn(__fmul_rn(f[2 * i], sam), w[2 * i]),
                         __fmul_rn(__fmul_rn(f[2 * i + 1], sam), w[2 * i + 1]));
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(
                   p.y + static_cast<int64_t>(m) * p.N + n0),
               "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]), "r"(h[4]), "r"(h[5]), "r"(h[6]),
               "r"(h[7])
               : "memory");
}

template <bool INT4, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const PairArgs p) {
  using C = PCfg<INT4>;
  constexpr int S = kPStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto sA = [&](int s) { return base + s * kPStageBytes; };               // activation codes
  auto sB = [&](int s) { return base + s * kPStageBytes + kPOpBytes; };   // fp16 weights
  auto sW8 = [&](int j) { return base + C::kA8Offset + j * 8192; };
  const uint32_t bars = base + C::kBarOffset;
  auto ready_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto full8_bar = [&](int j) { return bars + 8u * (C::kBar8 + j); };
  auto empty8_bar = [&](int j) { return bars + 8u * (C::kBar8 + kP8Slots + j); };
  auto accf_bar = [&](int b) { return bars + 8u * (C::kBar2 + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (C::kBar2 + 2 + b); };
  const uint32_t done_bar = bars + 8u * (C::kBar2 + 4);
  // turn token of issuer b: completes once per stage the other issuer has issued
  auto tok_bar = [&](int b) { return bars + 8u * (C::kBarTok + b); };
  const uint32_t red_bar = bars + 8u * C::kBarRed;
  const uint32_t tmem_slot = bars + 8u * C::kNumBars;
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * C::kNumBars + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  int* err = p.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(ready_bar(s), kPReadyCount);
      mbar_init(empty_bar(s), 1);
    }
    for (int j = 0; j < kP8Slots; ++j) {
      mbar_init(full8_bar(j), 1);
      mbar_init(empty8_bar(j), 4);     // the 4 warps of the converter group of this use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 2);       // both issuers, each after its own MMAs of the chunk
      mbar_init(acce_bar(b), 8);       // 4 epilogue warps x 2 CTAs
    }
    mbar_init(done_bar, 2);
    mbar_init(tok_bar(0), 1);
    mbar_init(tok_bar(1), 1);
    mbar_init(red_bar, 4);   // one arrival per epilogue warp
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // barriers of both CTAs initialised, tensor memory held
  tc_fence_after();
  pdl_wait();   // codes, scales and flags come from the quantization launch just before
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOffset + 8 * C::kNumBars);
  const int nu = pair_num_units(p, cid, nclusters);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint32_t ready_leader0 = mapa_shared(ready_bar(0), 0);
    int it = 0;
    for (int ui = 0; ui < nu; ++ui) {
      const PUnit u = pair_unit(p, cid, nclusters, ui);
      const int tile = u.tile, kb0 = u.kb0, kb1 = u.kb1;
      const int mt = tile % p.num_m_tiles;
      const int passes = pair_tile_fast(p, mt, lane) ? 1 : kPSlowPasses;
      if (lane == 0) {
        for (int pass = 0; pass < passes; ++pass)
          for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % S;
            const uint32_t ph = (it / S) & 1;
            if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kPWaitNs)) break;
            if (rank == 0) mbar_arrive_expect_tx(ready_bar(s), kPReadyBytes);
            for (int t = 0; t < kPSub; ++t) {
              const int k0 = kb * kPBK + t * kPSubK;
              tma_load_2d_pair(sA(s) + t * kPSubBytes, &tmX, ready_leader0 + 8u * s, k0,
                               mt * kPTileM + rank * kPHalf);
            }
          }
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else if (warp == 1 || warp == kPMma2Warp) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    // Issuer me (warp 1: 0, warp 15: 1) issues the stages with it % 2 == me.
    // A lone issuer needed ~1300 cycles per stage for its chain of barrier
    // waits, fences, commits and eight MMA issues (~75 cycles each), against
    // 1024 cycles of tensor-core work; two issuers overlap their chains.  The
    // MMAs still reach the tensor core in stage order: before issuing stage
    // it an issuer waits for its token, which the other issuer gives once it
    // has issued stage it - 1.  Both issuers pass every stage's "ready"
    // barrier in order (so no parity wait can be satisfied by an older phase)
    // and both commit "accumulator full" at the end of every chunk, each
    // after its own MMAs of the chunk (the barrier counts two arrivals).
    const int me = warp == 1 ? 0 : 1;
    if (rank == 0) {
      constexpr uint32_t idesc_fast = idesc_f16_f32(kPTileM, kPTileN);
      constexpr uint32_t idesc_slow = idesc_f16_f32(kPTileM, kPTileN / kPSlowPasses);
      int it = 0, ch = 0;
      for (int ui = 0; ui < nu; ++ui) {
        const PUnit u = pair_unit(p, cid, nclusters, ui);
        const int tile = u.tile, kb0 = u.kb0, kb1 = u.kb1;
        const int mt = tile % p.num_m_tiles;
        const bool fast = pair_tile_fast(p, mt, lane);
        if (lane == 0) {
          const int passes = fast ? 1 : kPSlowPasses;
          bool ok = true;
          for (int pass = 0; pass < passes && ok; ++pass) {
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
              const int kr = kb - kb0;
              const bool cstart = fast ? (kr == 0) : (kr % kPChunkKB) == 0;
              const bool cend =
                  fast ? (kb == kb1 - 1) : ((kr % kPChunkKB) == kPChunkKB - 1 || kb == kb1 - 1);
              const int b = ch & 1;
              const int s = it % S;
              const uint32_t ph = (it / S) & 1;
              if (!mbar_wait_bounded(ready_bar(s), ph, abort_flag, err, kPWaitNs)) {
                ok = false;
                break;
              }
              if ((it & 1) == me) {
                // accumulator b was last used by chunk ch - 2: wait until both CTAs drained it
                if (cstart && ch >= 2 &&
                    !mbar_wait_bounded(acce_bar(b), ((ch - 2) >> 1) & 1, abort_flag, err, kPWaitNs)) {
                  ok = false;
                  break;
                }
                // stage it - 1 is the other issuer's ((it - 1) >> 1)-th
                if (it >= 1 &&
                    !mbar_wait_bounded(tok_bar(me), ((it - 1) >> 1) & 1, abort_flag, err, kPWaitNs)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t adesc = smem_desc_k_sw128(sA(s));
                // slow pass p uses weight rows [32 p, 32 p + 32) of each CTA's 128
                const uint64_t bdesc = smem_desc_k_sw128(sB(s) + (fast ? 0 : pass * (32 * 128)));
#pragma unroll
                for (int j = 0; j < kPBK / kPUmmaK; ++j) {
                  // sub-tile j / 4, K step j % 4 (+32 bytes each) inside it
                  const uint64_t off =
                      static_cast<uint64_t>((j >> 2) * (kPSubBytes >> 4) + (j & 3) * 2);
                  tc_mma_ss_pair(tmem + b * kPAccCols, adesc + off, bdesc + off,
                                 fast ? idesc_fast : idesc_slow, (cstart && j == 0) ? 0u : 1u);
                }
                mbar_arrive(tok_bar(me ^ 1));   // the other issuer may issue stage it + 1
                tc_commit_pair_mc(empty_bar(s), 0x3);
              }
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
    for (int ui = 0; ui < nu; ++ui) {
      const PUnit u = pair_unit(p, cid, nclusters, ui);
      const int tile = u.tile, kb0 = u.kb0, kb1 = u.kb1;
      const int mt = tile % p.num_m_tiles;
      const int passes = pair_tile_fast(p, mt, lane) ? 1 : kPSlowPasses;
      for (int pass = 0; pass < passes; ++pass) {
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if ((it & 1) != group) continue;
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          uint8_t* drow = gbase + (sB(s) - base) + row * 128;
#pragma unroll 1
          for (int t = 0; t < kPSub; ++t) {
            const int v8 = it * kPSub + t;   // weight sub-tile index
            const int j8 = v8 % kP8Slots;
            const uint32_t ph8 = (v8 / kP8Slots) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(full8_bar(j8), ph8, abort_flag, err,
                                                           kPWaitNs)))
              goto done;
            uint32_t h[32];
            const uint8_t* arow = gbase + (sW8(j8) - base);
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
            if (t == 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(empty_bar(s), ph ^ 1u,
                                                                     abort_flag, err, kPWaitNs)))
              goto done;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(drow + t * kPSubBytes + ((c ^ (row & 7)) << 4)) =
                  make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(ready_leader0 + 8u * s);
        }
      }
    }
  } else if (warp == kPW8Warp) {
    // ------------------------------------------------------------ weight-code producer
    int it = 0;
    for (int ui = 0; ui < nu; ++ui) {
      const PUnit u = pair_unit(p, cid, nclusters, ui);
      const int tile = u.tile, kb0 = u.kb0, kb1 = u.kb1;
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const int passes = pair_tile_fast(p, mt, lane) ? 1 : kPSlowPasses;
      if (lane == 0) {
        bool ok = true;
        for (int pass = 0; pass < passes && ok; ++pass)
          for (int kb = kb0; kb < kb1 && ok; ++kb)
            for (int t = 0; t < kPSub; ++t, ++it) {
              const int j = it % kP8Slots;
              const uint32_t ph = (it / kP8Slots) & 1;
              if (!mbar_wait_bounded(empty8_bar(j), ph ^ 1u, abort_flag, err, kPWaitNs)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(full8_bar(j), C::kA8Bytes);
              const int k0 = kb * kPBK + t * kPSubK;
              tma_load_2d(sW8(j), &tmW, full8_bar(j), INT4 ? k0 / 2 : k0,
                          nt * kPTileN + rank * kPHalf);
            }
      }
      __syncwarp();
      if (*abort_flag) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // tensor-memory lane quarter of this warp
    // y rows start 32-byte aligned: sixteen outputs per store
    const bool y_wide = (reinterpret_cast<uintptr_t>(p.y) % 32 == 0) && (p.N % 16 == 0);
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    int ch = 0;
    for (int ui = 0; ui < nu; ++ui) {
      const PUnit u = pair_unit(p, cid, nclusters, ui);
      const int tile = u.tile, kb0 = u.kb0, kb1 = u.kb1;
      const int nch = (kb1 - kb0 + kPChunkKB - 1) / kPChunkKB;
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      const bool fast = pair_tile_fast(p, mt, lane);
      const int row = q * 32 + lane;   // token of this thread within the CTA's 128
      const int m = mt * kPTileM + static_cast<int>(rank) * kPHalf + row;
      const bool mvalid = m < p.M;
      const float sam = (EPI != kEpiAcc && mvalid) ? __ldg(p.sa + m) : 0.0f;
      const int n_tile = nt * kPTileN;
      const bool piece = u.kind == kUnitPiece;
      // partial slot of a pair: 16-byte column group j of this thread's token
      // row at [j][row], so that a warp's lanes touch consecutive 16 bytes
      auto slot = [&](int pair) {
        return p.part + (static_cast<int64_t>(pair) * 2 + rank) * (kPTileN / 4) * kPHalf + row;
      };
      // The tile's 256 weight scales, 8 per lane (lane l: weight rows 8 l ..
      // 8 l + 7), handed to the lanes that need them by shuffles: every lane
      // uses all 256 scales, and loading each one per lane from the cache
      // made the epilogue the slower half of the pipeline.
      float swr[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int n = n_tile + lane * 8 + i;
        swr[i] = (EPI != kEpiAcc && n < p.N) ? __ldg(p.sw + n) : 0.0f;
      }
      // scales of tile columns col .. col + 7 (col % 8 == 0); the whole warp calls this
      auto scales8 = [&](int col, float (&w)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = __shfl_sync(0xffffffffu, swr[i], col >> 3);
      };
      // dequantize and store eight exact accumulator values of weight rows n0 .. n0 + 7
      auto store8 = [&](int n0, const int (&iv)[8], const float (&w)[8]) {
        if (EPI == kEpiAcc) {
          const int64_t off = static_cast<int64_t>(m) * p.N + n0;
#pragma unroll
          for (int i = 0; i < 8; ++i) p.acc[off + i] = iv[i];
        } else {
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = __int2float_rn(iv[i]);
          store8_y<EPI == kEpiYb>(p, m, sam, n0, f, w);
        }
      };
      // eight exact accumulator values of tile columns col .. col + 7: the
      // result, or this piece's partial sums.  The whole warp calls this.
      auto emit8 = [&](int col, const int (&iv)[8]) {
        const int n0 = n_tile + col;
        if (piece) {
          if (mvalid && n0 < p.N) {   // N % 8 == 0: a group of 8 is all in or all out
            int4* d = slot(cid) + (col >> 2) * kPHalf;
            d[0] = make_int4(iv[0], iv[1], iv[2], iv[3]);
            d[kPHalf] = make_int4(iv[4], iv[5], iv[6], iv[7]);
          }
        } else {
          float w[8];
          if (EPI != kEpiAcc) scales8(col, w);
          if (mvalid && n0 < p.N) store8(n0, iv, w);
        }
      };
      if (fast) {
        const int b = ch & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(b), (ch >> 1) & 1, abort_flag, err,
                                                       kPWaitNs)))
          goto done;
        tc_fence_after();
        // column j of the accumulator is weight row nt * 256 + j
        const bool wide = !piece && EPI != kEpiAcc && y_wide;
#pragma unroll 1
        for (int c8 = 0; c8 < kPAccCols / 32; ++c8) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + b * kPAccCols + c8 * 32, v);
          tmem_wait_ld();
          if (c8 == kPAccCols / 32 - 1) {
            // the last columns are in registers: the accumulator is free for the next tile but one
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acce_leader0 + 8u * b);
          }
          if (wide) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const int col = c8 * 32 + g * 16;
              float f[16], w[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                f[i] = __int2float_rn(__float2int_rn(__uint_as_float(v[g * 16 + i])));
#pragma unroll
              for (int i = 0; i < 16; ++i) w[i] = __shfl_sync(0xffffffffu, swr[i & 7], (col >> 3) + (i >> 3));
              // N % 16 == 0 here: a group of 16 is all in or all out
              if (mvalid && n_tile + col < p.N) store16_y<EPI == kEpiYb>(p, m, sam, n_tile + col, f, w);
            }
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              int iv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) iv[i] = __float2int_rn(__uint_as_float(v[g * 8 + i]));
              emit8(c8 * 32 + g * 8, iv);
            }
          }
        }
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
          // N = 64 pass: column j is weight row 32 pass + (j % 32) of CTA j / 32's 128
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            int iv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) iv[i] = isum[g * 8 + i];
            emit8((g >> 2) * kPHalf + pass * 32 + (g & 3) * 8, iv);
          }
        }
      }
      // A CTA whose 128 token rows all lie past M (the second half of a
      // tile row at M <= 128) has no partial to share and nothing to store;
      // the other pieces' CTAs of the same half skip the exchange as well.
      if (piece && mt * kPTileM + static_cast<int>(rank) * kPHalf < p.M) {
        // every lane counts its own stores of the partial
        gpu_count_release(p.flags + (cid * 2 + rank) * 4 + q);
        const int s = p.sk_split, k = cid % s, c0 = cid - k;
        int j0, j1;
        piece_slice(k, s, &j0, &j1);
        // The slice [j0, j1) of every piece's partial (all 128 tokens) is
        // contiguous, (j1 - j0) x 2 KiB; the pipeline stages are free now (a
        // cut tile is a pair's last unit and its MMAs have completed), so the
        // s slices are copied there by bulk copies and summed from shared
        // memory: reading them from L2 one dependent round trip after another
        // was the slowest part of a cut tile.  Epilogue warp e copies pieces
        // e, e + 4, ... once all four lane quarters of each have stored.
        const int e = warp - kPEpiWarp0;
        const uint32_t slice_bytes = static_cast<uint32_t>(j1 - j0) * kPHalf * 16;
        const uint32_t sbuf = sA(0);
        for (int kk = e; kk < s; kk += 4)
          for (int qq = 0; qq < 4; ++qq)
            if (!__all_sync(0xffffffffu, gpu_count_wait_bounded(
                                             p.flags + ((c0 + kk) * 2 + rank) * 4 + qq, 32,
                                             abort_flag, err, kPWaitNs)))
              goto done;
        if (lane == 0) {
          // the partials (other SMs' stores, acquired above) are read by the TMA engine
          asm volatile("fence.proxy.async.global;" ::: "memory");
          uint32_t bytes = 0;
          for (int kk = e; kk < s; kk += 4) bytes += slice_bytes;
          mbar_arrive_expect_tx(red_bar, bytes);
          for (int kk = e; kk < s; kk += 4)
            bulk_load(sbuf + kk * slice_bytes,
                      p.part + (static_cast<int64_t>(c0 + kk) * 2 + rank) * (kPTileN / 4) * kPHalf +
                          static_cast<int64_t>(j0) * kPHalf,
                      slice_bytes, red_bar);
        }
        __syncwarp();
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(red_bar, 0, abort_flag, err, kPWaitNs)))
          goto done;
        const int4* sl = reinterpret_cast<const int4*>(gbase + (sbuf - base)) + row;
        // two column groups (8 weight rows) at a time
#pragma unroll 1
        for (int jb = j0; jb < j1; jb += 2) {
          int iv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) iv[i] = 0;
#pragma unroll 4
          for (int kk = 0; kk < s; ++kk) {
            const int4* src = sl + (kk * (j1 - j0) + (jb - j0)) * kPHalf;
            const int4 a = src[0], b = src[kPHalf];
            iv[0] += a.x; iv[1] += a.y; iv[2] += a.z; iv[3] += a.w;
            iv[4] += b.x; iv[5] += b.y; iv[6] += b.z; iv[7] += b.w;
          }
          const int col = jb * 4;
          float w[8];
          if (EPI != kEpiAcc) scales8(col, w);
          if (mvalid && n_tile + col < p.N) store8(n_tile + col, iv, w);
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

// CTA pairs that fit on the current device at once (one CTA per SM), cached
// per device.  All instantiations use the same shared memory and threads.
cudaError_t pair_max_clusters(int* out) {
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int nc = dev < 64 ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (nc <= 0) {
    auto kern = gemm_pair_kernel<false, kEpiY>;
    static std::atomic<uint64_t> attr_done{0};
    e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), PCfg<false>::kSmemBytes,
                                attr_done);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = PCfg<false>::kSmemBytes;
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

// Host side of the work split described at the top of this file.  Measured
// on GB300: after whole rounds, a last partial round of whole tiles runs
// faster than a full one (fewer pairs share the caches and HBM), so cutting
// it pays only when it saves many blocks (long K: 4096 x 2560 x 10240 went
// from 160 to 128 us; 4096 x 10240 x 2560, halves of 10 blocks, lost 2 %).
constexpr int kSkMinBlocks = 4;        // shortest piece worth giving a pair, in 128-K blocks
constexpr int kSkMaxSplit = 16;        // pieces per cut tile: their slices of the partials fit the stages
constexpr int kSkFixupBlocks = 2;      // storing, waiting for and adding partials, in blocks
constexpr int kSkAfterRoundsBlocks = 24;   // extra cost of cutting after whole rounds

struct PairPlan {
  int num_m_tiles, num_tiles, nkb;
  int clusters;     // pairs launched (P)
  int full_tiles;   // tiles dealt whole
  int sk_tiles;     // tiles cut into pieces (0: none)
  int sk_split;     // pieces per cut tile
};

// Whole rounds of tiles; then, when it is cheaper by the cost below (in units
// of one 128-K block of one pair), the r remaining tiles in s = P / r pieces
// each.  `allow_sk` false (no workspace) deals every tile whole.
PairPlan pair_plan(int64_t M, int64_t N, int64_t K, int nc, bool allow_sk) {
  PairPlan pl;
  pl.num_m_tiles = static_cast<int>((M + kPTileM - 1) / kPTileM);
  pl.num_tiles = pl.num_m_tiles * static_cast<int>((N + kPTileN - 1) / kPTileN);
  pl.nkb = static_cast<int>((K + kPBK - 1) / kPBK);
  pl.clusters = pl.num_tiles < nc ? pl.num_tiles : nc;
  pl.full_tiles = pl.num_tiles;
  pl.sk_tiles = 0;
  pl.sk_split = 1;
  if (!allow_sk || nc < 2) return pl;
  const int rounds = pl.num_tiles / nc, rem = pl.num_tiles % nc;
  if (rem == 0) return pl;
  int split = nc / rem;
  if (split > pl.nkb / kSkMinBlocks) split = pl.nkb / kSkMinBlocks;
  if (split > kSkMaxSplit) split = kSkMaxSplit;
  if (split < 2) return pl;
  const int64_t cost_whole = static_cast<int64_t>(rounds + 1) * pl.nkb;
  const int64_t cost_sk = static_cast<int64_t>(rounds) * pl.nkb + (pl.nkb + split - 1) / split +
                          kSkFixupBlocks + (rounds > 0 ? kSkAfterRoundsBlocks : 0);
  if (cost_sk >= cost_whole) return pl;
  pl.full_tiles = rounds * nc;
  pl.sk_tiles = rem;
  pl.sk_split = split;
  pl.clusters = rounds > 0 ? nc : rem * split;
  return pl;
}

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// A launch whose cut tiles make pieces wait on each other is cooperative:
// the runtime then starts it only with every CTA pair resident at once (or
// fails the launch), so no piece can wait on a partner that other work on
// the GPU keeps from starting.  The bounded waits stay as a backstop.
// After this library's quantization launch the kernel may also start before
// that launch ends (programmatic dependent launch): it sets up its barriers
// and tensor memory, then waits for the codes.
template <bool INT4, int EPI>
cudaError_t launch_pair(const CUtensorMap& tmX, const CUtensorMap& tmW, const PairArgs& a,
                        int clusters, cudaStream_t st, bool after_quant) {
  using C = PCfg<INT4>;
  auto kern = gemm_pair_kernel<INT4, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::kSmemBytes,
                                          attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (a.sk_tiles > 0) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n++].val.cooperative = 1;
  }
  if (after_quant) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n++].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, a);
}

}  // namespace

void pair_schedule(int64_t M, int64_t N, int64_t K, int pairs, int64_t capacity, int32_t* units,
                   int64_t* count, int32_t* info) {
  const PairPlan pl = pair_plan(M, N, K, pairs, true);
  PairArgs a{};
  a.num_m_tiles = pl.num_m_tiles;
  a.num_tiles = pl.num_tiles;
  a.nkb = pl.nkb;
  a.full_tiles = pl.full_tiles;
  a.sk_tiles = pl.sk_tiles;
  a.sk_split = pl.sk_split;
  info[0] = pl.clusters;
  info[1] = pl.full_tiles;
  info[2] = pl.sk_tiles;
  info[3] = pl.sk_split;
  info[4] = pl.nkb;
  info[5] = pl.num_tiles;
  int64_t n = 0;
  for (int c = 0; c < pl.clusters; ++c) {
    const int nu = pair_num_units(a, c, pl.clusters);
    for (int i = 0; i < nu; ++i, ++n) {
      if (n >= capacity) continue;
      const PUnit u = pair_unit(a, c, pl.clusters, i);
      int j0 = 0, j1 = kPTileN / 4;
      if (u.kind == kUnitPiece) piece_slice(c % pl.sk_split, pl.sk_split, &j0, &j1);
      int32_t* r = units + 7 * n;
      r[0] = c;
      r[1] = u.tile;
      r[2] = u.kb0;
      r[3] = u.kb1;
      r[4] = u.kind;
      r[5] = j0 * 4;   // weight rows of the tile this unit dequantizes and stores
      r[6] = j1 * 4;
    }
  }
  *count = n;
}

GemmScratch gemm_pair_scratch(int64_t M, int64_t N, int64_t K) {
  GemmScratch sc;
  int nc = 0;
  if (pair_max_clusters(&nc) != cudaSuccess) return sc;
  const PairPlan pl = pair_plan(M, N, K, nc, true);
  if (pl.sk_tiles == 0) return sc;
  const int pieces = pl.sk_tiles * pl.sk_split;
  const size_t part_bytes = static_cast<size_t>(pieces) * 2 * kPHalf * kPTileN * 4;
  sc.zero_offset = round256(part_bytes);
  sc.zero_words = pieces * 2 * 4;
  sc.bytes = sc.zero_offset + round256(static_cast<size_t>(sc.zero_words) * 4);
  return sc;
}

cudaError_t launch_gemm_pair(const __half* qa16, const float* sa, const int* row_l1, int64_t M,
                             int64_t N, int64_t K, const uint8_t* w, bool int4, const float* sw,
                             int mode, __half* y, int32_t* acc, void* workspace, cudaStream_t st,
                             bool after_quant) {
  CUtensorMap tmX, tmW;
  if (!make_tensor_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qa16, K, M, K * 2, kPSubK, kPHalf,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t wbytes = int4 ? K / 2 : K;
  if (!make_tensor_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, wbytes, N, wbytes,
                          int4 ? kPSubK / 2 : kPSubK, kPHalf,
                          int4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  int nc = 0;
  cudaError_t e = pair_max_clusters(&nc);
  if (e != cudaSuccess) return e;
  const PairPlan pl = pair_plan(M, N, K, nc, workspace != nullptr);
  PairArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.num_m_tiles = pl.num_m_tiles;
  a.num_tiles = pl.num_tiles;
  a.nkb = pl.nkb;
  a.full_tiles = pl.full_tiles;
  a.sk_tiles = pl.sk_tiles;
  a.sk_split = pl.sk_split;
  a.part = pl.sk_tiles ? static_cast<::int4*>(workspace) : nullptr;
  a.flags = pl.sk_tiles ? reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                                 gemm_pair_scratch(M, N, K).zero_offset)
                        : nullptr;
  a.sa = sa;
  a.sw = sw;
  a.y = y;
  a.acc = acc;
  a.row_l1 = row_l1;
  a.l1_limit = (1 << 23) / (int4 ? 8 : 127);
  e = device_error_word(&a.err);
  if (e != cudaSuccess) return e;
  if (int4)
    return mode == kEpiY    ? launch_pair<true, kEpiY>(tmX, tmW, a, pl.clusters, st, after_quant)
           : mode == kEpiYb ? launch_pair<true, kEpiYb>(tmX, tmW, a, pl.clusters, st, after_quant)
                            : launch_pair<true, kEpiAcc>(tmX, tmW, a, pl.clusters, st, after_quant);
  return mode == kEpiY    ? launch_pair<false, kEpiY>(tmX, tmW, a, pl.clusters, st, after_quant)
         : mode == kEpiYb ? launch_pair<false, kEpiYb>(tmX, tmW, a, pl.clusters, st, after_quant)
                          : launch_pair<false, kEpiAcc>(tmX, tmW, a, pl.clusters, st, after_quant);
}

}  // namespace cider
