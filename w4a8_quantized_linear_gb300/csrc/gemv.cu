// gemv.cu -- small-M (M <= 16) weight-streaming path: integer dot products
// with dp4a, fused dequant (Cider README, page "cider": "Architecture",
// decode path int8_mv, and "Limitations": the M = 1 kernel is bound by
// weight bandwidth).  Unlike the page's decode kernel, the activation is
// quantized per token here too, so results do not depend on M.
//
// Layout: each CTA (8 consumer warps + 1 producer warp) keeps the quantized
// activation rows (MB x K int8 codes, rows beyond M zero) in shared memory.
// In the fused form the CTA quantizes the fp16 rows itself (per-token amax,
// IEEE scale, round-half-even codes), which for one token or short rows costs
// far less than a separate launch; from 2 tokens with longer rows the codes
// come from one quantization launch instead, so that each of the many CTAs
// does not quantize the same rows again.  The producer warp issues the first
// weight loads before that staging, so HBM streaming starts at once: weight
// tiles of 16 rows x 256 bytes go by 2-D TMA into a ring of as many slots
// as a row block has tiles (at least 4, at most 12, as shared memory allows),
// each slot refilled by its own lane of the producer warp.
// Grids are sized to be resident in one wave; CTA c takes row blocks c,
// c + grid, ...
//
// For 4 to 16 tokens the dot products run on the tensor cores (mma.sync
// m16n8k16, fp16 operands holding the exact codes, fp32 accumulation drained
// after every 64 codes of int8 weights or 128 of int4 weights (per group at
// gs 64: every 64), so every partial sum stays far below 2^24 and exact; a
// packed INT4 word goes straight to fp16 pairs of its even and its odd codes,
// and the int8 activations are split the same way): each tile is split into
// four 64-byte quarters, one per warp, and the two sets of four warps take
// alternate tiles; the warps' partial sums meet in shared memory at the end
// of each 16-row block.  This form takes prequantized rows by one bulk copy
// per token row, and when the quantization launch precedes it on the stream
// it is launched as that kernel's programmatic dependent: it streams weights
// at once and waits (griddepcontrol.wait) before reading codes or scales.
// With dp4a at these M each weight byte costs M / 4 instructions plus
// shared-memory reloads of the activations, which made the kernel
// compute-bound well below the weight bandwidth.
//
// For 1 or 2 tokens (dp4a form) consumer warp w owns rows 2w, 2w+1 of a
// block; lane l works on row 2w + l/16 and its 16-byte chunk l%16 of each
// tile.  Accumulation is exact int32 (dp4a).  Per channel: the lane sums are reduced
// exactly and y = fp16((float(acc) * s_a) * s_w).  Per group: every chunk
// lies inside one group; the lane's exact partial of that group is scaled by
// s_w[n, g] and summed in fp32, y = fp16(s_a * sum) (a reassociation of the
// per-group formula); the accumulator mode reduces the lanes of a group
// exactly and stores acc_g.
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <utility>
#include <cuda.h>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kGemvWarps = 8;                        // consumer warps
constexpr int kGemvThreads = (kGemvWarps + 1) * 32;  // + one TMA producer warp
constexpr int kSmemActMax = 200 * 1024;
constexpr int kBoxRows = 16;                         // weight rows per tile (2 per consumer warp)
constexpr int kBoxBytes = 256;                       // weight bytes of a row per tile
constexpr int kTileBytes = kBoxRows * kBoxBytes;     // 4 KiB
constexpr int kRingMax = 12;
constexpr int kStageBatch = 4;    // 16-byte activation loads in flight per thread while staging
constexpr int kSmemBudget = 227 * 1024 - 4096;       // dynamic: leave room for static arrays
constexpr int kRedBytes = kGemvWarps * 32 * 8 * 4;   // tensor-core form: block reduction buffer

// 16 x 8 x 16 tensor-core product on fp16 fragments, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Eight codes (byte i = code i) in natural order, or for INT4 weights in the
// order [codes 0,2,4,6 | codes 1,3,5,7] that lines up with the low / high
// nibbles of a packed weight word.
template <bool INT4>
__device__ __forceinline__ uint2 arrange8(uint32_t lo, uint32_t hi) {
  if (INT4) return make_uint2(__byte_perm(lo, hi, 0x6420u), __byte_perm(lo, hi, 0x7531u));
  return make_uint2(lo, hi);
}

struct GemvArgs {
  const __half* x;
  const int8_t* qa;
  const float* sa;
  int M, K;
  int64_t N;
  const float* sw;
  int gs, G, NS;
  int ks, tps, Ka;    // K slices, tiles per slice, staged codes per token row
  int P;              // row pitch of the staged codes (bytes; >= Ka)
  __half* y;
  int32_t* acc;
  uint32_t* part;     // ks > 1: partial sums [ks][M][N] (int32 per channel, fp32 per group)
  int* err;
};

// The weight matrix streams through a ring of NS tiles of 16 rows x 256
// bytes, loaded by TMA (one 2D box per tile, zero-filled past N and past the
// end of a row) by the producer warp.  CTA c takes row blocks c, c + grid, ...
// and for each the tiles along K.  With K split into ks slices (few row
// blocks, long rows), CTA c takes slice c % ks of row blocks c / ks,
// c / ks + grid / ks, ..., stages only that slice's activation codes, and
// writes partial sums that gemv_combine_kernel adds up and dequantizes.  In
// the dp4a form consumer warp w owns rows 2w, 2w+1 of the block; lane l works
// on row 2w + l/16 and on its 16-byte chunk l%16 of each tile, accumulating
// over the tiles of the block, and the 16 lanes of a row are reduced at the
// block's end.
// The tensor-core form with int4 weights and per-group scales is built for
// three CTAs per SM (72 registers instead of ~92): its shared memory allows a
// third CTA at the sizes it serves, and the extra warps hide its latency
// chains.  (The int8 per-group form usually has no room for a third CTA.)
template <int MB, bool INT4, bool PG, int EPI, bool FUSEQ, bool MMA>
__global__ void __launch_bounds__(kGemvThreads, (MMA && PG && INT4) ? 3 : 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmW, const GemvArgs p) {
  static_assert(!MMA || (MB >= 4 && !(PG && EPI == kEpiAcc)), "tensor-core form");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KiB aligned
  uint8_t* ring = smem;
  uint8_t* s_act = smem + static_cast<size_t>(p.NS) * kTileBytes;
  __shared__ __align__(8) uint64_t s_full[kRingMax];
  __shared__ __align__(8) uint64_t s_empty[kRingMax];
  __shared__ __align__(8) uint64_t s_actbar;   // tensor-core form: the rows' bulk copies
  __shared__ float s_sa[16];
  __shared__ float s_rcp[16];
  __shared__ unsigned s_amax[16];
  __shared__ uint32_t s_abort;

  constexpr int VALS = INT4 ? 32 : 16;  // values per 16-byte chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = p.M, K = p.K, NS = p.NS;
  const int64_t N = p.N;
  const int64_t rowbytes = INT4 ? K / 2 : K;
  const int ntk = static_cast<int>((rowbytes + kBoxBytes - 1) / kBoxBytes);  // tiles per block
  const int64_t nblocks = (N + kBoxRows - 1) / kBoxRows;
  const int nchunks = K / VALS;
  // this CTA's K slice (the whole row when ks == 1)
  constexpr int kCodesPerTile = INT4 ? 2 * kBoxBytes : kBoxBytes;
  const int ks = p.ks;
  const int slice = static_cast<int>(blockIdx.x) % ks;
  const int64_t b_first = blockIdx.x / ks, b_step = gridDim.x / ks;
  const int kt0 = slice * p.tps;
  const int kt1 = kt0 + p.tps < ntk ? kt0 + p.tps : ntk;
  const int kbase = kt0 * kCodesPerTile;   // first code of the slice
  const int Ka = p.Ka;                     // staged codes per token row
  const int P = p.P;                       // their row pitch in shared memory
  // the tensor-core form takes prequantized rows by bulk copies, in natural
  // order (its INT4 converter picks even / odd codes itself)
  constexpr bool kBulkAct = MMA && !FUSEQ;
  const int act_bytes = Ka < K - kbase ? Ka : K - kbase;   // copied per row (a multiple of 32)

  if (threadIdx.x == 0) {
    s_abort = 0u;
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_empty[i]), MMA ? kGemvWarps / 2 : kGemvWarps);
    }
    mbar_init(smem_u32(&s_actbar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (ks > 1) pdl_launch_dependents();   // the combine launch may start now

  if (warp == kGemvWarps) {
    // ------------------------------------------------------------ producer
    // Lane s refills ring slot s (tiles it = s, s + NS, ...): the copies one
    // thread issues complete one after another (~0.45 us per 4 KB tile on
    // GB300, however many are in flight), so each slot gets its own issuer.
    if (lane == 0) prefetch_tensormap(&tmW);
    __syncwarp();
    if (kBulkAct && lane == 31) {
      // one bulk copy per token row of the slice's codes (q_a and its rows
      // start on 16-byte boundaries, K % 32 == 0); the rest stays zero.  The
      // codes may come from the launch before this one: wait for it (the
      // weight tiles above do not depend on it)
      pdl_wait();
      const uint32_t bar = smem_u32(&s_actbar);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(M * act_bytes));
      for (int m = 0; m < M; ++m)
        bulk_load(smem_u32(s_act + static_cast<size_t>(m) * P), p.qa + static_cast<int64_t>(m) * K + kbase,
                  static_cast<uint32_t>(act_bytes), bar);
    }
    if (lane < NS) {
      int it = 0;
      for (int64_t b = b_first; b < nblocks; b += b_step)
        for (int kt = kt0; kt < kt1; ++kt, ++it) {
          const int s = it % NS;
          if (s != lane) continue;
          if (!mbar_wait_bounded(smem_u32(&s_empty[s]), ((it / NS) & 1) ^ 1u, &s_abort, p.err,
                                 kKernelWaitTimeoutNs))
            break;
          mbar_arrive_expect_tx(smem_u32(&s_full[s]), kTileBytes);
          tma_load_2d(smem_u32(ring + s * kTileBytes), &tmW, smem_u32(&s_full[s]), kt * kBoxBytes,
                      static_cast<int32_t>(b * kBoxRows));
        }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int cthreads = kGemvWarps * 32;
  const int ctid = threadIdx.x;
  pdl_wait();   // rows, codes and scales may come from the launch before this one
  if (FUSEQ) {
    // per-token amax (|x| >= 0, so its float bits order like unsigned
    // integers), then the codes; x is [M, K] row-major, vector i is row i/nvec
    const int nvec = K / 8;
    const int tot = M * nvec;
    const uint4* xv = reinterpret_cast<const uint4*>(p.x);
    if (ctid < 16) s_amax[ctid] = 0u;
    named_barrier_sync(1, cthreads);
    // short rows (every vector of the MB rows in one batch per thread): the
    // rows stay in registers from the max pass to the code pass, and a
    // single token's max is reduced in the warp before the one atomic per
    // warp (the prologue runs before any weight tile is consumed, so every
    // round trip here delays the stream)
    const bool one_batch = MB * nvec <= cthreads * kStageBatch;
    uint4 vkeep[kStageBatch];
    float wmax = 0.0f;   // this thread's max for a single token
    for (int b0 = ctid; b0 < tot; b0 += cthreads * kStageBatch) {
      uint4 v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = b0 + u * cthreads;
        v[u] = i < tot ? xv[i] : make_uint4(0u, 0u, 0u, 0u);
        vkeep[u] = v[u];
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = b0 + u * cthreads;
        if (i < tot) {
          const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
          __half2 a2 = __habs2(h[0]);
#pragma unroll
          for (int q = 1; q < 4; ++q) a2 = __hmax2(a2, __habs2(h[q]));
          const float a = fmaxf(__low2float(a2), __high2float(a2));
          if (MB == 1)
            wmax = fmaxf(wmax, a);
          else
            atomicMax(&s_amax[i / nvec], __float_as_uint(a));
        }
      }
    }
    if (MB == 1) {
      // after the loop, which a thread past the row's vectors never entered:
      // every lane of every consumer warp takes part in the reduction
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      if ((ctid & 31) == 0) atomicMax(&s_amax[0], __float_as_uint(wmax));
    }
    named_barrier_sync(1, cthreads);
    if (ctid < MB) {
      const float amax = __uint_as_float(s_amax[ctid]);
      const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
      s_sa[ctid] = sc;
      s_rcp[ctid] = __frcp_rn(sc);
    }
    named_barrier_sync(1, cthreads);
    for (int b0 = ctid; b0 < MB * nvec; b0 += cthreads * kStageBatch) {
      uint4 v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = b0 + u * cthreads;
        v[u] = one_batch ? vkeep[u] : (i < tot ? xv[i] : make_uint4(0u, 0u, 0u, 0u));
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = b0 + u * cthreads;
        if (i < MB * nvec) {
          uint2 out = make_uint2(0u, 0u);
          if (i < tot) {
            const int m = i / nvec;
            const float sc = s_sa[m], r = s_rcp[m];
            const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
            uint32_t word[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const float2 f0 = __half22float2(h[2 * q]), f1 = __half22float2(h[2 * q + 1]);
              const int c0 = static_cast<int>(act_code(f0.x, sc, r));
              const int c1 = static_cast<int>(act_code(f0.y, sc, r));
              const int c2 = static_cast<int>(act_code(f1.x, sc, r));
              const int c3 = static_cast<int>(act_code(f1.y, sc, r));
              word[q] = (static_cast<uint32_t>(c0 & 0xFF)) | (static_cast<uint32_t>(c1 & 0xFF) << 8) |
                        (static_cast<uint32_t>(c2 & 0xFF) << 16) | (static_cast<uint32_t>(c3 & 0xFF) << 24);
            }
            out = arrange8<INT4 && !MMA>(word[0], word[1]);
          }
          const int m = i / nvec;
          *reinterpret_cast<uint2*>(s_act + static_cast<size_t>(m) * P + 8 * (i - m * nvec)) = out;
        }
      }
    }
  } else if (kBulkAct) {
    // zeros where no copy lands: rows past M, and codes past K in a row
    const int tail16 = (Ka - act_bytes) / 16;
    for (int i = ctid; i < MB * (Ka / 16); i += cthreads) {
      const int m = i / (Ka / 16), c = i - m * (Ka / 16);
      if (m >= M || c >= (Ka / 16) - tail16)
        *reinterpret_cast<uint4*>(s_act + static_cast<size_t>(m) * P + c * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
  } else {
    // codes [kbase, kbase + Ka) of every token row (zeros past K and past M)
    const int n16 = Ka / 16;
    for (int i = ctid; i < MB * n16; i += cthreads) {
      const int m = i / n16, c = i - m * n16;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < M && kbase + c * 16 < K)
        v = *reinterpret_cast<const uint4*>(p.qa + static_cast<int64_t>(m) * K + kbase + c * 16);
      const uint2 a = arrange8<INT4>(v.x, v.y), b = arrange8<INT4>(v.z, v.w);
      *reinterpret_cast<uint4*>(s_act + static_cast<size_t>(m) * P + c * 16) = make_uint4(a.x, a.y, b.x, b.y);
    }
  }
  if (!FUSEQ) {
    if (ctid < MB) s_sa[ctid] = (p.sa != nullptr && ctid < M) ? p.sa[ctid] : 0.0f;
  }
  named_barrier_sync(1, cthreads);

  if constexpr (MMA) {
    // ---------------------------------------------------- tensor-core form
    __shared__ int s_red[kGemvWarps][32 * 8];
    const int q = warp & 3;         // 64-code quarter of every tile
    const int par = warp >> 2;      // takes the tiles with it % 2 == par
    const int g8 = lane >> 2, t4 = lane & 3;
    // fragment k order: in k-step j, thread t4 holds codes 16 t4 + 4 j .. + 3
    // of its quarter for both operands (the same permutation of K for A and B)
    // staged rows start at code kbase: the code at k lives at row + (k - kbase)
    const uint8_t* arow0 = s_act + static_cast<size_t>(g8) * P;
    const uint8_t* arow1 = s_act + static_cast<size_t>(g8 + 8) * P;
    if (kBulkAct && !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_actbar), 0u, &s_abort, p.err,
                                                               kKernelWaitTimeoutNs)))
      return;
    int it = 0;
    for (int64_t b = b_first; b < nblocks; b += b_step) {
      int iacc[8];    // [n-block][4]: tokens g8 (0, 1) / g8 + 8 (2, 3), rows 2 t4 (+1)
      float facc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        iacc[i] = 0;
        facc[i] = 0.0f;
      }
      for (int kt = kt0; kt < kt1; ++kt, ++it) {
        if ((it & 1) != par) continue;
        const int s = it % NS;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_full[s]), (it / NS) & 1,
                                                       &s_abort, p.err, kKernelWaitTimeoutNs)))
          return;
        const uint8_t* wt = ring + s * kTileBytes + q * 64;   // the quarter: 64 bytes per row
        // scale the exact partial sums of one group (per group) or add them (per channel)
        auto drain = [&](float (&c0)[4], float (&c1)[4], int gi) {
          if (!PG) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              iacc[i] += __float2int_rn(c0[i]);   // exact integers below 2^20
              iacc[4 + i] += __float2int_rn(c1[i]);
            }
          } else {
            // one weight scale per (row, group), shared by both tokens of the
            // fragment; s_a is applied once to the finished sum (rows past N
            // read row N - 1's scale and are never stored)
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                int64_t n = b * kBoxRows + nb * 8 + 2 * t4 + e;
                n = n < N ? n : N - 1;
                const float sw = __ldg(p.sw + n * p.G + gi);
                const float* c = nb ? c1 : c0;
                facc[4 * nb + e] = fmaf(sw, c[e], facc[4 * nb + e]);
                facc[4 * nb + 2 + e] = fmaf(sw, c[2 + e], facc[4 * nb + 2 + e]);
              }
            }
          }
        };
        if (!INT4) {
          // thread t4 holds codes 16 t4 .. + 15 of the quarter; k-step j uses its word j
          const int k0 = kt * kBoxBytes + q * 64 + 16 * t4;
          uint4 al = make_uint4(0u, 0u, 0u, 0u), ah = al;
          if (k0 < K && g8 < MB) al = *reinterpret_cast<const uint4*>(arow0 + (k0 - kbase));
          if (k0 < K && MB == 16) ah = *reinterpret_cast<const uint4*>(arow1 + (k0 - kbase));
          const uint4 w0 = *reinterpret_cast<const uint4*>(wt + g8 * kBoxBytes + 16 * t4);
          const uint4 w1 = *reinterpret_cast<const uint4*>(wt + (8 + g8) * kBoxBytes + 16 * t4);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s_empty[s]));  // the tile is in registers now
          const uint32_t av[4] = {al.x, al.y, al.z, al.w}, hv[4] = {ah.x, ah.y, ah.z, ah.w};
          const uint32_t bv0[4] = {w0.x, w0.y, w0.z, w0.w}, bv1[4] = {w1.x, w1.y, w1.z, w1.w};
          float c0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t a0, a2, a1 = 0u, a3 = 0u, x0, x1, y0, y1;
            s8x4_to_h2x2(av[j], a0, a2);
            if (MB == 16) s8x4_to_h2x2(hv[j], a1, a3);
            s8x4_to_h2x2(bv0[j], x0, x1);
            s8x4_to_h2x2(bv1[j], y0, y1);
            mma_16816(c0, a0, a1, a2, a3, x0, x1);
            mma_16816(c1, a0, a1, a2, a3, y0, y1);
          }
          drain(c0, c1, PG ? (kt * kBoxBytes + q * 64) / p.gs : 0);
        } else {
          // the quarter holds 128 codes in two 64-code halves; thread t4 holds codes
          // 16 t4 .. + 15 of each half (8 packed bytes), so every k-step stays inside
          // one half (one group when gs = 64).  A packed word's low nibbles are its
          // even codes: each 8 codes go through two k-steps, even codes then odd.
          const int cb = kt * (2 * kBoxBytes) + q * 128;
          // both halves lie in one group unless gs is 64: one drain for the quarter
          const bool drain_half = PG && (p.gs % 128) != 0;
          float c0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k0 = cb + 64 * h + 16 * t4;
            uint4 al = make_uint4(0u, 0u, 0u, 0u), ah = al;
            if (k0 < K && g8 < MB) al = *reinterpret_cast<const uint4*>(arow0 + (k0 - kbase));
            if (k0 < K && MB == 16) ah = *reinterpret_cast<const uint4*>(arow1 + (k0 - kbase));
            const uint2 w0 = *reinterpret_cast<const uint2*>(wt + g8 * kBoxBytes + 32 * h + 8 * t4);
            const uint2 w1 = *reinterpret_cast<const uint2*>(wt + (8 + g8) * kBoxBytes + 32 * h + 8 * t4);
            if (h == 1) {
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&s_empty[s]));  // the tile is in registers now
            }
            const uint32_t av[4] = {al.x, al.y, al.z, al.w}, hv[4] = {ah.x, ah.y, ah.z, ah.w};
            const uint32_t wv0[2] = {w0.x, w0.y}, wv1[2] = {w1.x, w1.y};
#pragma unroll
            for (int j = 0; j < 2; ++j) {          // packed word j: codes 8 j .. 8 j + 7
              uint32_t we0[2], wo0[2], we1[2], wo1[2];   // rows g8 and 8 + g8: even / odd pairs
              s4x8_to_h2_eo(wv0[j], we0, wo0);
              s4x8_to_h2_eo(wv1[j], we1, wo1);
              uint32_t ae[2], ao[2], he[2] = {0u, 0u}, ho[2] = {0u, 0u};   // tokens g8 / 8 + g8
              s8x8_to_h2_eo(av[2 * j], av[2 * j + 1], ae, ao);
              if (MB == 16) s8x8_to_h2_eo(hv[2 * j], hv[2 * j + 1], he, ho);
              mma_16816(c0, ae[0], he[0], ae[1], he[1], we0[0], we0[1]);   // even codes
              mma_16816(c1, ae[0], he[0], ae[1], he[1], we1[0], we1[1]);
              mma_16816(c0, ao[0], ho[0], ao[1], ho[1], wo0[0], wo0[1]);   // odd codes
              mma_16816(c1, ao[0], ho[0], ao[1], ho[1], wo1[0], wo1[1]);
            }
            if (h == 1 || drain_half) {   // sums of 128 products stay far below 2^24: exact
              drain(c0, c1, PG ? (cb + 64 * h) / p.gs : 0);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                c0[i] = 0.0f;
                c1[i] = 0.0f;
              }
            }
          }
        }
      }
      // the 8 warps' partials of the block's 16 tokens x 16 rows meet in shared memory
#pragma unroll
      for (int i = 0; i < 8; ++i) s_red[warp][lane * 8 + i] = PG ? __float_as_int(facc[i]) : iacc[i];
      named_barrier_sync(1, cthreads);
      {
        const int m = ctid >> 4, nl = ctid & 15;   // one output per consumer thread
        const int src = ((m & 7) * 4 + ((nl & 7) >> 1)) * 8 + (nl >> 3) * 4 + (m >> 3) * 2 + (nl & 1);
        const int64_t n = b * kBoxRows + nl;
        if (m < M && n < N) {
          const int64_t off = static_cast<int64_t>(m) * N + n;
          if (!PG) {
            int v = 0;
#pragma unroll
            for (int w = 0; w < kGemvWarps; ++w) v += s_red[w][src];
            if (EPI == kEpiAcc)
              p.acc[off] = v;
            else if (ks > 1)
              p.part[(static_cast<int64_t>(slice) * M + m) * N + n] = static_cast<uint32_t>(v);
            else
              reinterpret_cast<uint16_t*>(p.y)[off] = y_bits<EPI == kEpiYb>(
                  __fmul_rn(__fmul_rn(__int2float_rn(v), s_sa[m]), __ldg(p.sw + n)));
          } else {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kGemvWarps; ++w) v += __int_as_float(s_red[w][src]);
            v = __fmul_rn(v, s_sa[m]);
            if (ks > 1)
              p.part[(static_cast<int64_t>(slice) * M + m) * N + n] = __float_as_uint(v);
            else
              reinterpret_cast<uint16_t*>(p.y)[off] = y_bits<EPI == kEpiYb>(v);
          }
        }
      }
      named_barrier_sync(1, cthreads);   // s_red is rewritten by the next block
    }
  } else {
  // ---------------------------------------------------- dp4a form
  const int rl = 2 * warp + (lane >> 4);  // row within the block
  const int ch = lane & 15;               // 16-byte chunk within the tile row
  int it = 0;
  for (int64_t b = b_first; b < nblocks; b += b_step) {
    const int64_t n = b * kBoxRows + rl;
    const bool nvalid = n < N;
    int acc[MB];
    float fs[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      acc[m] = 0;
      fs[m] = 0.0f;
    }
    for (int kt = kt0; kt < kt1; ++kt, ++it) {
      const int s = it % NS;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_full[s]), (it / NS) & 1, &s_abort,
                                                     p.err, kKernelWaitTimeoutNs)))
        return;
      const int c = kt * (kBoxBytes / 16) + ch;  // chunk index along the row
      const bool live = c < nchunks;
      const uint4 wv = *reinterpret_cast<const uint4*>(ring + s * kTileBytes + rl * kBoxBytes + ch * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_empty[s]));  // the tile is in registers now
      uint32_t wq[8];
      {
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (INT4) {
            const uint32_t u = ww[q] ^ 0x88888888u;
            wq[2 * q] = offset_nibbles_to_s8x4(u & 0x0F0F0F0Fu);
            wq[2 * q + 1] = offset_nibbles_to_s8x4((u >> 4) & 0x0F0F0F0Fu);
          } else {
            wq[q] = ww[q];
          }
        }
      }
      const int g = PG ? (c * VALS) / p.gs : 0;
      const float swg = (PG && EPI != kEpiAcc && live && nvalid) ? __ldg(p.sw + n * p.G + g) : 0.0f;
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        uint4 a0 = make_uint4(0u, 0u, 0u, 0u), a1 = a0;
        if (live) {
          // staged rows start at code kbase
          const uint8_t* ap = s_act + static_cast<size_t>(m) * P + (c * VALS - kbase);
          a0 = *reinterpret_cast<const uint4*>(ap);
          if (INT4) a1 = *reinterpret_cast<const uint4*>(ap + 16);
        }
        int pv = PG ? 0 : acc[m];
        pv = __dp4a(static_cast<int>(wq[0]), static_cast<int>(a0.x), pv);
        pv = __dp4a(static_cast<int>(wq[1]), static_cast<int>(a0.y), pv);
        pv = __dp4a(static_cast<int>(wq[2]), static_cast<int>(a0.z), pv);
        pv = __dp4a(static_cast<int>(wq[3]), static_cast<int>(a0.w), pv);
        if (INT4) {
          pv = __dp4a(static_cast<int>(wq[4]), static_cast<int>(a1.x), pv);
          pv = __dp4a(static_cast<int>(wq[5]), static_cast<int>(a1.y), pv);
          pv = __dp4a(static_cast<int>(wq[6]), static_cast<int>(a1.z), pv);
          pv = __dp4a(static_cast<int>(wq[7]), static_cast<int>(a1.w), pv);
        }
        if (!PG) {
          acc[m] = pv;
        } else if (EPI != kEpiAcc) {
          fs[m] = fmaf(swg, static_cast<float>(pv), fs[m]);
        } else {
          // exact per-group accumulators: reduce the lanes of each group (a
          // group is gs / VALS consecutive chunks of one row, within one tile)
          const int L = p.gs / VALS;
          for (int o = 1; o < L; o <<= 1) pv += __shfl_xor_sync(0xffffffffu, pv, o);
          if (live && nvalid && (ch % L) == 0 && m < M)
            p.acc[(static_cast<int64_t>(m) * N + n) * p.G + g] = pv;
        }
      }
    }
    if (PG && EPI == kEpiAcc) continue;
    // reduce the 16 lanes of each row (exact int32 per channel, fp32 per group)
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      uint32_t bits;
      if (!PG) {
        int v = acc[m];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        bits = static_cast<uint32_t>(v);
      } else {
        float v = fs[m];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        bits = __float_as_uint(v);
      }
      if (ch == (m & 15) && m < M && nvalid) {
        const int64_t off = static_cast<int64_t>(m) * N + n;
        if (EPI == kEpiAcc) {
          p.acc[off] = static_cast<int32_t>(bits);
        } else if (ks > 1) {
          p.part[(static_cast<int64_t>(slice) * M + m) * N + n] = bits;
        } else if (!PG) {
          reinterpret_cast<uint16_t*>(p.y)[off] = y_bits<EPI == kEpiYb>(
              __fmul_rn(__fmul_rn(__int2float_rn(static_cast<int>(bits)), s_sa[m]), __ldg(p.sw + n)));
        } else {
          reinterpret_cast<uint16_t*>(p.y)[off] =
              y_bits<EPI == kEpiYb>(__fmul_rn(__uint_as_float(bits), s_sa[m]));
        }
      }
    }
  }
}  // dp4a form
}

// Row pitch of the staged codes: in the tensor-core form a quarter-warp's
// 16-byte loads cover 64 bytes of each of two token rows, so the rows start
// 64 bytes apart modulo 128 and the two halves fall in different banks.
int64_t act_pitch(int64_t Ka, bool mma) { return mma ? (Ka + 127) / 128 * 128 + 64 : Ka; }

int ring_slots(int64_t MB, int64_t K, bool mma = false) {
  const int64_t room = kSmemBudget - (mma ? kRedBytes : 0) - MB * act_pitch(K, mma);
  int64_t ns = room / kTileBytes;
  if (ns > kRingMax) ns = kRingMax;
  return static_cast<int>(ns);
}

// Partial sums of the K slices -> y: per channel the exact int32 sum, then
// (acc * s_a) * s_w; per group the fp32 sum of the slices' partials, times
// s_a unless the partials already carry it (tensor-core form).
template <bool PG, bool PG_SCALED, bool BF16>
__global__ void __launch_bounds__(256) gemv_combine_kernel(const uint32_t* __restrict__ part,
                                                           int ks, int M, int64_t N,
                                                           const float* __restrict__ sa,
                                                           const float* __restrict__ sw,
                                                           __half* __restrict__ y) {
  const int64_t total = static_cast<int64_t>(M) * N;
  pdl_wait();   // the partials are the GEMV's, launched just before
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i / N);
    const int64_t n = i - static_cast<int64_t>(m) * N;
    if (!PG) {
      int v = 0;
      for (int s = 0; s < ks; ++s) v += static_cast<int>(part[s * total + i]);
      reinterpret_cast<uint16_t*>(y)[i] =
          y_bits<BF16>(__fmul_rn(__fmul_rn(__int2float_rn(v), __ldg(sa + m)), __ldg(sw + n)));
    } else {
      float v = 0.0f;
      for (int s = 0; s < ks; ++s) v += __uint_as_float(part[s * total + i]);
      reinterpret_cast<uint16_t*>(y)[i] = y_bits<BF16>(PG_SCALED ? v : __fmul_rn(v, __ldg(sa + m)));
    }
  }
}

// K split of the small-M path: ks slices of tps weight tiles, Ka codes staged
// per token row.
struct GemvSplit {
  int ks, tps, Ka;
};

// Cost model (in weight tiles streamed by one CTA): rounds of (row block,
// slice) units over the resident CTAs times tiles per unit, plus ~2 tiles for
// the combine launch.  Resident CTAs per SM are estimated from shared memory
// and, for registers, as 2 for the tensor-core form and 4 for the dp4a form
// (the kernels' measured register counts).  A split must win by 20 %.
GemvSplit gemv_plan(int64_t MB, int64_t N, int64_t K, bool int4, bool mma, bool allow,
                    int num_sms) {
  const int64_t rowbytes = int4 ? K / 2 : K;
  const int ntk = static_cast<int>((rowbytes + kBoxBytes - 1) / kBoxBytes);
  const int cpt = int4 ? 2 * kBoxBytes : kBoxBytes;
  const int64_t nblocks = (N + kBoxRows - 1) / kBoxRows;
  GemvSplit best{1, ntk, static_cast<int>(K)};
  auto cost = [&](int tps, int kse, int Ka) {
    int ns = ring_slots(MB, Ka, mma);
    if (ns > 8) ns = 8;
    const int64_t sm = static_cast<int64_t>(ns) * kTileBytes + MB * act_pitch(Ka, mma) + 1024;
    int64_t occ = (228 * 1024) / (sm + (mma ? kRedBytes : 0) + 2 * 1024);
    const int64_t cap = mma ? 2 : 4;
    if (occ > cap) occ = cap;
    if (occ < 1) occ = 1;
    const int64_t slots = static_cast<int64_t>(num_sms) * occ;
    const int64_t units = nblocks * kse;
    return static_cast<double>((units + slots - 1) / slots) * tps + (kse > 1 ? 2.0 : 0.0);
  };
  // only long rows: with few tiles per row block one CTA's chain is short
  // and the extra launches (quantization, combine) cost more than they save
  if (!allow || ntk < 16) return best;
  const double c1 = cost(ntk, 1, static_cast<int>(K));
  double bc = c1;
  for (int ks = 2; ks <= 16 && ntk / ks >= 2; ++ks) {
    const int tps = (ntk + ks - 1) / ks;
    const int kse = (ntk + tps - 1) / tps;
    if (kse != ks) continue;
    const int64_t ka = static_cast<int64_t>(tps) * cpt;
    const int Ka = static_cast<int>(ka < K ? ka : K);
    const double c = cost(tps, kse, Ka);
    if (c < bc && c < 0.8 * c1) {
      bc = c;
      best = GemvSplit{kse, tps, Ka};
    }
  }
  return best;
}

// Sizes of one weight-streaming launch: ring slots (enough for every tile of
// a (row block, slice) when that is more than four, so that all of a CTA's
// weight tiles are requested at once; fewer than four: it does not fit), the
// staged rows' pitch and the dynamic shared memory.
struct GemvSizes {
  int NS;
  int64_t pitch;
  size_t smem;
};

GemvSizes gemv_sizes(int64_t MB, const GemvSplit& sp, bool mma) {
  const int room = ring_slots(MB, sp.Ka, mma);
  const int want = sp.tps > 4 ? sp.tps : 4;
  GemvSizes z;
  z.NS = room < want ? room : want;
  z.pitch = act_pitch(sp.Ka, mma);
  z.smem = static_cast<size_t>(z.NS > 0 ? z.NS : 0) * kTileBytes + static_cast<size_t>(MB * z.pitch) +
           1024;
  return z;
}

// A launch that, when `dependent`, may begin before the launch before it on
// the stream has finished (the kernel waits for it with pdl_wait()).
template <typename... Params, typename... Args>
cudaError_t launch_maybe_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t st, bool dependent, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int MB, bool INT4, bool PG, int EPI, bool FUSEQ, bool MMA>
cudaError_t launch_one(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                       int64_t K, const uint8_t* w, const float* sw, int gs, __half* y,
                       int32_t* acc, const GemvSplit& sp, uint32_t* part, int num_sms,
                       cudaStream_t st, bool after_quant) {
  auto kern = gemv_kernel<MB, INT4, PG, EPI, FUSEQ, MMA>;
  const GemvSizes z = gemv_sizes(MB, sp, MMA);
  if (z.NS < 4) return cudaErrorInvalidValue;
  const int NS = z.NS;
  const int64_t pitch = z.pitch;
  const size_t smem = z.smem;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                          kSmemBudget - (MMA ? kRedBytes : 0) + 1024, attr_done);
  if (e != cudaSuccess) return e;
  CUtensorMap tmW;
  const uint64_t rowbytes = static_cast<uint64_t>(INT4 ? K / 2 : K);
  if (!make_tensor_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, rowbytes, static_cast<uint64_t>(N),
                          rowbytes, kBoxBytes, kBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  GemvArgs a;
  a.x = x;
  a.qa = qa;
  a.sa = sa;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = N;
  a.sw = sw;
  a.gs = gs;
  a.G = gs > 0 ? static_cast<int>(K / gs) : 1;
  a.NS = NS;
  a.ks = sp.ks;
  a.tps = sp.tps;
  a.Ka = sp.Ka;
  a.P = static_cast<int>(pitch);
  a.y = y;
  a.acc = acc;
  a.part = part;
  e = device_error_word(&a.err);
  if (e != cudaSuccess) return e;
  // Resident CTAs per SM from shared memory and the kernel's registers
  // (queried once): the grid is sized so that typical problems run in one wave.
  static std::atomic<int> regs_cache{0};
  int regs = regs_cache.load(std::memory_order_relaxed);
  if (regs == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
    regs = fa.numRegs > 0 ? fa.numRegs : 128;
    regs_cache.store(regs, std::memory_order_relaxed);
  }
  int occ = static_cast<int>((228 * 1024) / (smem + (MMA ? kRedBytes : 0) + 2 * 1024));
  const int by_regs = 65536 / (((regs + 7) / 8) * 8 * kGemvThreads);
  if (by_regs < occ) occ = by_regs;
  if (occ > 2048 / kGemvThreads) occ = 2048 / kGemvThreads;
  if (occ < 1) occ = 1;
  const int64_t nblocks = (N + kBoxRows - 1) / kBoxRows;
  int64_t blocks = nblocks * sp.ks;   // (row block, slice) units
  const int64_t cap = static_cast<int64_t>(num_sms) * occ;
  if (blocks > cap) blocks = cap / sp.ks * sp.ks;   // every CTA keeps one slice
  // after this library's own quantization launch the GEMV may start early
  // (programmatic dependent launch): its weight stream does not depend on the
  // codes, and it waits for them before reading them
  e = launch_maybe_dependent(kern, dim3(static_cast<unsigned>(blocks)), dim3(kGemvThreads), smem, st,
                             after_quant, tmW, a);
  if (e != cudaSuccess || sp.ks == 1) return e;
  const int64_t total = M * N;
  const unsigned cb = static_cast<unsigned>((total + 255) / 256 < 1024 ? (total + 255) / 256 : 1024);
  return launch_maybe_dependent(gemv_combine_kernel<PG, PG && MMA, EPI == kEpiYb>, dim3(cb), dim3(256), 0,
                                st, true, static_cast<const uint32_t*>(part), sp.ks, static_cast<int>(M),
                                N, sa, sw, y);
}

// The tensor-core form serves 4..16 tokens, int8 or int4 weights (not the
// exact per-group accumulators, which keep the dp4a lanes' group reductions).
bool gemv_uses_mma(int64_t MB, int64_t K, bool pg, int mode) {
  return MB >= 4 && !(pg && mode == kEpiAcc) && ring_slots(MB, K, true) >= 4;
}

template <int MB>
cudaError_t dispatch_mb(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                        int64_t K, const uint8_t* w, bool int4, const float* sw, int gs, int mode,
                        __half* y, int32_t* acc, uint32_t* part, int num_sms, cudaStream_t st,
                        bool after_quant) {
  const bool pg = gs > 0;
  const bool fq = x != nullptr;
  constexpr bool kMmaMB = MB >= 4;
  const bool mma = gemv_uses_mma(MB, K, pg, mode);
  const GemvSplit sp = gemv_plan(MB, N, K, int4, mma, part != nullptr && !fq && mode != kEpiAcc,
                                 num_sms);
  if (kMmaMB && mma) {
#define CIDER_GEMV_MMA_CASE(I4, P, E, F)                                                      \
  if (int4 == I4 && pg == P && mode == E && fq == F)                                          \
    return launch_one<MB, I4, P, E, F, kMmaMB>(x, qa, sa, M, N, K, w, sw, gs, y, acc, sp, part,    \
                                               num_sms, st, after_quant);
    CIDER_GEMV_MMA_CASE(false, false, kEpiY, true)
    CIDER_GEMV_MMA_CASE(false, true, kEpiY, true)
    CIDER_GEMV_MMA_CASE(false, false, kEpiY, false)
    CIDER_GEMV_MMA_CASE(false, true, kEpiY, false)
    CIDER_GEMV_MMA_CASE(false, false, kEpiAcc, false)
    CIDER_GEMV_MMA_CASE(true, false, kEpiY, true)
    CIDER_GEMV_MMA_CASE(true, true, kEpiY, true)
    CIDER_GEMV_MMA_CASE(true, false, kEpiY, false)
    CIDER_GEMV_MMA_CASE(true, true, kEpiY, false)
    CIDER_GEMV_MMA_CASE(true, false, kEpiAcc, false)
    CIDER_GEMV_MMA_CASE(false, false, kEpiYb, false)
    CIDER_GEMV_MMA_CASE(false, true, kEpiYb, false)
    CIDER_GEMV_MMA_CASE(true, false, kEpiYb, false)
    CIDER_GEMV_MMA_CASE(true, true, kEpiYb, false)
#undef CIDER_GEMV_MMA_CASE
  }
#define CIDER_GEMV_CASE(I4, P, E, F)                                                          \
  if (int4 == I4 && pg == P && mode == E && fq == F)                                          \
    return launch_one<MB, I4, P, E, F, false>(x, qa, sa, M, N, K, w, sw, gs, y, acc, sp, part,     \
                                              num_sms, st, after_quant);
  CIDER_GEMV_CASE(false, false, kEpiY, true)
  CIDER_GEMV_CASE(false, true, kEpiY, true)
  CIDER_GEMV_CASE(true, false, kEpiY, true)
  CIDER_GEMV_CASE(true, true, kEpiY, true)
  CIDER_GEMV_CASE(false, false, kEpiY, false)
  CIDER_GEMV_CASE(false, true, kEpiY, false)
  CIDER_GEMV_CASE(false, false, kEpiAcc, false)
  CIDER_GEMV_CASE(false, true, kEpiAcc, false)
  CIDER_GEMV_CASE(true, false, kEpiY, false)
  CIDER_GEMV_CASE(true, true, kEpiY, false)
  CIDER_GEMV_CASE(true, false, kEpiAcc, false)
  CIDER_GEMV_CASE(true, true, kEpiAcc, false)
  CIDER_GEMV_CASE(false, false, kEpiYb, false)
  CIDER_GEMV_CASE(false, true, kEpiYb, false)
  CIDER_GEMV_CASE(true, false, kEpiYb, false)
  CIDER_GEMV_CASE(true, true, kEpiYb, false)
#undef CIDER_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

bool gemv_fits(int64_t M, int64_t K) {
  if (M < 1 || M > 16) return false;
  int64_t mb = 1;
  while (mb < M) mb *= 2;
  return mb * K <= kSmemActMax && ring_slots(mb, K) >= 4;
}

int gemv_slices(int64_t M, int64_t N, int64_t K, bool int4, int group_size, int mode,
                int num_sms) {
  if (mode == kEpiAcc) return 1;
  int64_t mb = 1;
  while (mb < M) mb *= 2;
  return gemv_plan(mb, N, K, int4, gemv_uses_mma(mb, K, group_size > 0, mode), true, num_sms).ks;
}

void gemv_launch_info(int64_t M, int64_t N, int64_t K, bool int4, int group_size, bool split_allowed,
                      int num_sms, int32_t* info) {
  int64_t mb = 1;
  while (mb < M) mb *= 2;
  const bool mma = gemv_uses_mma(mb, K, group_size > 0, kEpiY);
  const GemvSplit sp = gemv_plan(mb, N, K, int4, mma, split_allowed, num_sms);
  const GemvSizes z = gemv_sizes(mb, sp, mma);
  info[0] = static_cast<int32_t>(mb);
  info[1] = mma ? 1 : 0;
  info[2] = sp.ks;
  info[3] = sp.tps;
  info[4] = sp.Ka;
  info[5] = static_cast<int32_t>(z.pitch);
  info[6] = z.NS;
  info[7] = static_cast<int32_t>(z.smem);
  info[8] = kSmemBudget - (mma ? kRedBytes : 0) + 1024;   // the launch's dynamic shared memory cap
  info[9] = int4 ? 2 * kBoxBytes : kBoxBytes;              // codes per weight tile row
}

size_t gemv_part_bytes(int64_t M, int64_t N, int64_t K, bool int4, int group_size, int mode,
                       int num_sms) {
  const int ks = gemv_slices(M, N, K, int4, group_size, mode, num_sms);
  return ks > 1 ? static_cast<size_t>(ks) * M * N * 4 : 0;
}

cudaError_t launch_gemv(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                        int64_t K, const uint8_t* w, bool int4, const float* sw, int group_size,
                        int mode, __half* y, int32_t* acc, void* part, int num_sms, cudaStream_t st,
                        bool after_quant) {
  uint32_t* pp = static_cast<uint32_t*>(part);
  if (M <= 1) return dispatch_mb<1>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, pp, num_sms, st, after_quant);
  if (M <= 2) return dispatch_mb<2>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, pp, num_sms, st, after_quant);
  if (M <= 4) return dispatch_mb<4>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, pp, num_sms, st, after_quant);
  if (M <= 8) return dispatch_mb<8>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, pp, num_sms, st, after_quant);
  return dispatch_mb<16>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, pp, num_sms, st, after_quant);
}

}  // namespace cider
