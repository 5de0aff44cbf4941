// gemv.cu -- small-M (M <= 16) weight-streaming path: integer dot products
// with dp4a, fused dequant (Cider README, page "cider": "Architecture",
// decode path int8_mv, and "Limitations": the M = 1 kernel is bound by
// weight bandwidth).  Unlike the page's decode kernel, the activation is
// quantized per token here too, so results do not depend on M.
//
// Layout: each CTA (8 warps) keeps the quantized activation rows (MB x K int8
// codes, rows beyond M zero) in shared memory.  In the fused form the CTA
// quantizes the fp16 rows itself (per-token amax, IEEE scale, round-half-even
// codes), which for decode-sized M costs far less than a separate launch.  The
// first weight loads are issued before that staging, so HBM streaming starts
// at once.  Weights stream with 16-byte loads: lane l of a warp takes chunks
// l, l+32, ... of a row (16 int8 or 32 packed INT4 values per chunk), so one
// warp load instruction covers 512 contiguous bytes; each warp keeps kRows
// rows and D chunk loads per row in flight.  Warps may split K (KS > 1) when
// N is too small to fill the GPU with whole rows; partial sums then meet in
// shared memory.  Grids are sized to be resident in one wave.
//
// Accumulation is exact int32 (dp4a).  Per channel: the lane sums are reduced
// exactly and y = fp16((float(acc) * s_a) * s_w).  Per group: every chunk
// lies inside one group; the lane's exact partial of that group is scaled by
// s_w[n, g] and summed in fp32, y = fp16(s_a * sum) (a reassociation of the
// per-group formula); the accumulator mode reduces the lanes of a group
// exactly and stores acc_g.
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
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
constexpr int kRingMax = 8;
constexpr int kStageBatch = 4;    // 16-byte activation loads in flight per thread while staging
constexpr int kSmemBudget = 227 * 1024 - 4096;       // dynamic: leave room for static arrays

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
  __half* y;
  int32_t* acc;
  int* err;
};

// The weight matrix streams through a ring of NS tiles of 16 rows x 256
// bytes, loaded by TMA (one 2D box per tile, zero-filled past N and past the
// end of a row) by the producer warp.  CTA c takes row blocks c, c + grid, ...
// and for each the tiles along K.  Consumer warp w owns rows 2w, 2w+1 of the
// block; lane l works on row 2w + l/16 and on its 16-byte chunk l%16 of each
// tile, accumulating over the tiles of the block, and the 16 lanes of a row
// are reduced at the block's end.
template <int MB, bool INT4, bool PG, int EPI, bool FUSEQ>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmW, const GemvArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KiB aligned
  uint8_t* ring = smem;
  uint8_t* s_act = smem + static_cast<size_t>(p.NS) * kTileBytes;
  __shared__ __align__(8) uint64_t s_full[kRingMax];
  __shared__ __align__(8) uint64_t s_empty[kRingMax];
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

  if (threadIdx.x == 0) {
    s_abort = 0u;
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_empty[i]), kGemvWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kGemvWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      int it = 0;
      for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x)
        for (int kt = 0; kt < ntk; ++kt, ++it) {
          const int s = it % NS;
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
  if (FUSEQ) {
    // per-token amax (|x| >= 0, so its float bits order like unsigned
    // integers), then the codes; x is [M, K] row-major, vector i is row i/nvec
    const int nvec = K / 8;
    const int tot = M * nvec;
    const uint4* xv = reinterpret_cast<const uint4*>(p.x);
    if (ctid < 16) s_amax[ctid] = 0u;
    named_barrier_sync(1, cthreads);
    for (int b0 = ctid; b0 < tot; b0 += cthreads * kStageBatch) {
      uint4 v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = b0 + u * cthreads;
        v[u] = i < tot ? xv[i] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = b0 + u * cthreads;
        if (i < tot) {
          const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
          __half2 a2 = __habs2(h[0]);
#pragma unroll
          for (int q = 1; q < 4; ++q) a2 = __hmax2(a2, __habs2(h[q]));
          atomicMax(&s_amax[i / nvec], __float_as_uint(fmaxf(__low2float(a2), __high2float(a2))));
        }
      }
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
        v[u] = i < tot ? xv[i] : make_uint4(0u, 0u, 0u, 0u);
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
            out = arrange8<INT4>(word[0], word[1]);
          }
          reinterpret_cast<uint2*>(s_act)[i] = out;
        }
      }
    }
  } else {
    const int n16 = K / 16;
    for (int i = ctid; i < MB * n16; i += cthreads) {
      const int m = i / n16, c = i - m * n16;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < M) v = *reinterpret_cast<const uint4*>(p.qa + static_cast<int64_t>(m) * K + c * 16);
      const uint2 a = arrange8<INT4>(v.x, v.y), b = arrange8<INT4>(v.z, v.w);
      *reinterpret_cast<uint4*>(s_act + static_cast<size_t>(m) * K + c * 16) = make_uint4(a.x, a.y, b.x, b.y);
    }
    if (ctid < MB) s_sa[ctid] = (p.sa != nullptr && ctid < M) ? p.sa[ctid] : 0.0f;
  }
  named_barrier_sync(1, cthreads);

  const int rl = 2 * warp + (lane >> 4);  // row within the block
  const int ch = lane & 15;               // 16-byte chunk within the tile row
  int it = 0;
  for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
    const int64_t n = b * kBoxRows + rl;
    const bool nvalid = n < N;
    int acc[MB];
    float fs[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      acc[m] = 0;
      fs[m] = 0.0f;
    }
    for (int kt = 0; kt < ntk; ++kt, ++it) {
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
      const float swg = (PG && EPI == kEpiY && live && nvalid) ? __ldg(p.sw + n * p.G + g) : 0.0f;
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        uint4 a0 = make_uint4(0u, 0u, 0u, 0u), a1 = a0;
        if (live) {
          const uint8_t* ap = s_act + static_cast<size_t>(m) * K + static_cast<size_t>(c) * VALS;
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
        } else if (EPI == kEpiY) {
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
        } else if (!PG) {
          p.y[off] = __float2half_rn(
              __fmul_rn(__fmul_rn(__int2float_rn(static_cast<int>(bits)), s_sa[m]), __ldg(p.sw + n)));
        } else {
          p.y[off] = __float2half_rn(__fmul_rn(__uint_as_float(bits), s_sa[m]));
        }
      }
    }
  }
}

int ring_slots(int64_t MB, int64_t K) {
  const int64_t room = kSmemBudget - MB * K;
  int64_t ns = room / kTileBytes;
  if (ns > kRingMax) ns = kRingMax;
  return static_cast<int>(ns);
}

template <int MB, bool INT4, bool PG, int EPI, bool FUSEQ>
cudaError_t launch_one(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                       int64_t K, const uint8_t* w, const float* sw, int gs, __half* y,
                       int32_t* acc, int num_sms, cudaStream_t st) {
  auto kern = gemv_kernel<MB, INT4, PG, EPI, FUSEQ>;
  const int NS = ring_slots(MB, K);
  if (NS < 4) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(NS) * kTileBytes + static_cast<size_t>(MB) * K + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), kSmemBudget + 1024,
                                          attr_done);
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
  a.y = y;
  a.acc = acc;
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
  int occ = static_cast<int>((228 * 1024) / (smem + 2 * 1024));
  const int by_regs = 65536 / (((regs + 7) / 8) * 8 * kGemvThreads);
  if (by_regs < occ) occ = by_regs;
  if (occ > 2048 / kGemvThreads) occ = 2048 / kGemvThreads;
  if (occ < 1) occ = 1;
  const int64_t nblocks = (N + kBoxRows - 1) / kBoxRows;
  int64_t blocks = nblocks;
  const int64_t cap = static_cast<int64_t>(num_sms) * occ;
  if (blocks > cap) blocks = cap;
  kern<<<static_cast<unsigned>(blocks), kGemvThreads, smem, st>>>(tmW, a);
  return cudaGetLastError();
}

template <int MB>
cudaError_t dispatch_mb(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                        int64_t K, const uint8_t* w, bool int4, const float* sw, int gs, int mode,
                        __half* y, int32_t* acc, int num_sms, cudaStream_t st) {
  const bool pg = gs > 0;
  const bool fq = x != nullptr;
#define CIDER_GEMV_CASE(I4, P, E, F)                                                          \
  if (int4 == I4 && pg == P && mode == E && fq == F)                                          \
    return launch_one<MB, I4, P, E, F>(x, qa, sa, M, N, K, w, sw, gs, y, acc, num_sms, st);
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

cudaError_t launch_gemv(const __half* x, const int8_t* qa, const float* sa, int64_t M, int64_t N,
                        int64_t K, const uint8_t* w, bool int4, const float* sw, int group_size,
                        int mode, __half* y, int32_t* acc, int num_sms, cudaStream_t st) {
  if (M <= 1) return dispatch_mb<1>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  if (M <= 2) return dispatch_mb<2>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  if (M <= 4) return dispatch_mb<4>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  if (M <= 8) return dispatch_mb<8>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  return dispatch_mb<16>(x, qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
}

}  // namespace cider
