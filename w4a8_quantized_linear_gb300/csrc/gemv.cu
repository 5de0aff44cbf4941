// gemv.cu -- small-M (M <= 16) weight-streaming path: integer dot products
// with dp4a, fused dequant (Cider README, page "cider": "Architecture",
// decode path int8_mv, and "Limitations": the M = 1 kernel is bound by
// weight bandwidth).  Unlike the page's decode kernel, the activation is
// quantized per token here too, so results do not depend on M.
//
// Layout: the CTA copies the quantized activation rows (MB x K int8, rows
// beyond M zero) into shared memory once, then streams weight rows from HBM
// with 16-byte loads: lane l of a warp takes chunks l, l+32, ... of each row
// (16 int8 or 32 packed INT4 values per chunk), so one warp load instruction
// covers 512 contiguous bytes.  Each warp keeps kRows rows and kDepth chunk
// loads per row in flight.  Warps may split K (KS > 1) when N is too small
// to fill the GPU with whole rows; partial sums then meet in shared memory.
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

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kGemvWarps = 16;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kRows = 2;
constexpr int kSmemActMax = 200 * 1024;

template <int MB>
struct Depth {
  static constexpr int value = MB >= 8 ? 2 : 4;
};

template <bool INT4>
__device__ __forceinline__ void load_chunks(const uint8_t* __restrict__ w, int64_t rowbytes,
                                            int64_t n0, int64_t N, int st, int s_end, int lane,
                                            int nchunks, uint4 (&dst)[kRows]) {
  const int c = st * 32 + lane;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (st < s_end && c < nchunks && n0 + r < N)
      dst[r] = ld_stream_v4(w + (n0 + r) * rowbytes + static_cast<int64_t>(c) * 16);
    else
      dst[r] = make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int MB, bool INT4, bool PG, int EPI>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const int8_t* __restrict__ qa, const float* __restrict__ sa, int M, int64_t N,
                int K, const uint8_t* __restrict__ w, const float* __restrict__ sw, int gs, int G,
                int KS, __half* __restrict__ y, int32_t* __restrict__ acc_out) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* s_act = smem;
  uint32_t* s_red = reinterpret_cast<uint32_t*>(smem + static_cast<size_t>(MB) * K);

  // Stage the activation codes.  INT4: each group of 8 codes is stored as
  // [codes 0,2,4,6 | codes 1,3,5,7] to line up with the low / high nibbles
  // of a packed weight word.
  const int n16 = K / 16;
  for (int i = threadIdx.x; i < MB * n16; i += kGemvThreads) {
    const int m = i / n16, c = i - m * n16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < M) v = *reinterpret_cast<const uint4*>(qa + static_cast<int64_t>(m) * K + c * 16);
    if (INT4) {
      uint4 d;
      d.x = __byte_perm(v.x, v.y, 0x6420u);
      d.y = __byte_perm(v.x, v.y, 0x7531u);
      d.z = __byte_perm(v.z, v.w, 0x6420u);
      d.w = __byte_perm(v.z, v.w, 0x7531u);
      v = d;
    }
    *reinterpret_cast<uint4*>(s_act + static_cast<size_t>(m) * K + c * 16) = v;
  }
  __syncthreads();

  constexpr int D = Depth<MB>::value;
  constexpr int VALS = INT4 ? 32 : 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = kGemvWarps / KS;
  const int rg = warp / KS, ks = warp - rg * KS;
  const int rows_per_pass = kRows * groups;
  const int nchunks = K / VALS;
  const int steps = (nchunks + 31) >> 5;
  const int s_begin = (ks * steps) / KS, s_end = ((ks + 1) * steps) / KS;
  const int64_t rowbytes = INT4 ? K / 2 : K;

  for (int64_t base = static_cast<int64_t>(blockIdx.x) * rows_per_pass; base < N;
       base += static_cast<int64_t>(gridDim.x) * rows_per_pass) {
    const int64_t n0 = base + rg * kRows;
    int acc[kRows][MB];
    float fs[kRows][MB];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        acc[r][m] = 0;
        fs[r][m] = 0.0f;
      }

    uint4 wb[D][kRows];
#pragma unroll
    for (int d = 0; d < D; ++d)
      load_chunks<INT4>(w, rowbytes, n0, N, s_begin + d, s_end, lane, nchunks, wb[d]);

    for (int st0 = s_begin; st0 < s_end; st0 += D) {
#pragma unroll
      for (int d = 0; d < D; ++d) {
        const int st = st0 + d;
        if (st >= s_end) break;
        const int c = st * 32 + lane;
        const bool live = c < nchunks;
        // weight words as int8 codes (INT4: low / high nibbles sign-extended)
        uint32_t wq[kRows][8];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const uint32_t* wv = reinterpret_cast<const uint32_t*>(&wb[d][r]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (INT4) {
              const uint32_t u = wv[j] ^ 0x88888888u;
              wq[r][2 * j] = offset_nibbles_to_s8x4(u & 0x0F0F0F0Fu);
              wq[r][2 * j + 1] = offset_nibbles_to_s8x4((u >> 4) & 0x0F0F0F0Fu);
            } else {
              wq[r][j] = wv[j];
            }
          }
        }
        load_chunks<INT4>(w, rowbytes, n0, N, st + D, s_end, lane, nchunks, wb[d]);

        float swg[kRows];
        const int g = PG ? (c * VALS) / gs : 0;
        if (PG && EPI == kEpiY) {
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            swg[r] = (live && n0 + r < N) ? __ldg(sw + (n0 + r) * G + g) : 0.0f;
        }
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          uint4 a0 = make_uint4(0u, 0u, 0u, 0u), a1 = a0;
          if (live) {
            const uint8_t* ap = s_act + static_cast<size_t>(m) * K + static_cast<size_t>(c) * VALS;
            a0 = *reinterpret_cast<const uint4*>(ap);
            if (INT4) a1 = *reinterpret_cast<const uint4*>(ap + 16);
          }
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            int p = PG ? 0 : acc[r][m];
            p = __dp4a(static_cast<int>(wq[r][0]), static_cast<int>(a0.x), p);
            p = __dp4a(static_cast<int>(wq[r][1]), static_cast<int>(a0.y), p);
            p = __dp4a(static_cast<int>(wq[r][2]), static_cast<int>(a0.z), p);
            p = __dp4a(static_cast<int>(wq[r][3]), static_cast<int>(a0.w), p);
            if (INT4) {
              p = __dp4a(static_cast<int>(wq[r][4]), static_cast<int>(a1.x), p);
              p = __dp4a(static_cast<int>(wq[r][5]), static_cast<int>(a1.y), p);
              p = __dp4a(static_cast<int>(wq[r][6]), static_cast<int>(a1.z), p);
              p = __dp4a(static_cast<int>(wq[r][7]), static_cast<int>(a1.w), p);
            }
            if (!PG)
              acc[r][m] = p;
            else if (EPI == kEpiY)
              fs[r][m] = fmaf(swg[r], static_cast<float>(p), fs[r][m]);
            else
              acc[r][m] = p;
          }
        }
        if (PG && EPI == kEpiAcc) {
          // exact per-group accumulators: reduce the lanes of each group
          const int L = gs / VALS;
#pragma unroll
          for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int m = 0; m < MB; ++m) {
              int v = acc[r][m];
              for (int o = 1; o < L; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
              if (live && (lane % L) == 0 && m < M && n0 + r < N)
                acc_out[(static_cast<int64_t>(m) * N + n0 + r) * G + g] = v;
            }
        }
      }
    }

    if (PG && EPI == kEpiAcc) continue;

    // Reduce the lanes (exact int32 for per channel, fp32 for per group).
    uint32_t tot[kRows][MB];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (!PG) {
          tot[r][m] = static_cast<uint32_t>(__reduce_add_sync(0xffffffffu, acc[r][m]));
        } else {
          float v = fs[r][m];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          tot[r][m] = __float_as_uint(v);
        }
      }

    auto finish = [&](int r, int m, uint32_t bits) {
      const int64_t n = n0 + r;
      if (m >= M || n >= N) return;
      if (EPI == kEpiAcc) {
        acc_out[static_cast<int64_t>(m) * N + n] = static_cast<int32_t>(bits);
      } else if (!PG) {
        const float v = __fmul_rn(__fmul_rn(__int2float_rn(static_cast<int>(bits)), __ldg(sa + m)),
                                  __ldg(sw + n));
        y[static_cast<int64_t>(m) * N + n] = __float2half_rn(v);
      } else {
        y[static_cast<int64_t>(m) * N + n] =
            __float2half_rn(__fmul_rn(__uint_as_float(bits), __ldg(sa + m)));
      }
    };

    if (KS == 1) {
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m)
          if (lane == ((r * MB + m) & 31)) finish(r, m, tot[r][m]);
    } else {
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
          for (int m = 0; m < MB; ++m) s_red[(warp * kRows + r) * MB + m] = tot[r][m];
      }
      __syncthreads();
      if (ks == 0) {
        for (int idx = lane; idx < kRows * MB; idx += 32) {
          const int r = idx / MB, m = idx - r * MB;
          uint32_t bits;
          if (!PG) {
            int s = 0;
            for (int k = 0; k < KS; ++k)
              s += static_cast<int>(s_red[((rg * KS + k) * kRows + r) * MB + m]);
            bits = static_cast<uint32_t>(s);
          } else {
            float s = 0.0f;
            for (int k = 0; k < KS; ++k)
              s += __uint_as_float(s_red[((rg * KS + k) * kRows + r) * MB + m]);
            bits = __float_as_uint(s);
          }
          finish(r, m, bits);
        }
      }
      __syncthreads();
    }
  }
}

template <int MB, bool INT4, bool PG, int EPI>
cudaError_t launch_one(const int8_t* qa, const float* sa, int64_t M, int64_t N, int64_t K,
                       const uint8_t* w, const float* sw, int gs, __half* y, int32_t* acc,
                       int num_sms, cudaStream_t st) {
  auto kern = gemv_kernel<MB, INT4, PG, EPI>;
  const size_t smem = static_cast<size_t>(MB) * K + kGemvWarps * kRows * MB * 4;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                          kSmemActMax + kGemvWarps * kRows * 16 * 4, attr_done);
  if (e != cudaSuccess) return e;
  int occ = 1;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kGemvThreads, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  constexpr int VALS = INT4 ? 32 : 16;
  const int64_t steps = (K / VALS + 31) / 32;
  int KS = 1;
  while (KS < 8 && 2 * KS <= steps &&
         (N + (kRows * kGemvWarps / KS) - 1) / (kRows * kGemvWarps / KS) < num_sms)
    KS *= 2;
  const int64_t rows_per_pass = kRows * (kGemvWarps / KS);
  int64_t blocks = (N + rows_per_pass - 1) / rows_per_pass;
  const int64_t cap = static_cast<int64_t>(num_sms) * occ;
  if (blocks > cap) blocks = cap;
  const int G = gs > 0 ? static_cast<int>(K / gs) : 1;
  kern<<<static_cast<unsigned>(blocks), kGemvThreads, smem, st>>>(
      qa, sa, static_cast<int>(M), N, static_cast<int>(K), w, sw, gs, G, KS, y, acc);
  return cudaGetLastError();
}

template <int MB>
cudaError_t dispatch_mb(const int8_t* qa, const float* sa, int64_t M, int64_t N, int64_t K,
                        const uint8_t* w, bool int4, const float* sw, int gs, int mode,
                        __half* y, int32_t* acc, int num_sms, cudaStream_t st) {
  const bool pg = gs > 0;
#define CIDER_GEMV_CASE(I4, P, E)                                                            \
  if (int4 == I4 && pg == P && mode == E)                                                     \
    return launch_one<MB, I4, P, E>(qa, sa, M, N, K, w, sw, gs, y, acc, num_sms, st);
  CIDER_GEMV_CASE(false, false, kEpiY)
  CIDER_GEMV_CASE(false, true, kEpiY)
  CIDER_GEMV_CASE(false, false, kEpiAcc)
  CIDER_GEMV_CASE(false, true, kEpiAcc)
  CIDER_GEMV_CASE(true, false, kEpiY)
  CIDER_GEMV_CASE(true, true, kEpiY)
  CIDER_GEMV_CASE(true, false, kEpiAcc)
  CIDER_GEMV_CASE(true, true, kEpiAcc)
#undef CIDER_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

bool gemv_fits(int64_t M, int64_t K) {
  if (M < 1 || M > 16) return false;
  int64_t mb = 1;
  while (mb < M) mb *= 2;
  return mb * K <= kSmemActMax;
}

cudaError_t launch_gemv(const int8_t* qa, const float* sa, int64_t M, int64_t N, int64_t K,
                        const uint8_t* w, bool int4, const float* sw, int group_size, int mode,
                        __half* y, int32_t* acc, int num_sms, cudaStream_t st) {
  if (M <= 1) return dispatch_mb<1>(qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  if (M <= 2) return dispatch_mb<2>(qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  if (M <= 4) return dispatch_mb<4>(qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  if (M <= 8) return dispatch_mb<8>(qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
  return dispatch_mb<16>(qa, sa, M, N, K, w, int4, sw, group_size, mode, y, acc, num_sms, st);
}

}  // namespace cider
