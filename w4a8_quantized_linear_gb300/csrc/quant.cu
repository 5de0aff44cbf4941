// quant.cu -- per-token activation quantization and offline weight
// quantization kernels.
//
// Activation quantization follows the Cider README (page "cider"),
// "Architecture / Metal kernel pipeline", step quantize_per_token, and the
// "Quantization" table row "Activations: symmetric INT8, per token":
//   s_a = max_k |x[m,k]| / 127 (IEEE fp32 divide; 1 for an all-zero row),
//   q   = clamp(rint(x / s_a), -127, 127) with ties to even.
// Weight quantization follows "Notes" (min-max scales) and the "Quantization"
// table (INT8 per channel or per group of 64 / 128; INT4 for W4A8, "Modes").
// Activations may be fp16 or bf16 (the "auto dtype float16/bfloat16" item of
// the README's roadmap); both widen to fp32 exactly before the same steps.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "cider_device.cuh"
#include "cider_internal.h"

namespace cider {
namespace {

constexpr int kQuantThreads = 128;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float block_max_128(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  v = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  return v;
}

// Code of x for scale s.  fp16 rows use the reciprocal-based correctly rounded
// quotient of act_code (its conditions hold on the fp16 range); bf16 rows
// reach scales down to ~2^-140, where 1/s overflows, so they divide.
template <typename InT>
__device__ __forceinline__ float quant_code(float x, float s, float r) {
  if constexpr (std::is_same<InT, __half>::value) return act_code(x, s, r);
  const float q = rintf(__fdiv_rn(x, s));
  return fminf(fmaxf(q, -127.0f), 127.0f);
}

// Two packed 16-bit activations -> two fp32 values (exact widening).
template <typename InT>
__device__ __forceinline__ float2 widen2(uint32_t w);
template <>
__device__ __forceinline__ float2 widen2<__half>(uint32_t w) {
  __half2 h;
  memcpy(&h, &w, 4);
  return __half22float2(h);
}
template <>
__device__ __forceinline__ float2 widen2<__nv_bfloat16>(uint32_t w) {
  __nv_bfloat162 h;
  memcpy(&h, &w, 4);
  return __bfloat1622float2(h);
}

// max |v| over eight packed activations
template <typename InT>
__device__ __forceinline__ float amax8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float a = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = widen2<InT>(w[j]);
    a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return a;
}

// Eight activations -> eight codes, stored as int8 (8 bytes) or as fp16
// integers (16 bytes; exact, the operand format of the tensor-core GEMM).
template <typename InT>
__device__ __forceinline__ int store_codes(int8_t* q, int64_t off, const uint4& v, float s,
                                           float r) {
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
  uint32_t w[2];
  int l1 = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t b = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float2 f = widen2<InT>(vw[2 * j + e]);
      int c0 = static_cast<int>(quant_code<InT>(f.x, s, r));
      int c1 = static_cast<int>(quant_code<InT>(f.y, s, r));
      l1 += abs(c0) + abs(c1);
      b |= (static_cast<uint32_t>(c0 & 0xFF) << (16 * e)) |
           (static_cast<uint32_t>(c1 & 0xFF) << (16 * e + 8));
    }
    w[j] = b;
  }
  *reinterpret_cast<uint2*>(q + off) = make_uint2(w[0], w[1]);
  return l1;
}
template <typename InT>
__device__ __forceinline__ int store_codes(__half* q, int64_t off, const uint4& v, float s,
                                           float r) {
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
  float l1 = 0.0f;  // a sum of at most 8 codes: exact
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 f = widen2<InT>(vw[j]);
    const float c0 = quant_code<InT>(f.x, s, r), c1 = quant_code<InT>(f.y, s, r);
    l1 += fabsf(c0) + fabsf(c1);
    __half2 r = __floats2half2_rn(c0, c1);
    ow[j] = *reinterpret_cast<uint32_t*>(&r);
  }
  *reinterpret_cast<uint4*>(q + off) = o;
  return static_cast<int>(l1);
}

__device__ __forceinline__ int block_sum_128(int v, int* red) {
  v = __reduce_add_sync(0xffffffffu, v);
  __syncthreads();  // red may still be read by a previous reduction
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  return red[0] + red[1] + red[2] + red[3];
}

// The first CTA clears a small array for the kernel that follows on the
// stream (the GEMM's flags), which saves a separate launch.
__device__ __forceinline__ void clear_words(int* zero, int n) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n; i += blockDim.x) zero[i] = 0;
}

// One CTA of 128 threads per row; the row stays in registers between the
// amax pass and the quantization pass (VPT 16-byte vectors per thread).
template <typename OutT, int VPT, typename InT>
__global__ void __launch_bounds__(kQuantThreads) quant_act_kernel(const InT* __restrict__ x,
                                                                  int64_t K, OutT* __restrict__ q,
                                                                  float* __restrict__ sa,
                                                                  int* __restrict__ row_l1,
                                                                  int* __restrict__ zero,
                                                                  int zero_words, bool release) {
  __shared__ float red[4];
  __shared__ int ired[4];
  const int64_t m = blockIdx.x;
  // the library's GEMM / GEMV launched next may start its set-up now
  if (release) pdl_launch_dependents();
  clear_words(zero, zero_words);
  const uint4* row = reinterpret_cast<const uint4*>(x + m * K);
  const int nvec = static_cast<int>(K >> 3);
  uint4 v[VPT];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * kQuantThreads;
    if (idx < nvec) {
      v[i] = ld_stream_v4(row + idx);
      amax = fmaxf(amax, amax8<InT>(v[i]));
    }
  }
  amax = block_max_128(amax, red);
  const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
  const float r = __frcp_rn(s);
  if (threadIdx.x == 0) sa[m] = s;
  int l1 = 0;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * kQuantThreads;
    if (idx < nvec) l1 += store_codes<InT>(q, m * K + static_cast<int64_t>(idx) * 8, v[i], s, r);
  }
  if (row_l1 != nullptr) {
    l1 = block_sum_128(l1, ired);
    if (threadIdx.x == 0) row_l1[m] = l1;
  }
}

// Rows longer than the register-resident variants: two passes over global
// memory (the second pass hits L1/L2).
template <typename OutT, typename InT>
__global__ void __launch_bounds__(kQuantThreads) quant_act_long_kernel(const InT* __restrict__ x,
                                                                       int64_t K,
                                                                       OutT* __restrict__ q,
                                                                       float* __restrict__ sa,
                                                                       int* __restrict__ row_l1,
                                                                       int* __restrict__ zero,
                                                                       int zero_words, bool release) {
  __shared__ float red[4];
  __shared__ int ired[4];
  const int64_t m = blockIdx.x;
  if (release) pdl_launch_dependents();
  clear_words(zero, zero_words);
  const uint4* row = reinterpret_cast<const uint4*>(x + m * K);
  const int64_t nvec = K >> 3;
  float amax = 0.0f;
  for (int64_t idx = threadIdx.x; idx < nvec; idx += kQuantThreads) amax = fmaxf(amax, amax8<InT>(row[idx]));
  amax = block_max_128(amax, red);
  const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
  const float r = __frcp_rn(s);
  if (threadIdx.x == 0) sa[m] = s;
  int l1 = 0;
  for (int64_t idx = threadIdx.x; idx < nvec; idx += kQuantThreads)
    l1 += store_codes<InT>(q, m * K + idx * 8, row[idx], s, r);
  if (row_l1 != nullptr) {
    l1 = block_sum_128(l1, ired);
    if (threadIdx.x == 0) row_l1[m] = l1;
  }
}

template <typename OutT, typename InT>
cudaError_t launch_quant_act(const InT* x, int64_t M, int64_t K, OutT* q, float* sa,
                             int* row_l1, int* zero, int zero_words, cudaStream_t st, bool release) {
  const int64_t nvec = K / 8;
  const int vpt = static_cast<int>((nvec + kQuantThreads - 1) / kQuantThreads);
  const dim3 grid(static_cast<unsigned>(M));
  if (vpt <= 1)
    quant_act_kernel<OutT, 1, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 2)
    quant_act_kernel<OutT, 2, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 3)
    quant_act_kernel<OutT, 3, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 4)
    quant_act_kernel<OutT, 4, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 6)
    quant_act_kernel<OutT, 6, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 8)
    quant_act_kernel<OutT, 8, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 12)
    quant_act_kernel<OutT, 12, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else if (vpt <= 16)
    quant_act_kernel<OutT, 16, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  else
    quant_act_long_kernel<OutT, InT><<<grid, kQuantThreads, 0, st>>>(x, K, q, sa, row_l1, zero, zero_words, release);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- weights
// One warp per (row, block): block = the whole row (per channel) or
// group_size consecutive elements (per group).  Each lane takes element
// pairs (2j, 2j+1) so the INT4 variant writes whole packed bytes.
template <bool INT4>
__global__ void __launch_bounds__(256) quant_weight_kernel(const float* __restrict__ w, int64_t N,
                                                           int64_t K, int64_t bs, int64_t G,
                                                           uint8_t* __restrict__ q,
                                                           float* __restrict__ sw) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (blk >= N * G) return;
  const int64_t n = blk / G, g = blk % G;
  const float2* src = reinterpret_cast<const float2*>(w + n * K + g * bs);
  const int64_t npairs = bs / 2;
  float amax = 0.0f;
  for (int64_t j = lane; j < npairs; j += 32) {
    float2 v = src[j];
    amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
  }
  amax = warp_max(amax);
  const float qdiv = INT4 ? 7.0f : 127.0f;
  const float qmin = INT4 ? -8.0f : -127.0f;
  const float qmax = INT4 ? 7.0f : 127.0f;
  const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, qdiv);
  if (lane == 0) sw[n * G + g] = s;
  for (int64_t j = lane; j < npairs; j += 32) {
    float2 v = src[j];
    int c0 = static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(v.x, s)), qmin), qmax));
    int c1 = static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(v.y, s)), qmin), qmax));
    if (INT4) {
      q[n * (K / 2) + g * (bs / 2) + j] =
          static_cast<uint8_t>((c0 & 0xF) | ((c1 & 0xF) << 4));
    } else {
      uint8_t* dst = q + n * K + g * bs + 2 * j;
      *reinterpret_cast<uint16_t*>(dst) =
          static_cast<uint16_t>((c0 & 0xFF) | ((c1 & 0xFF) << 8));
    }
  }
}

// ---------------------------------------------------------------- clipped weight scales
// Percentile-clipped weight scales (Cider README, "Notes": min-max scales by
// default, or a percentile, clip_percentile = 99.9).  For a block of n
// values, the clip is the p-th percentile of |W| with linear interpolation
// between the order statistics lo and hi = lo + 1 at the fractional rank
// (n - 1) p / 100 (lo, hi and the weight t come from the host, in double);
// clip = a_lo + t (a_hi - a_lo) in fp32 without FMA, s = clip / qmax (1 when
// clip == 0), and codes clamp as for min-max scales.

// Scale and codes of one block given its clip value; `src` holds the block's
// bs values, element pairs (2j, 2j + 1) go to lanes / threads j (mod `step`).
template <bool INT4>
__device__ __forceinline__ float clipped_scale(float alo, float ahi, float t) {
  const float clip = __fadd_rn(alo, __fmul_rn(t, __fsub_rn(ahi, alo)));
  return (clip == 0.0f) ? 1.0f : __fdiv_rn(clip, INT4 ? 7.0f : 127.0f);
}

template <bool INT4>
__device__ __forceinline__ void store_block_codes(const float* src, int64_t bs, float s, int64_t first,
                                                  int64_t step, uint8_t* q_row, int64_t off) {
  const float qmin = INT4 ? -8.0f : -127.0f;
  const float qmax = INT4 ? 7.0f : 127.0f;
  const float2* src2 = reinterpret_cast<const float2*>(src);
  for (int64_t j = first; j < bs / 2; j += step) {
    const float2 v = src2[j];
    const int c0 = static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(v.x, s)), qmin), qmax));
    const int c1 = static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(v.y, s)), qmin), qmax));
    if (INT4) {
      q_row[off / 2 + j] = static_cast<uint8_t>((c0 & 0xF) | ((c1 & 0xF) << 4));
    } else {
      *reinterpret_cast<uint16_t*>(q_row + off + 2 * j) =
          static_cast<uint16_t>((c0 & 0xFF) | ((c1 & 0xFF) << 8));
    }
  }
}

// Per group (GS = 64 or 128 values): one warp per block.  Each element's
// rank is the number of block values below it (ties broken by position), so
// exactly one element has each rank.
template <bool INT4, int GS>
__global__ void __launch_bounds__(256) quant_weight_clip_group_kernel(
    const float* __restrict__ w, int64_t N, int64_t K, int64_t G, int lo, int hi, float t,
    uint8_t* __restrict__ q, float* __restrict__ sw) {
  constexpr int PER = GS / 32;
  const int lane = threadIdx.x & 31;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (blk >= N * G) return;   // uniform per warp
  const int64_t n = blk / G, g = blk % G;
  const float* src = w + n * K + g * GS;
  float v[PER];
  int rank[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    v[j] = fabsf(src[lane + 32 * j]);
    rank[j] = 0;
  }
#pragma unroll
  for (int j2 = 0; j2 < PER; ++j2)
    for (int l = 0; l < 32; ++l) {
      const float o = __shfl_sync(0xffffffffu, v[j2], l);
      const int oi = l + 32 * j2;
#pragma unroll
      for (int j = 0; j < PER; ++j)
        rank[j] += (o < v[j] || (o == v[j] && oi < lane + 32 * j)) ? 1 : 0;
    }
  float alo = -1.0f, ahi = -1.0f;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if (rank[j] == lo) alo = v[j];
    if (rank[j] == hi) ahi = v[j];
  }
  alo = warp_max(alo);
  ahi = warp_max(ahi);
  const float s = clipped_scale<INT4>(alo, ahi, t);
  if (lane == 0) sw[n * G + g] = s;
  store_block_codes<INT4>(src, GS, s, lane, 32, q + n * (INT4 ? K / 2 : K), g * GS);
}

// Per channel (a whole row of K values): one CTA per row; a radix select over
// the bit patterns of |w| (non-negative floats order like unsigned integers),
// 8 bits per pass, finds the value of rank lo; the value of rank hi is the
// same when more than lo + 1 values are <= it, else the smallest value above.
constexpr int kClipThreads = 256;

template <bool INT4>
__global__ void __launch_bounds__(kClipThreads) quant_weight_clip_row_kernel(
    const float* __restrict__ w, int64_t K, int64_t lo, int64_t hi, float t,
    uint8_t* __restrict__ q, float* __restrict__ sw) {
  __shared__ unsigned hist[256];
  __shared__ uint32_t s_bucket;
  __shared__ unsigned long long s_rest;
  __shared__ unsigned long long s_cnt[kClipThreads / 32];
  __shared__ uint32_t s_min[kClipThreads / 32];
  const int64_t n = blockIdx.x;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(w + n * K);
  uint32_t prefix = 0u, mask = 0u;
  unsigned long long k = static_cast<unsigned long long>(lo);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kClipThreads) hist[i] = 0u;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < K; i += kClipThreads) {
      const uint32_t b = row[i] & 0x7FFFFFFFu;
      if ((b & mask) == prefix) atomicAdd(&hist[(b >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long cum = 0;
      uint32_t d = 0;
      for (; d < 255u; ++d) {
        if (cum + hist[d] > k) break;
        cum += hist[d];
      }
      s_bucket = d;
      s_rest = k - cum;
    }
    __syncthreads();
    prefix |= s_bucket << shift;
    mask |= 0xFFu << shift;
    k = s_rest;
    __syncthreads();
  }
  const float alo = __uint_as_float(prefix);
  float ahi = alo;
  if (hi != lo) {
    unsigned long long le = 0;
    uint32_t above = 0xFFFFFFFFu;
    for (int64_t i = threadIdx.x; i < K; i += kClipThreads) {
      const uint32_t b = row[i] & 0x7FFFFFFFu;
      if (b <= prefix) ++le;
      else above = min(above, b);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      le += __shfl_xor_sync(0xffffffffu, le, o);
      above = min(above, __shfl_xor_sync(0xffffffffu, above, o));
    }
    if ((threadIdx.x & 31) == 0) {
      s_cnt[threadIdx.x >> 5] = le;
      s_min[threadIdx.x >> 5] = above;
    }
    __syncthreads();
    le = 0;
    above = 0xFFFFFFFFu;
    for (int i = 0; i < kClipThreads / 32; ++i) {
      le += s_cnt[i];
      above = min(above, s_min[i]);
    }
    if (le <= static_cast<unsigned long long>(lo) + 1) ahi = __uint_as_float(above);
  }
  const float s = clipped_scale<INT4>(alo, ahi, t);
  if (threadIdx.x == 0) sw[n] = s;
  store_block_codes<INT4>(w + n * K, K, s, threadIdx.x, kClipThreads, q + n * (INT4 ? K / 2 : K), 0);
}

// int8 codes -> the same codes as fp16 integers (exact), one CTA per row,
// plus the row's sum of |code|.
__global__ void __launch_bounds__(kQuantThreads) codes_s8_to_f16_kernel(const int8_t* __restrict__ qa,
                                                                        int64_t K,
                                                                        __half* __restrict__ out,
                                                                        int* __restrict__ row_l1,
                                                                        int* __restrict__ zero,
                                                                        int zero_words) {
  __shared__ int ired[4];
  const int64_t m = blockIdx.x;
  pdl_launch_dependents();
  clear_words(zero, zero_words);
  const int64_t n16 = K / 16;
  int l1 = 0;
  for (int64_t i = threadIdx.x; i < n16; i += kQuantThreads) {
    const uint4 v = ld_stream_v4(qa + m * K + i * 16);
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int b0 = static_cast<int8_t>(vw[j] & 0xFF), b1 = static_cast<int8_t>((vw[j] >> 8) & 0xFF);
      const int b2 = static_cast<int8_t>((vw[j] >> 16) & 0xFF), b3 = static_cast<int8_t>(vw[j] >> 24);
      l1 += abs(b0) + abs(b1) + abs(b2) + abs(b3);
    }
    uint4 o0, o1;
    s8x4_to_h2x2(v.x, o0.x, o0.y);
    s8x4_to_h2x2(v.y, o0.z, o0.w);
    s8x4_to_h2x2(v.z, o1.x, o1.y);
    s8x4_to_h2x2(v.w, o1.z, o1.w);
    uint4* dst = reinterpret_cast<uint4*>(out + m * K + i * 16);
    dst[0] = o0;
    dst[1] = o1;
  }
  l1 = block_sum_128(l1, ired);
  if (threadIdx.x == 0) row_l1[m] = l1;
}

// Offset-binary INT4 (each nibble u holds the value u - 8: the "zp = 8" form
// of the README's "Quantization" table) -> the library's two's complement
// nibbles, (u - 8) mod 16 = u ^ 8 in each nibble.  16 bytes per thread and
// step; the last n % 16 bytes one at a time.
__global__ void __launch_bounds__(256) int4_from_offset_kernel(const uint8_t* src,
                                                               uint8_t* dst,
                                                               int64_t n) {
  const int64_t n16 = n / 16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16; i += stride) {
    uint4 v = reinterpret_cast<const uint4*>(src)[i];
    v.x ^= 0x88888888u;
    v.y ^= 0x88888888u;
    v.z ^= 0x88888888u;
    v.w ^= 0x88888888u;
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
  for (int64_t i = n16 * 16 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += stride)
    dst[i] = static_cast<uint8_t>(src[i] ^ 0x88u);
}

}  // namespace

cudaError_t launch_int4_from_offset(const uint8_t* src, uint8_t* dst, int64_t nbytes,
                                    cudaStream_t st) {
  const int64_t n16 = (nbytes + 15) / 16;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  int4_from_offset_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(src, dst, nbytes);
  return cudaGetLastError();
}

cudaError_t launch_quant_act_s8(const __half* x, int64_t M, int64_t K, int8_t* q, float* sa,
                                cudaStream_t st, bool release) {
  return launch_quant_act<int8_t, __half>(x, M, K, q, sa, nullptr, nullptr, 0, st, release);
}

cudaError_t launch_quant_act_s8_bf16(const __nv_bfloat16* x, int64_t M, int64_t K, int8_t* q,
                                     float* sa, cudaStream_t st, bool release) {
  return launch_quant_act<int8_t, __nv_bfloat16>(x, M, K, q, sa, nullptr, nullptr, 0, st, release);
}

cudaError_t launch_quant_act_f16(const __half* x, int64_t M, int64_t K, __half* q, float* sa,
                                 int* row_l1, int* zero, int zero_words, cudaStream_t st,
                                 bool release) {
  return launch_quant_act<__half, __half>(x, M, K, q, sa, row_l1, zero, zero_words, st, release);
}

cudaError_t launch_quant_act_f16_from_bf16(const __nv_bfloat16* x, int64_t M, int64_t K, __half* q,
                                           float* sa, int* row_l1, int* zero, int zero_words,
                                           cudaStream_t st, bool release) {
  return launch_quant_act<__half, __nv_bfloat16>(x, M, K, q, sa, row_l1, zero, zero_words, st,
                                                 release);
}

cudaError_t launch_quant_weight(const float* w, int64_t N, int64_t K, int group_size, bool int4,
                                uint8_t* q, float* sw, cudaStream_t st) {
  const int64_t bs = group_size > 0 ? group_size : K;
  const int64_t G = K / bs;
  const int64_t blocks = (N * G + 7) / 8;
  if (int4)
    quant_weight_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(w, N, K, bs, G, q, sw);
  else
    quant_weight_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(w, N, K, bs, G, q, sw);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight_clip(const float* w, int64_t N, int64_t K, int group_size,
                                     double clip_percentile, bool int4, uint8_t* q, float* sw,
                                     cudaStream_t st) {
  const int64_t bs = group_size > 0 ? group_size : K;
  const int64_t G = K / bs;
  // fractional rank of the percentile in a block of bs values (in double, as
  // the definition states), its two order statistics and the fp32 weight
  const double h = static_cast<double>(bs - 1) * clip_percentile / 100.0;
  int64_t lo = static_cast<int64_t>(floor(h));
  if (lo > bs - 1) lo = bs - 1;
  const int64_t hi = lo + 1 < bs ? lo + 1 : bs - 1;
  const float t = static_cast<float>(h - static_cast<double>(lo));
  if (group_size == 0) {
    if (int4)
      quant_weight_clip_row_kernel<true><<<static_cast<unsigned>(N), kClipThreads, 0, st>>>(
          w, K, lo, hi, t, q, sw);
    else
      quant_weight_clip_row_kernel<false><<<static_cast<unsigned>(N), kClipThreads, 0, st>>>(
          w, K, lo, hi, t, q, sw);
    return cudaGetLastError();
  }
  const unsigned blocks = static_cast<unsigned>((N * G + 7) / 8);
  const int l = static_cast<int>(lo), h2 = static_cast<int>(hi);
  if (group_size == 64) {
    if (int4)
      quant_weight_clip_group_kernel<true, 64><<<blocks, 256, 0, st>>>(w, N, K, G, l, h2, t, q, sw);
    else
      quant_weight_clip_group_kernel<false, 64><<<blocks, 256, 0, st>>>(w, N, K, G, l, h2, t, q, sw);
  } else {
    if (int4)
      quant_weight_clip_group_kernel<true, 128><<<blocks, 256, 0, st>>>(w, N, K, G, l, h2, t, q, sw);
    else
      quant_weight_clip_group_kernel<false, 128><<<blocks, 256, 0, st>>>(w, N, K, G, l, h2, t, q, sw);
  }
  return cudaGetLastError();
}

cudaError_t launch_codes_s8_to_f16(const int8_t* qa, int64_t M, int64_t K, __half* out,
                                   int* row_l1, int* zero, int zero_words, cudaStream_t st) {
  codes_s8_to_f16_kernel<<<static_cast<unsigned>(M), kQuantThreads, 0, st>>>(qa, K, out, row_l1,
                                                                              zero, zero_words);
  return cudaGetLastError();
}

}  // namespace cider
