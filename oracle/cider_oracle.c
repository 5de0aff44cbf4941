/*
 * cider_oracle.c -- plain, slow, single-threaded CPU oracle for the
 * online-activation-quantized linear layer (W8A8 / W4A8).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) may include, link or call this file; only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark do.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * What it computes, and where that is defined (Cider README, page "cider"):
 *   - "Quantization" table: activations symmetric INT8 per token; weights
 *     symmetric INT8 per channel or per group (gs = 64/128); INT32
 *     accumulation; output dequant C_fp16 = C_int32 * s_act * s_weight.
 *   - "Architecture / Metal kernel pipeline": quantize_per_token (fp16 -> int8
 *     + per-token scale), then INT8 x INT8 -> INT32 -> FP16 with the scales
 *     fused into the store.
 *   - "Notes": weight scales are min-max (max |W| / qmax).
 *   - "W8A8 quantization granularity": per-group = one scale per gs
 *     consecutive input elements.
 *   - "Modes": W4A8 weights are INT4 packed two per uint8.
 * Readings where the page is silent (all listed with the design notes):
 *   - round-half-even (nearbyintf in the default rounding mode), IEEE binary32
 *     division x / s (never a reciprocal multiply), clamp to [-127, 127];
 *   - amax == 0 gives s = 1 and q = 0 (activations and weight blocks alike);
 *   - INT4: s = max|W| / 7, q = clamp(rint(W / s), -8, 7), two's complement
 *     nibbles, element 2j in the low nibble of byte j, 2j+1 in the high one;
 *   - per-group dequant: s = 0; for g = 0..G-1 in increasing order
 *     s += (s_a * s_w[n,g]) * (float)acc_g; y = (fp16)s;
 *   - per-channel dequant evaluated left to right: ((float)acc * s_a) * s_w.
 * Compile with -O2 -ffp-contract=off (no FMA contraction) and without any
 * fast-math flag.  fp16 <-> fp32 conversions use the compiler's _Float16 type
 * (IEEE binary16, round-to-nearest-even on narrowing).
 */
#include "cider_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- fp16 helpers (library conversions, no arithmetic of the method) ---- */

static float f16_bits_to_f32(uint16_t bits) {
  _Float16 h;
  memcpy(&h, &bits, sizeof h);
  return (float)h;
}

static uint16_t f32_to_f16_bits(float f) {
  _Float16 h = (_Float16)f; /* IEEE round-to-nearest-even, overflow -> inf */
  uint16_t bits;
  memcpy(&bits, &h, sizeof bits);
  return bits;
}

/* bf16 is the upper half of an IEEE binary32: widening appends 16 zero bits. */
static float bf16_bits_to_f32(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return f;
}

/* fp32 -> bf16 bit pattern, round to nearest with ties to even on the 16
 * bits dropped from the binary32 (so values past the bf16 range round to
 * +-inf); NaN stays a quiet NaN.  Written from the definition of the bf16
 * format: the upper half of a binary32. */
static uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

float oracle_f16_to_f32(uint16_t bits) { return f16_bits_to_f32(bits); }
uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_bits(f); }
uint16_t oracle_f32_to_f16(float f) { return f32_to_f16_bits(f); }

/* ---- symmetric quantization of one block (shared by a1 and a2) ----
 * Cider README "Quantization" table (symmetric, min-max per "Notes").
 * scale = amax / qdiv (IEEE fp32 divide); amax == 0 -> scale = 1.
 * q = clamp(rint(v / scale), qmin, qmax), rint = round-half-even. */
static float block_scale(float amax, float qdiv) {
  return (amax == 0.0f) ? 1.0f : amax / qdiv;
}

static int quantize_value(float v, float scale, int qmin, int qmax) {
  float r = nearbyintf(v / scale);
  if (r < (float)qmin) r = (float)qmin;
  if (r > (float)qmax) r = (float)qmax;
  return (int)r;
}

/* a1: per-token activation quantization (Cider README, "Metal kernel
 * pipeline" step quantize_per_token; "Quantization" row "Activations").
 * `widen` turns one stored activation into its exact fp32 value. */
static void quantize_act_rows(const uint16_t* x, int64_t M, int64_t K,
                              float (*widen)(uint16_t), int8_t* qa, float* sa) {
  for (int64_t m = 0; m < M; ++m) {
    const uint16_t* row = x + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(widen(row[k]));
      if (a > amax) amax = a;
    }
    float s = block_scale(amax, 127.0f);
    sa[m] = s;
    for (int64_t k = 0; k < K; ++k)
      qa[m * K + k] = (int8_t)quantize_value(widen(row[k]), s, -127, 127);
  }
}

void oracle_quantize_act(const uint16_t* x_f16, int64_t M, int64_t K,
                         int8_t* qa, float* sa) {
  quantize_act_rows(x_f16, M, K, f16_bits_to_f32, qa, sa);
}

/* The same for bf16 activations (the README's roadmap: "auto dtype
 * float16/bfloat16"). */
void oracle_quantize_act_bf16(const uint16_t* x_bf16, int64_t M, int64_t K,
                              int8_t* qa, float* sa) {
  quantize_act_rows(x_bf16, M, K, bf16_bits_to_f32, qa, sa);
}

/* a2: symmetric weight quantization, per output channel (group_size = 0) or
 * per group of group_size consecutive K elements (Cider README,
 * "Quantization" row "W8A8 weights" and "W8A8 quantization granularity").
 * qdiv = 127, range [-127,127] for INT8; qdiv = 7, range [-8,7] for INT4. */
static void quantize_weight(const float* W, int64_t N, int64_t K,
                            int64_t group_size, float qdiv, int qmin, int qmax,
                            int8_t* q, float* sw) {
  int64_t gs = group_size > 0 ? group_size : K;
  int64_t G = K / gs;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < G; ++g) {
      const float* blk = W + n * K + g * gs;
      float amax = 0.0f;
      for (int64_t j = 0; j < gs; ++j) {
        float a = fabsf(blk[j]);
        if (a > amax) amax = a;
      }
      float s = block_scale(amax, qdiv);
      sw[n * G + g] = s;
      for (int64_t j = 0; j < gs; ++j)
        q[n * K + g * gs + j] = (int8_t)quantize_value(blk[j], s, qmin, qmax);
    }
  }
}

/* a2, percentile-clipped scales (Cider README "Notes": scales are min-max by
 * default, or from a percentile with clip_percentile = 99.9).  Reading: the
 * block's |W| values sorted ascending a_0 <= ... <= a_{n-1}; the p-th
 * percentile with linear interpolation between closest ranks, at the
 * fractional rank h = (n - 1) p / 100 (in double): lo = floor(h),
 * hi = min(lo + 1, n - 1), t = (float)(h - lo) and
 * clip = a_lo + t * (a_hi - a_lo) in fp32 (three roundings, no FMA).  The
 * scale is clip / qdiv (1 when clip == 0) and codes clamp as for min-max, so
 * values above clip saturate; p = 100 gives exactly the min-max result. */
static int cmp_float(const void* a, const void* b) {
  const float x = *(const float*)a, y = *(const float*)b;
  return (x > y) - (x < y);
}

static float clipped_max(const float* blk, int64_t n, double p, float* tmp) {
  for (int64_t j = 0; j < n; ++j) tmp[j] = fabsf(blk[j]);
  qsort(tmp, (size_t)n, sizeof(float), cmp_float);
  const double h = (double)(n - 1) * p / 100.0;
  int64_t lo = (int64_t)floor(h);
  if (lo > n - 1) lo = n - 1;
  const int64_t hi = lo + 1 < n ? lo + 1 : n - 1;
  const float t = (float)(h - (double)lo);
  const float d = tmp[hi] - tmp[lo];
  const float td = t * d;
  return tmp[lo] + td;
}

static void quantize_weight_clip(const float* W, int64_t N, int64_t K, int64_t group_size,
                                 double p, float qdiv, int qmin, int qmax, int8_t* q,
                                 float* sw, float* tmp) {
  int64_t gs = group_size > 0 ? group_size : K;
  int64_t G = K / gs;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      const float* blk = W + n * K + g * gs;
      float s = block_scale(clipped_max(blk, gs, p, tmp), qdiv);
      sw[n * G + g] = s;
      for (int64_t j = 0; j < gs; ++j)
        q[n * K + g * gs + j] = (int8_t)quantize_value(blk[j], s, qmin, qmax);
    }
}

/* tmp: scratch of K floats */
void oracle_quantize_weight_int8_clip(const float* W, int64_t N, int64_t K, int64_t group_size,
                                      double clip_percentile, int8_t* qw, float* sw, float* tmp) {
  quantize_weight_clip(W, N, K, group_size, clip_percentile, 127.0f, -127, 127, qw, sw, tmp);
}

void oracle_quantize_weight_int4_clip(const float* W, int64_t N, int64_t K, int64_t group_size,
                                      double clip_percentile, int8_t* q4, float* sw, float* tmp) {
  quantize_weight_clip(W, N, K, group_size, clip_percentile, 7.0f, -8, 7, q4, sw, tmp);
}

void oracle_quantize_weight_int8(const float* W, int64_t N, int64_t K,
                                 int64_t group_size, int8_t* qw, float* sw) {
  quantize_weight(W, N, K, group_size, 127.0f, -127, 127, qw, sw);
}

void oracle_quantize_weight_int4(const float* W, int64_t N, int64_t K,
                                 int64_t group_size, int8_t* q4, float* sw) {
  quantize_weight(W, N, K, group_size, 7.0f, -8, 7, q4, sw);
}

/* a2/a4: INT4 packing, two per uint8 (Cider README "Modes": "INT4 packed
 * (uint8)"); reading: two's complement nibbles, even element low. */
void oracle_pack_int4(const int8_t* q, int64_t N, int64_t K, uint8_t* packed) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t j = 0; j < K / 2; ++j) {
      unsigned lo = (unsigned)(q[n * K + 2 * j] & 0xF);
      unsigned hi = (unsigned)(q[n * K + 2 * j + 1] & 0xF);
      packed[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
    }
}

/* Nibble -> signed value: a 4-bit two's complement number t in [0,15] is t
 * when t < 8 and t - 16 otherwise. */
static int nibble_value(unsigned t) { return (t < 8u) ? (int)t : (int)t - 16; }

/* Offset-binary INT4 ("Symmetric INT4 (zp=8)", README "Quantization" table):
 * nibble u in [0,15] holds the value u - 8.  Re-encode every byte's two
 * values as two's complement nibbles, low nibble first as in the packing. */
void oracle_int4_from_offset_binary(const uint8_t* src, int64_t nbytes, uint8_t* dst) {
  for (int64_t i = 0; i < nbytes; ++i) {
    int lo = (int)(src[i] & 0xFu) - 8;
    int hi = (int)(src[i] >> 4) - 8;
    dst[i] = (uint8_t)(((unsigned)lo & 0xFu) | (((unsigned)hi & 0xFu) << 4));
  }
}

void oracle_unpack_int4(const uint8_t* packed, int64_t N, int64_t K, int8_t* q) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t j = 0; j < K / 2; ++j) {
      unsigned b = packed[n * (K / 2) + j];
      q[n * K + 2 * j] = (int8_t)nibble_value(b & 0xFu);
      q[n * K + 2 * j + 1] = (int8_t)nibble_value(b >> 4);
    }
}

/* a3: integer GEMM with INT32 accumulation (Cider README "Quantization" row
 * "Accumulation: INT32").  acc[(m*N + n)*G + g] = sum over k in group g of
 * qa[m,k] * qw[n,k], summed in int64 and then checked to fit in int32.
 * group_size = 0 means a single group spanning K.  Returns 0, or -1 when a
 * sum does not fit in int32. */
int oracle_gemm_acc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N,
                    int64_t K, int64_t group_size, int32_t* acc) {
  int64_t gs = group_size > 0 ? group_size : K;
  int64_t G = K / gs;
  int status = 0;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t g = 0; g < G; ++g) {
        int64_t s = 0;
        for (int64_t j = 0; j < gs; ++j) {
          int64_t k = g * gs + j;
          s += (int64_t)qa[m * K + k] * (int64_t)qw[n * K + k];
        }
        if (s > INT32_MAX || s < INT32_MIN) status = -1;
        acc[(m * N + n) * G + g] = (int32_t)s;
      }
  return status;
}

/* a5: per-channel dequant, C_fp16 = C_int32 * s_act * s_weight (Cider README
 * "Quantization" row "Output dequant"), evaluated left to right in fp32 and
 * rounded once to the output format (fp16, or bf16: the README roadmap's
 * "auto dtype float16/bfloat16"). */
static void dequant_pc(const int32_t* acc, const float* sa, const float* sw, int64_t M, int64_t N,
                       uint16_t (*narrow)(float), uint16_t* y) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      float v = (float)acc[m * N + n];
      v = v * sa[m];
      v = v * sw[n];
      y[m * N + n] = narrow(v);
    }
}

/* a5: per-group dequant: fp32 sum over groups in increasing g of
 * (s_a * s_w[n,g]) * acc_g, then one rounding to the output format. */
static void dequant_pg(const int32_t* acc, const float* sa, const float* sw, int64_t M, int64_t N,
                       int64_t G, uint16_t (*narrow)(float), uint16_t* y) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      float s = 0.0f;
      for (int64_t g = 0; g < G; ++g) {
        float scale = sa[m] * sw[n * G + g];
        float term = scale * (float)acc[(m * N + n) * G + g];
        s = s + term;
      }
      y[m * N + n] = narrow(s);
    }
}

void oracle_dequant_pc(const int32_t* acc, const float* sa, const float* sw,
                       int64_t M, int64_t N, uint16_t* y) {
  dequant_pc(acc, sa, sw, M, N, f32_to_f16_bits, y);
}

void oracle_dequant_pg(const int32_t* acc, const float* sa, const float* sw,
                       int64_t M, int64_t N, int64_t G, uint16_t* y) {
  dequant_pg(acc, sa, sw, M, N, G, f32_to_f16_bits, y);
}

void oracle_dequant_pc_bf16(const int32_t* acc, const float* sa, const float* sw,
                            int64_t M, int64_t N, uint16_t* y) {
  dequant_pc(acc, sa, sw, M, N, f32_to_bf16_bits, y);
}

void oracle_dequant_pg_bf16(const int32_t* acc, const float* sa, const float* sw,
                            int64_t M, int64_t N, int64_t G, uint16_t* y) {
  dequant_pg(acc, sa, sw, M, N, G, f32_to_bf16_bits, y);
}

/* The whole layer for activation rows [m0, m1): quantize those rows, form the
 * integer accumulators, dequantize.  qw holds unpacked weight values (INT8, or
 * INT4 values after oracle_unpack_int4).  group_size = 0 -> per-channel.
 * y receives (m1 - m0) rows of N fp16 (or bf16) values.  acc_scratch must
 * hold N * G int32; qa_scratch K int8.  Returns the GEMM status. */
static int linear_rows(const uint16_t* x, float (*widen)(uint16_t), int64_t K, int64_t N,
                       const int8_t* qw, const float* sw, int64_t group_size,
                       int64_t m0, int64_t m1, int8_t* qa_scratch,
                       int32_t* acc_scratch, uint16_t (*narrow)(float), uint16_t* y) {
  int64_t G = group_size > 0 ? K / group_size : 1;
  int status = 0;
  for (int64_t m = m0; m < m1; ++m) {
    float sa;
    quantize_act_rows(x + m * K, 1, K, widen, qa_scratch, &sa);
    if (oracle_gemm_acc(qa_scratch, qw, 1, N, K, group_size, acc_scratch) != 0)
      status = -1;
    uint16_t* yrow = y + (m - m0) * N;
    if (group_size > 0)
      dequant_pg(acc_scratch, &sa, sw, 1, N, G, narrow, yrow);
    else
      dequant_pc(acc_scratch, &sa, sw, 1, N, narrow, yrow);
  }
  return status;
}

int oracle_linear_rows(const uint16_t* x_f16, int64_t K, int64_t N,
                       const int8_t* qw, const float* sw, int64_t group_size,
                       int64_t m0, int64_t m1, int8_t* qa_scratch,
                       int32_t* acc_scratch, uint16_t* y) {
  return linear_rows(x_f16, f16_bits_to_f32, K, N, qw, sw, group_size, m0, m1, qa_scratch,
                     acc_scratch, f32_to_f16_bits, y);
}

int oracle_linear_rows_bf16(const uint16_t* x_bf16, int64_t K, int64_t N,
                            const int8_t* qw, const float* sw, int64_t group_size,
                            int64_t m0, int64_t m1, int8_t* qa_scratch,
                            int32_t* acc_scratch, uint16_t* y) {
  return linear_rows(x_bf16, bf16_bits_to_f32, K, N, qw, sw, group_size, m0, m1, qa_scratch,
                     acc_scratch, f32_to_f16_bits, y);
}

int oracle_linear_rows_ex(const uint16_t* x, int x_bf16, int64_t K, int64_t N,
                          const int8_t* qw, const float* sw, int64_t group_size,
                          int64_t m0, int64_t m1, int8_t* qa_scratch,
                          int32_t* acc_scratch, int y_bf16, uint16_t* y) {
  return linear_rows(x, x_bf16 ? bf16_bits_to_f32 : f16_bits_to_f32, K, N, qw, sw, group_size,
                     m0, m1, qa_scratch, acc_scratch, y_bf16 ? f32_to_bf16_bits : f32_to_f16_bits,
                     y);
}
