/*
 * cider_oracle.h -- CPU oracle for the W8A8 / W4A8 online-activation-quantized
 * linear layer.  TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check
 * and the benchmark's CPU-baseline leg, never by the product library.
 *
 * All arrays are dense row-major host memory owned by the caller.
 * fp16 and bf16 values travel as their uint16_t bit patterns.
 */
#ifndef CIDER_ORACLE_H
#define CIDER_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

float oracle_f16_to_f32(uint16_t bits);
uint16_t oracle_f32_to_f16(float f);
uint16_t oracle_f32_to_bf16(float f);

/* x_f16 [M,K] -> qa int8 [M,K], sa fp32 [M] */
void oracle_quantize_act(const uint16_t* x_f16, int64_t M, int64_t K,
                         int8_t* qa, float* sa);
/* the same from x_bf16 [M,K] */
void oracle_quantize_act_bf16(const uint16_t* x_bf16, int64_t M, int64_t K,
                              int8_t* qa, float* sa);

/* W fp32 [N,K] -> qw int8 [N,K], sw fp32 [N, G] (G = 1 when group_size = 0) */
void oracle_quantize_weight_int8(const float* W, int64_t N, int64_t K,
                                 int64_t group_size, int8_t* qw, float* sw);
/* W fp32 [N,K] -> q4 int8 [N,K] holding values in [-8,7], sw fp32 [N, G] */
void oracle_quantize_weight_int4(const float* W, int64_t N, int64_t K,
                                 int64_t group_size, int8_t* q4, float* sw);

/* The same with percentile-clipped scales (clip_percentile in (0, 100]);
 * tmp: scratch of K floats. */
void oracle_quantize_weight_int8_clip(const float* W, int64_t N, int64_t K, int64_t group_size,
                                      double clip_percentile, int8_t* qw, float* sw, float* tmp);
void oracle_quantize_weight_int4_clip(const float* W, int64_t N, int64_t K, int64_t group_size,
                                      double clip_percentile, int8_t* q4, float* sw, float* tmp);

/* q int8 [N,K] with values in [-8,7] <-> packed uint8 [N, K/2] */
void oracle_pack_int4(const int8_t* q, int64_t N, int64_t K, uint8_t* packed);
void oracle_unpack_int4(const uint8_t* packed, int64_t N, int64_t K, int8_t* q);
/* offset-binary INT4 bytes (nibble u = value + 8) -> two's complement bytes */
void oracle_int4_from_offset_binary(const uint8_t* src, int64_t nbytes, uint8_t* dst);

/* acc int32 [M, N, G]; returns 0, or -1 if some sum overflows int32 */
int oracle_gemm_acc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N,
                    int64_t K, int64_t group_size, int32_t* acc);

/* acc [M,N] -> y fp16 [M,N] */
void oracle_dequant_pc(const int32_t* acc, const float* sa, const float* sw,
                       int64_t M, int64_t N, uint16_t* y);
/* acc [M,N,G], sw [N,G] -> y fp16 [M,N] */
void oracle_dequant_pg(const int32_t* acc, const float* sa, const float* sw,
                       int64_t M, int64_t N, int64_t G, uint16_t* y);

/* bf16 outputs */
void oracle_dequant_pc_bf16(const int32_t* acc, const float* sa, const float* sw,
                            int64_t M, int64_t N, uint16_t* y);
void oracle_dequant_pg_bf16(const int32_t* acc, const float* sa, const float* sw,
                            int64_t M, int64_t N, int64_t G, uint16_t* y);

/* rows [m0, m1) of the whole layer; see the .c file */
int oracle_linear_rows(const uint16_t* x_f16, int64_t K, int64_t N,
                       const int8_t* qw, const float* sw, int64_t group_size,
                       int64_t m0, int64_t m1, int8_t* qa_scratch,
                       int32_t* acc_scratch, uint16_t* y);
/* the same with x_bf16 */
int oracle_linear_rows_bf16(const uint16_t* x_bf16, int64_t K, int64_t N,
                            const int8_t* qw, const float* sw, int64_t group_size,
                            int64_t m0, int64_t m1, int8_t* qa_scratch,
                            int32_t* acc_scratch, uint16_t* y);

/* fp16 (x_bf16 = 0) or bf16 activations, fp16 (y_bf16 = 0) or bf16 outputs */
int oracle_linear_rows_ex(const uint16_t* x, int x_bf16, int64_t K, int64_t N,
                          const int8_t* qw, const float* sw, int64_t group_size,
                          int64_t m0, int64_t m1, int8_t* qa_scratch,
                          int32_t* acc_scratch, int y_bf16, uint16_t* y);

#ifdef __cplusplus
}
#endif
#endif
