/*
 * cider.h -- C ABI of the GB300 (sm_103a) online-activation-quantized linear
 * layer, W8A8 and W4A8.
 *
 * Operation (Cider README, page "cider"):
 *   "Quantization" table -- activations symmetric INT8 per token; weights
 *   symmetric INT8 per channel or per group (gs = 64 / 128), or INT4 packed two
 *   per uint8 ("Modes" table, W4A8); INT32 accumulation; output dequant
 *   C_fp16 = C_int32 * s_act * s_weight.
 *   "Architecture / Metal kernel pipeline" -- quantize_per_token (fp16 ->
 *   INT8 + per-token scale), then INT8 x INT8 -> INT32 -> FP16 with the scales
 *   applied in the store.
 *   "Low-level API" -- perchannel_linear(x, w_int8, scale) and
 *   w4a8_linear(x, packed_w4, scale4) return fp16; quantize_weight_int8 and
 *   pack_weight_int4 prepare weights.
 * Precise definitions used here (the page leaves them open):
 *   s_a[m] = max_k |x[m,k]| / 127 in fp32 (IEEE divide), 1 when the row is 0;
 *   q_a[m,k] = clamp(rint(x[m,k] / s_a[m]), -127, 127), ties to even;
 *   acc[m,n,g] = sum_{k in group g} q_a[m,k] * q_w[n,k]   (exact integer);
 *   per channel: y[m,n] = fp16((float(acc) * s_a[m]) * s_w[n]);
 *   per group:   y[m,n] = fp16(sum over g, increasing, of
 *                               (s_a[m] * s_w[n,g]) * float(acc[m,n,g])).
 *   INT4 weight values lie in [-8, 7]; byte j of a packed row holds element 2j
 *   in its low nibble and element 2j+1 in its high nibble, two's complement.
 *
 * Conventions for every entry point
 *   - Tensors are dense, row-major, caller-owned DEVICE memory on the current
 *     CUDA device (for example PyTorch allocations).  The library keeps no
 *     pointer after the call returns and holds no state besides a per-device
 *     stream-ordered memory pool for its scratch buffers.
 *   - fp16 tensors are IEEE binary16 (passed as void*).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued on it; no entry point synchronizes.  Launch errors are returned
 *     as CIDER_ERR_CUDA; faults inside kernels surface at the caller's next
 *     synchronization, as with any CUDA library.
 *   - A linear may enqueue two or three kernels; the later ones are
 *     programmatic dependent launches that start before the earlier ones end
 *     and wait for their results inside the kernel.  The call's first kernel
 *     starts after the stream's earlier work has finished, and its last one
 *     does not release later work early, so the call as a whole is ordered on
 *     the stream like a single kernel.
 *   - Argument checks run on the host before any launch, in this order:
 *     an empty problem (M == 0 or N == 0) returns CIDER_OK and launches
 *     nothing; null pointers, negative sizes, K < 32, K % 32 != 0, N % 8 != 0,
 *     a bad granularity / group size (per channel: group_size 0; per group:
 *     group_size 64 or 128 with K % group_size == 0) give
 *     CIDER_ERR_INVALID_ARGUMENT; a pointer not aligned to 16 bytes (fp16 and
 *     integer matrices) or 4 bytes (fp32 scale vectors, int32 accumulators)
 *     gives CIDER_ERR_MISALIGNED; a current device that is not sm_103 gives
 *     CIDER_ERR_UNSUPPORTED_DEVICE.  There is no CPU fallback.
 *   - Inputs must be finite; results for NaN / Inf inputs are unspecified.
 */
#ifndef CIDER_H
#define CIDER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CIDER_OK = 0,
  CIDER_ERR_INVALID_ARGUMENT = 1,
  CIDER_ERR_MISALIGNED = 2,
  CIDER_ERR_UNSUPPORTED_DEVICE = 3,
  CIDER_ERR_CUDA = 4,
  CIDER_ERR_TIMEOUT = 5
} cider_status_t;

typedef enum { CIDER_PER_CHANNEL = 0, CIDER_PER_GROUP = 1 } cider_granularity_t;

/* Element type of an activation or output matrix (the Cider README's roadmap,
 * "auto dtype float16/bfloat16"): IEEE binary16, or bfloat16 (the upper half
 * of an IEEE binary32). */
typedef enum { CIDER_F16 = 0, CIDER_BF16 = 1 } cider_dtype_t;

/* 1 when the current CUDA device is an sm_103 GPU this library was built
 * for, else 0 (the Cider README's is_available(), "Conditional compilation").
 * The environment variable CIDER_FORCE_UNSUPPORTED=1 forces 0. */
int cider_is_available(void);

/* Static, NUL-terminated description of a status code.  Never NULL. */
const char* cider_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int cider_version(void);

/* Per-token activation quantization (Cider README, "Metal kernel pipeline",
 * step quantize_per_token).
 *   x   fp16 [M, K]  input
 *   qa  int8 [M, K]  output codes in [-127, 127]
 *   sa  fp32 [M]     output per-token scales */
cider_status_t cider_quantize_act(const void* x, int64_t M, int64_t K,
                                  int8_t* qa, float* sa, void* stream);

/* As cider_quantize_act for bf16 activations (the README's roadmap, "auto
 * dtype float16/bfloat16"): x bf16 [M, K] is widened to fp32 exactly, then
 * quantized by the same steps. */
cider_status_t cider_quantize_act_bf16(const void* x, int64_t M, int64_t K,
                                       int8_t* qa, float* sa, void* stream);

/* Symmetric min-max INT8 weight quantization (Cider README, "Notes": min-max
 * scales; "Quantization": per channel or per group).  s_w = max|W| / 127 per
 * row (group_size 0) or per group_size-element block (64 or 128),
 * q = clamp(rint(W / s_w), -127, 127), an all-zero block gets s_w = 1.
 *   w   fp32 [N, K]  input
 *   qw  int8 [N, K]  output
 *   sw  fp32 [N, G]  output, G = 1 (per channel) or K / group_size */
cider_status_t cider_quantize_weight_int8(const float* w, int64_t N, int64_t K,
                                          int group_size, int8_t* qw, float* sw,
                                          void* stream);

/* Symmetric min-max INT4 weight quantization and packing (Cider README,
 * "Modes": W4A8 "INT4 packed (uint8)"; "Low-level API": pack_weight_int4).
 * s_w = max|W| / 7 per row or group, q = clamp(rint(W / s_w), -8, 7), packed
 * two per byte, element 2j in the low nibble.
 *   w          fp32  [N, K]
 *   qw_packed  uint8 [N, K/2]  output
 *   sw         fp32  [N, G]    output */
cider_status_t cider_quantize_weight_int4(const float* w, int64_t N, int64_t K,
                                          int group_size, uint8_t* qw_packed,
                                          float* sw, void* stream);

/* The two weight quantizers with percentile-clipped scales (Cider README,
 * "Notes": scales are min-max by default, or a percentile method,
 * clip_percentile=99.9).  Per block (a row for group_size 0, else each
 * group_size-element block) of n values: the |W| values sorted ascending
 * a_0 <= ... <= a_{n-1}; the fractional rank h = (n - 1) * clip_percentile /
 * 100 (in double), lo = floor(h), hi = min(lo + 1, n - 1),
 * t = (float)(h - lo); clip = a_lo + t * (a_hi - a_lo) in fp32 (no FMA);
 * s_w = clip / 127 (INT8) or clip / 7 (INT4), 1 when clip is 0; codes as in
 * the min-max quantizers, so values above the clip saturate at the code range.
 * clip_percentile = 100 gives exactly the min-max result.
 *   clip_percentile  in (0, 100]; anything else (or NaN) gives
 *                    CIDER_ERR_INVALID_ARGUMENT before any other check.
 *   Other arguments, layouts and checks as cider_quantize_weight_int8 / _int4. */
cider_status_t cider_quantize_weight_int8_clip(const float* w, int64_t N, int64_t K,
                                               int group_size, double clip_percentile,
                                               int8_t* qw, float* sw, void* stream);
cider_status_t cider_quantize_weight_int4_clip(const float* w, int64_t N, int64_t K,
                                               int group_size, double clip_percentile,
                                               uint8_t* qw_packed, float* sw, void* stream);

/* W8A8 linear: y = dequant(quant(x) x qw^T) (Cider README, "Low-level API":
 * perchannel_linear; "Metal kernel pipeline": quantize_per_token then
 * matmul_fused_dequant).  Quantizes x per token on the device (scratch from
 * the library's stream-ordered pool), then runs the integer GEMM with the
 * dequant fused into its store.  M <= 16 uses the weight-streaming GEMV path,
 * larger M the tensor-core GEMM (for M = 1, or M * K <= 8192, the small-M
 * kernel quantizes the rows itself and needs no scratch).
 *   x     fp16 [M, K]
 *   qw    int8 [N, K]       (out_features x in_features, nn.Linear layout)
 *   sw    fp32 [N] (granularity CIDER_PER_CHANNEL, group_size 0)
 *         or   [N, K/group_size] (CIDER_PER_GROUP, group_size 64 or 128)
 *   y     fp16 [M, N]       output */
cider_status_t cider_w8a8_linear(const void* x, int64_t M, int64_t N, int64_t K,
                                 const int8_t* qw, const float* sw,
                                 int granularity, int group_size, void* y,
                                 void* stream);

/* W4A8 linear (Cider README, "Low-level API": w4a8_linear; "Architecture":
 * INT4 -> INT8 unpack ahead of the matrix multiply).  As cider_w8a8_linear
 * with qw_packed uint8 [N, K/2] holding INT4 values. */
cider_status_t cider_w4a8_linear(const void* x, int64_t M, int64_t N, int64_t K,
                                 const uint8_t* qw_packed, const float* sw,
                                 int granularity, int group_size, void* y,
                                 void* stream);

/* The two linears for bf16 activations x bf16 [M, K]; everything else,
 * including the fp16 output y, as cider_w8a8_linear / cider_w4a8_linear.
 * The rows are always quantized by a separate kernel (scratch from the
 * library's pool), for every M. */
cider_status_t cider_w8a8_linear_bf16(const void* x, int64_t M, int64_t N, int64_t K,
                                      const int8_t* qw, const float* sw,
                                      int granularity, int group_size, void* y,
                                      void* stream);
cider_status_t cider_w4a8_linear_bf16(const void* x, int64_t M, int64_t N, int64_t K,
                                      const uint8_t* qw_packed, const float* sw,
                                      int granularity, int group_size, void* y,
                                      void* stream);

/* Import of INT4 weights stored offset-binary (each nibble u holds the value
 * u - 8: the "Symmetric INT4 (zp=8)" form of the README's "Quantization"
 * table) into this library's two's complement nibbles (value v stored as
 * v & 0xF), nibble order unchanged: dst[i] = src[i] with 8 subtracted from
 * each nibble value.  nbytes bytes, device pointers aligned to 16 bytes; dst
 * may equal src.  Returns CIDER_ERR_INVALID_ARGUMENT for nbytes < 0 or NULL
 * pointers, CIDER_ERR_MISALIGNED for unaligned pointers. */
cider_status_t cider_int4_from_offset_binary(const uint8_t* src, uint8_t* dst,
                                             int64_t nbytes, void* stream);

/* The two linears with the activation already quantized (qa int8 [M, K],
 * sa fp32 [M], as produced by cider_quantize_act).  Several projections that
 * read the same input (Q/K/V, gate/up) quantize it once and share it
 * (the idea of the pages' shared input preparation, "_InputGroup"). */
cider_status_t cider_w8a8_linear_prequant(const int8_t* qa, const float* sa,
                                          int64_t M, int64_t N, int64_t K,
                                          const int8_t* qw, const float* sw,
                                          int granularity, int group_size,
                                          void* y, void* stream);
cider_status_t cider_w4a8_linear_prequant(const int8_t* qa, const float* sa,
                                          int64_t M, int64_t N, int64_t K,
                                          const uint8_t* qw_packed,
                                          const float* sw, int granularity,
                                          int group_size, void* y, void* stream);

/* Raw integer accumulators of the same kernels (the dispatch by M and the
 * main loops of the linears above, with an int32 store in place of the
 * dequant): acc[m, n, g] = sum over k in group g of qa[m,k] * q_w[n,k],
 * layout [M, N, G], G = 1 for group_size 0 (one group spanning K), else
 * K / group_size.  For verification.
 *   qa  int8 [M, K];  qw int8 [N, K] or qw_packed uint8 [N, K/2];
 *   acc int32 [M, N, G] output. */
cider_status_t cider_w8a8_accumulators(const int8_t* qa, int64_t M, int64_t N,
                                       int64_t K, const int8_t* qw,
                                       int group_size, int32_t* acc,
                                       void* stream);
cider_status_t cider_w4a8_accumulators(const int8_t* qa, int64_t M, int64_t N,
                                       int64_t K, const uint8_t* qw_packed,
                                       int group_size, int32_t* acc,
                                       void* stream);

/* The linears with the activation and output element types chosen per call
 * (Cider README, "Roadmap": "auto dtype float16/bfloat16").
 *   x       [M, K] of x_dtype (CIDER_F16 or CIDER_BF16); a bf16 value widens
 *           exactly to fp32, then the steps are those of cider_w8a8_linear.
 *   y       [M, N] of y_dtype: the same fp32 result as for fp16 output (per
 *           channel (acc * s_a) * s_w; per group the sum over g of
 *           (s_a * s_w[n,g]) * acc_g), rounded once to y_dtype, round to
 *           nearest even (so bf16 y is not fp16 y converted).
 *   Other arguments, checks and errors as cider_w8a8_linear / cider_w4a8_linear;
 *   an x_dtype or y_dtype outside the enum gives CIDER_ERR_INVALID_ARGUMENT.
 *   (dtypes F16/F16 is cider_w8a8_linear, BF16/F16 cider_w8a8_linear_bf16.) */
cider_status_t cider_w8a8_linear_ex(const void* x, int x_dtype, int64_t M, int64_t N, int64_t K,
                                    const int8_t* qw, const float* sw, int granularity,
                                    int group_size, void* y, int y_dtype, void* stream);
cider_status_t cider_w4a8_linear_ex(const void* x, int x_dtype, int64_t M, int64_t N, int64_t K,
                                    const uint8_t* qw_packed, const float* sw, int granularity,
                                    int group_size, void* y, int y_dtype, void* stream);

/* Size of the fixed scratch array used by cider_w8a8_linear_noalloc: 32 MiB
 * of device global memory per GPU on which the library has been used. */
#define CIDER_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* W8A8 linear that allocates no memory.  The Cider README has no counterpart: this
 * entry exists for callers that must not allocate device memory while they
 * run, for example an inference engine that reserved almost all of HBM for
 * weights and KV cache before serving, or a decode loop that cannot let a
 * memory pool grow (growth can fail under memory pressure or wait on the
 * driver).  Arguments, results, checks and kernels are those of
 * cider_w8a8_linear; its scratch comes from one fixed array of
 * CIDER_NOALLOC_SCRATCH_BYTES in device memory instead of a pool.  Required
 * scratch, each part rounded up to 256-byte blocks: none for M <= 16 when
 * M == 1 or M * K <= 8192 (the small-M kernel quantizes the rows itself);
 * M * K + 4 * M bytes for other M <= 16 (int8 codes and scales); for M > 16
 * 2 * M * K + 4 * M + 4 * M bytes (fp16 codes, scales, per-token code sums).
 * A problem that needs more returns CIDER_ERR_INVALID_ARGUMENT before the
 * device is touched (for K = 2560: M above 6543).  The work-split buffers of
 * the small-M K slices and of the per-channel GEMM's K pieces are used when
 * they fit beside that, and left out otherwise (then whole row blocks / whole
 * output tiles per CTA: the same results, possibly slower).
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 *   - The first call on each device looks up the array's device address (a
 *     runtime call that allocates nothing).
 *   - All calls share the one array and each call overwrites what it uses.
 *     Calls whose kernels may overlap on the GPU (different streams without
 *     ordering, or different host threads) race and give wrong results;
 *     calls ordered on one stream are safe. */
cider_status_t cider_w8a8_linear_noalloc(const void* x, int64_t M, int64_t N,
                                         int64_t K, const int8_t* qw,
                                         const float* sw, int granularity,
                                         int group_size, void* y, void* stream);

/* Kernel timing for benchmarks.  After cider_timing_begin(capacity), each of
 * the next `capacity` linear / accumulator calls made from the calling host
 * thread records a pair of CUDA events (created here, owned by the library)
 * on its stream immediately before and after launching its integer-GEMM
 * kernel (the tensor-core GEMM, or the GEMV for M <= 16); during a stream
 * capture the records become graph nodes and time the kernel at each replay.
 * cider_timing_end waits for those events, writes the number of timed
 * launches and their summed device time in milliseconds, releases the events
 * and stops timing.  Returns CIDER_ERR_CUDA if an event call fails,
 * CIDER_ERR_INVALID_ARGUMENT for capacity < 1 or NULL outputs. */
cider_status_t cider_timing_begin(int64_t capacity);
cider_status_t cider_timing_end(int64_t* count, double* total_ms);

/* Scratch memory of the library's per-device pool: every linear takes its
 * scratch (activation codes and scales, work-split partial sums) from a
 * stream-ordered pool on the current device that keeps freed blocks for the
 * next calls, so the pool holds as much as the largest call so far needed
 * (e.g. ~200 MB for M = 8192, K = 12288).  This call synchronizes `stream`
 * and returns pool memory beyond `keep_bytes` to the device (the next larger
 * call allocates again).  CIDER_ERR_INVALID_ARGUMENT for keep_bytes < 0;
 * CIDER_OK when the pool was never used on this device. */
cider_status_t cider_trim_scratch_pool(int64_t keep_bytes, void* stream);

/* Device-side error word shared by the library's kernels on the current
 * device.  Every wait inside a kernel is bounded; a wait that runs out sets
 * this word and the kernel returns early instead of hanging.  This call
 * synchronizes `stream`, reads and clears the word, and returns CIDER_OK or
 * CIDER_ERR_TIMEOUT (CIDER_ERR_CUDA if the synchronization itself fails). */
cider_status_t cider_check_device_error(void* stream);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on a
 * barrier nothing will ever complete, giving up after `max_polls` polls.
 * Returns the launch status; the timeout itself is reported by a following
 * cider_check_device_error. */
cider_status_t cider_debug_wait_timeout(int64_t max_polls, void* stream);

/* K split of the small-M path (M <= 16), for inspection and the benchmark's
 * launch count: pure host arithmetic, no GPU needed.  For a linear with y
 * output on a GPU with num_sms SMs, writes the number of K slices the
 * weight-streaming kernel uses (1: none; > 1: each row block's K is cut into
 * that many slices on separate CTAs, the activation rows are quantized by a
 * separate kernel first, and a second kernel adds the slices' partial sums and
 * dequantizes).  int4 nonzero for W4A8.  Returns CIDER_ERR_INVALID_ARGUMENT
 * for M outside [1, 16], N, K or num_sms < 1, or a NULL output. */
cider_status_t cider_debug_small_m_slices(int64_t M, int64_t N, int64_t K, int int4,
                                          int group_size, int num_sms, int32_t* slices);

/* Launch sizes of the small-M path, for tests of its shared-memory bounds:
 * pure host arithmetic, no GPU needed.  For a linear with y output that takes
 * the weight-streaming kernel (M <= 16 and the rows fit in shared memory),
 * writes info[0..9] = {token rows padded to a power of two, 1 if the
 * tensor-core form (4..16 tokens) is used, K slices, weight tiles per slice,
 * staged activation codes per token row, the staged rows' pitch in bytes,
 * weight-ring slots, dynamic shared memory bytes, the kernel's cap on them,
 * codes per weight-tile row}.  split_allowed nonzero: the rows come
 * pre-quantized and there is scratch for the slices' partial sums (the only
 * case in which K is split).  In the tensor-core form each token row's codes
 * of a slice are copied in by one bulk copy of min(staged codes, K - the
 * slice's first code) bytes.  Returns CIDER_ERR_INVALID_ARGUMENT when the
 * problem does not take this path, for N, K or num_sms < 1, or a NULL info. */
cider_status_t cider_debug_small_m_launch(int64_t M, int64_t N, int64_t K, int int4,
                                          int group_size, int split_allowed, int num_sms,
                                          int32_t* info);

/* Work split of the per-channel tensor-core GEMM, for inspection and tests:
 * pure host arithmetic, no GPU needed.  For an M x N x K problem on `pairs`
 * CTA pairs (`pairs` >= 1 stands for the device's count), the GEMM's 256 x 256
 * output tiles are dealt whole for whole rounds, and (when that is cheaper)
 * each remaining tile is cut along K into equal pieces on several pairs, each
 * of which then adds up all pieces' partial sums for its own share of the
 * tile's weight rows.  Writes info[0..5] = {pairs launched, tiles dealt whole,
 * tiles cut, pieces per cut tile, 128-K blocks per tile, tiles} and, for every
 * launched pair in the order it processes them, one row of seven int32 per
 * unit: {pair, tile, first block, end block, kind (0 whole, 1 piece), first
 * and end weight row (within the tile) that the unit dequantizes and stores}.
 * `units` holds `capacity` rows; `count` receives the number of rows (which
 * may exceed `capacity`: then only `capacity` are written).  Returns
 * CIDER_ERR_INVALID_ARGUMENT for sizes < 1, pairs < 1 or NULL outputs. */
cider_status_t cider_debug_pair_schedule(int64_t M, int64_t N, int64_t K, int pairs,
                                         int64_t capacity, int32_t* units, int64_t* count,
                                         int32_t* info);

#ifdef __cplusplus
}
#endif
#endif /* CIDER_H */
