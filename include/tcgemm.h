/*
 * tcgemm — bf16 GEMM with fp32 accumulation on tcgen05 tensor cores (sm_103a).
 *
 *   C = alpha * A * B + beta * C
 *
 * The operation is the matrix product C[m,n] = A[m,k] x B[k,n] of the H100 work
 * log "在 H100 上超越 cuBLAS：一份工作日志" (section "Simon 博客的快速回顾"), with
 * the layouts of its section "实验设置": bf16 inputs, A row-major, B and C
 * column-major.  The alpha/beta update is the BLAS form named in the "DeepGEMM"
 * article (demingchina.com), section 1.1; fp32 accumulation is that article's
 * precision contract (section 3.1).
 *
 * Layouts (element (i,j) of each matrix):
 *   A: M x K, row-major,    A[i,k] at ((const bf16*)A)[i*lda + k], lda >= K
 *   B: K x N, column-major, B[k,j] at ((const bf16*)B)[j*ldb + k], ldb >= K
 *   C: M x N, column-major, C[i,j] at ((T*)C)[j*ldc + i],          ldc >= M
 * where bf16 is the 16-bit brain-float format and T is float (out_dtype
 * TCGEMM_OUT_F32) or bf16 (TCGEMM_OUT_BF16).  With beta != 0, C is read first
 * and has the output type; with beta == 0, C is never read (NaN in C is fine).
 *
 * Pointers: A, B and C are device pointers (CUDA global memory) on the current
 * device.  The caller owns every buffer and the stream; the library keeps no
 * reference to any of them after the call returns.  `stream` is a cudaStream_t
 * passed as void* (NULL means the legacy default stream).
 *
 * Rules checked on the host before anything is launched (error return, nothing
 * written):
 *   - M, N, K >= 0 and below 2^31; lda >= max(K,1), ldb >= max(K,1), ldc >= max(M,1);
 *   - A, B, C 16-byte aligned; lda*2, ldb*2 and ldc*sizeof(T) multiples of 16
 *     bytes (the tensor-memory-accelerator copy rules)   -> TCGEMM_ERR_ALIGNMENT;
 *   - C does not overlap A or B                           -> TCGEMM_ERR_INVALID_ARG;
 *   - the current device is compute capability 10.3      -> TCGEMM_ERR_UNSUPPORTED_DEVICE.
 * M == 0 or N == 0 is a no-op.  K == 0 sets C = beta*C (0 when beta == 0).
 *
 * Asynchrony: calls enqueue work on `stream` and return.  Launch failures return
 * TCGEMM_ERR_CUDA.  A device-side wait that exceeds its time limit (a hang
 * guard; it never fires in a correct run) is reported through
 * tcgemm_check_device_status().  Concurrent calls from several host threads are
 * safe.
 */
#ifndef TCGEMM_H
#define TCGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TCGEMM_OUT_F32 = 0,
    TCGEMM_OUT_BF16 = 1,
    TCGEMM_OUT_I8 = 2    /* int8 codes; only through gemm_quant_i8 */
} tcgemm_dtype_t;

typedef enum {
    TCGEMM_OK = 0,
    TCGEMM_ERR_INVALID_ARG = 1,
    TCGEMM_ERR_ALIGNMENT = 2,
    TCGEMM_ERR_UNSUPPORTED_DEVICE = 3,
    TCGEMM_ERR_CUDA = 4,
    TCGEMM_ERR_TIMEOUT = 5
} tcgemm_status_t;

/* Kernel variants (see gemm_bf16_variant).  TCGEMM_VARIANT_AUTO picks by shape. */
typedef enum {
    TCGEMM_VARIANT_AUTO = 0,
    TCGEMM_VARIANT_1CTA = 1,  /* one CTA per SM, 128 x 256 tiles, cta_group::1 MMA   */
    TCGEMM_VARIANT_2CTA = 2,  /* CTA pairs, cta_group::2 MMA (M=256), tiles 256 x 256 or 256 x 224,
                                 whichever finishes the persistent rounds sooner */
    /* 3 is not a variant: the number is kept unused so that no other variant
       is renumbered; passing it is TCGEMM_ERR_INVALID_ARG. */
    TCGEMM_VARIANT_1CTA_N64 = 4, /* one CTA per SM, narrow 128 x 64 tiles, 8-stage pipeline (12
                                   stages and 64-row A tiles when M <= 64): the choice for
                                   M <= 128, where B is streamed from memory once */
    TCGEMM_VARIANT_2CTA_W256 = 5, /* as TCGEMM_VARIANT_2CTA with the tile width fixed at 256 */
    TCGEMM_VARIANT_SWAP_N64 = 6,  /* the transposed product C^T = B^T A^T on 128 x 64 tiles (128
                                    columns of C by up to 64 rows): the choice for M <= 64 */
    TCGEMM_VARIANT_SWAP_N64_KS2 = 7 /* as TCGEMM_VARIANT_SWAP_N64 (128 x 128 tiles of C^T when
                                      M > 64), each tile computed by a cluster of 2 CTAs that
                                      split its k-blocks in halves; each CTA then finishes half of
                                      the tile, adding the peer's fp32 partial of that half
                                      through distributed shared memory (a sum of two terms: the
                                      same bits whichever CTA adds), so no workspace and no
                                      second kernel: the choice for M <= 128 when the tiles fill
                                      3/4 to 1 round of 2-CTA clusters */,
    TCGEMM_VARIANT_SWAP_PAIR = 8 /* the transposed product on CTA pairs (M <= 128): one
                                   cta_group::2 MMA per k-block over a tile of 2*r columns of C
                                   (r per CTA, r a multiple of 8 chosen so that the tiles give
                                   every SM of the device one) by all M rows; each CTA streams its
                                   r columns of B over the whole of K and half of A's rows, so
                                   there is no K split and no exchange; bf16 operands in the
                                   layouts of gemm_bf16, fp32 or bf16 output */
} tcgemm_variant_t;

/* C = alpha*A*B + beta*C as described above.  Returns TCGEMM_OK once the work
 * is enqueued. */
int gemm_bf16(int64_t M, int64_t N, int64_t K,
              const void* A, int64_t lda,
              const void* B, int64_t ldb,
              void* C, int64_t ldc,
              float alpha, float beta, int out_dtype, void* stream);

/* Same operation with an explicit kernel variant (tcgemm_variant_t); used by
 * tests and tuning to run every variant on the same shapes.  Same rules and
 * errors as gemm_bf16; an unknown variant is TCGEMM_ERR_INVALID_ARG. */
int gemm_bf16_variant(int64_t M, int64_t N, int64_t K,
                      const void* A, int64_t lda,
                      const void* B, int64_t ldb,
                      void* C, int64_t ldc,
                      float alpha, float beta, int out_dtype, void* stream, int variant);

/* Same operation on HOST buffers: A, B and C are host pointers (pinned
 * memory, e.g. from cudaHostAlloc, lets the copies run asynchronously; pageable
 * memory works too, with the copies staged by the driver).  On `stream` the
 * call enqueues one pitched host-to-device copy of A and of B (their M x K and
 * N x K elements; padding is not copied) and of C when beta != 0, the GEMM
 * (automatic variant) on the library's device copies, and one pitched
 * device-to-host copy of C's M x N elements (its ldc padding on the host is
 * never written), then returns.  C holds the result once `stream` has completed that work;
 * the caller must neither write A, B, C nor read C before then.  The device
 * copies belong to the library: one set per device and stream, allocated by
 * cudaMalloc on the first call that needs them (or needs more), held until
 * the process exits; calls that overlap on the GPU must use different
 * streams.  out_dtype TCGEMM_OUT_F32 or _BF16.  Rules and errors as
 * gemm_bf16, applied to the host pointers (16-byte alignment, leading
 * dimensions, no overlap of C with A or B); a failed copy or allocation ->
 * TCGEMM_ERR_CUDA.  The pages this library follows time device-resident
 * operands only; this entry point serves callers whose matrices live in host
 * memory. */
int gemm_bf16_host(int64_t M, int64_t N, int64_t K,
                   const void* A, int64_t lda,
                   const void* B, int64_t ldb,
                   void* C, int64_t ldc,
                   float alpha, float beta, int out_dtype, void* stream);

/* Same operation with a caller-supplied workspace instead of the library's
 * own.  When the tiles do not fill the last round of the persistent CTAs, the
 * k-blocks of that round's tiles are shared out evenly ("stream-K"); the fp32
 * partial tiles this needs live in the workspace (see
 * tcgemm_workspace_bytes), and a second kernel on the same stream adds them up.  `workspace` is device memory of at least
 * tcgemm_workspace_bytes(M, N, K, variant, SMs) bytes, 256-byte aligned (no
 * initialisation needed).  Calls that overlap on the GPU must not share a
 * workspace.  With a plan that needs none, `workspace` may be NULL.
 * Too small, misaligned or NULL when needed -> TCGEMM_ERR_INVALID_ARG.
 * (gemm_bf16 and gemm_bf16_variant use a library-owned workspace per device
 * and stream instead: about 38 MiB, allocated on the first call that needs
 * one on that stream, so make that first call before any stream capture.) */
int gemm_bf16_ws(int64_t M, int64_t N, int64_t K,
                 const void* A, int64_t lda,
                 const void* B, int64_t ldb,
                 void* C, int64_t ldc,
                 float alpha, float beta, int out_dtype, void* stream, int variant,
                 void* workspace, int64_t workspace_bytes);

/* Same operation for callers that cannot allocate device memory once they are
 * running (a fixed memory budget, an allocator that owns all device memory, or
 * code that must not stall on cudaMalloc's implicit device synchronisation).
 * Nothing is allocated: shapes that share out their last round of work keep
 * their partial tiles in a fixed scratch array compiled into this library
 * (tcgemm_noalloc_scratch_bytes(), 40 MiB per GPU that loads the library, held
 * until the process exits).  A shape that would need more scratch than that
 * is rejected with TCGEMM_ERR_INVALID_ARG and tcgemm_last_error() says how
 * much it needs.  The first call on a device looks up the array's device
 * address (once per device, with that device current); make that first call
 * before any stream capture.  Every call shares the one array (which keeps
 * the previous call's partial tiles; nothing in it needs to start at zero), so
 * calls that overlap on the GPU (other streams, other host threads) race on
 * it and must be serialised by the caller.  The pages this library follows have no counterpart of this entry
 * point.  Other rules and errors as gemm_bf16_variant. */
int gemm_bf16_noalloc(int64_t M, int64_t N, int64_t K,
                      const void* A, int64_t lda,
                      const void* B, int64_t ldb,
                      void* C, int64_t ldc,
                      float alpha, float beta, int out_dtype, void* stream, int variant);

/* Fused epilogue activations (gemm_bf16_bias_act). */
typedef enum {
    TCGEMM_ACT_NONE = 0,
    TCGEMM_ACT_RELU = 1,      /* max(x, 0); NaN stays NaN                                  */
    TCGEMM_ACT_GELU = 2,      /* x * Phi(x), Phi the standard normal distribution function  */
    TCGEMM_ACT_GELU_TANH = 3  /* x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))          */
} tcgemm_activation_t;

/* Element type of the fused epilogue's bias vector. */
typedef enum {
    TCGEMM_BIAS_NONE = 0,
    TCGEMM_BIAS_F32 = 1,
    TCGEMM_BIAS_BF16 = 2
} tcgemm_bias_t;

/* GEMM with the fused epilogue of the "DeepGEMM" article, section 6.1 (after
 * a fully connected layer the output gets a bias and then ReLU or GELU, done
 * at the end of the GEMM kernel instead of in a second pass over C):
 *
 *   C[i,j] = act( alpha * sum_k A[i,k] B[k,j] + beta * C[i,j] + bias[j] )
 *
 * computed in fp32 from the fp32 accumulator and rounded once to out_dtype.
 * The article fixes the order (bias, then activation); where alpha and beta
 * enter, the bias axis and the GELU form are this library's readings: bias[j]
 * is one value per column j of C (per output feature when B holds a layer's
 * weights), and TCGEMM_ACT_GELU is the exact definition (Hendrycks and Gimpel,
 * "Gaussian Error Linear Units", 2016; evaluated as x * erfc(-x/sqrt 2) / 2),
 * TCGEMM_ACT_GELU_TANH that paper's tanh approximation (evaluated as
 * x * sigmoid(2z)).  The GPU evaluates erfc as t * exp(-z^2 + P(t)),
 * t = 1/(1 + z/2) (the form of "Numerical Recipes", section 6.2) with a
 * fitted degree-9 P, and exp with CUDA's __expf: the activations are within a
 * relative 4e-5 of their exact values (tested on a dense grid).
 *
 * bias:       device pointer to N values of bias_dtype (fp32 or bf16), aligned
 *             to the element size, not overlapping C; NULL exactly when
 *             bias_dtype is TCGEMM_BIAS_NONE.  Read only; the caller owns it.
 * bias_dtype: tcgemm_bias_t.
 * activation: tcgemm_activation_t.
 * variant:    as gemm_bf16_variant (0 = chosen by shape).
 * With TCGEMM_BIAS_NONE and TCGEMM_ACT_NONE this is gemm_bf16_variant.  K == 0
 * gives act(beta * C + bias[j]).  Errors: an unknown activation or bias dtype,
 * a bias pointer that is NULL when needed (or given with TCGEMM_BIAS_NONE), or
 * a bias overlapping C -> TCGEMM_ERR_INVALID_ARG; a misaligned bias ->
 * TCGEMM_ERR_ALIGNMENT; all other rules and errors as gemm_bf16_variant. */
int gemm_bf16_bias_act(int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda,
                       const void* B, int64_t ldb,
                       void* C, int64_t ldc,
                       float alpha, float beta, int out_dtype,
                       const void* bias, int bias_dtype, int activation,
                       void* stream, int variant);

/* 8-bit float operand formats (gemm_fp8): the two formats of the OCP 8-bit
 * floating point specification. */
typedef enum {
    TCGEMM_FP8_E4M3 = 0,  /* sign, 4 exponent bits (bias 7), 3 fraction bits; no infinities; max 448 */
    TCGEMM_FP8_E5M2 = 1   /* sign, 5 exponent bits (bias 15), 2 fraction bits; IEEE-style inf/NaN  */
} tcgemm_fp8_format_t;

/* The same GEMM on 8-bit float operands, the input path the "DeepGEMM"
 * article (section 6.3) names as its next step:
 *
 *   C[i,j] = alpha * sum_k A[i,k] B[k,j] + beta * C[i,j]
 *
 * with A and B both in `in_format` (tcgemm_fp8_format_t), one byte per
 * element, in the layouts of gemm_bf16 (A row-major M x K, B column-major
 * K x N; lda, ldb in elements, i.e. bytes, multiples of 16).  Products are
 * exact and accumulate in fp32 on the tensor cores (tcgen05 kind::f8f6f4);
 * per-tensor scale factors go into alpha.  C is fp32 or bf16 as in
 * gemm_bf16.  The article gives no formats or scaling rules: the OCP formats
 * and alpha as the scale are this library's readings.
 * variant: 0 (chosen by shape), TCGEMM_VARIANT_2CTA, _2CTA_W256, _1CTA_N64 or
 * _SWAP_N64; TCGEMM_VARIANT_1CTA is not built for 8-bit operands
 * -> TCGEMM_ERR_INVALID_ARG, as is an unknown in_format.  Other
 * rules and errors as gemm_bf16_variant (16-byte rules in bytes). */
int gemm_fp8(int64_t M, int64_t N, int64_t K,
             const void* A, int64_t lda,
             const void* B, int64_t ldb,
             void* C, int64_t ldc,
             float alpha, float beta, int out_dtype, int in_format,
             void* stream, int variant);

/* gemm_fp8 with each operand in its own 8-bit format and a caller-owned
 * split workspace.  a_format is A's tcgemm_fp8_format_t, b_format B's; they
 * may differ (E4M3 x E5M2 either way: kind::f8f6f4 takes a format per
 * operand; products stay exact and accumulate in fp32).  workspace NULL: as
 * gemm_fp8 (the library's own split workspace when the plan needs one);
 * otherwise, as gemm_bf16_ws: a device buffer of at least
 * tcgemm_workspace_bytes(M, N, K, variant, SMs) bytes for 8-bit operands
 * (tcgemm_plan_kind with in_kind 1 reports it), 256-byte aligned, owned by
 * the caller, used by this call only until `stream` has completed it.  The
 * automatic choice consults the tuned-choice table only when both formats
 * agree.  Other rules and errors as gemm_fp8; an unknown format in either
 * position -> TCGEMM_ERR_INVALID_ARG. */
int gemm_fp8_ex(int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, int a_format,
                const void* B, int64_t ldb, int b_format,
                void* C, int64_t ldc,
                float alpha, float beta, int out_dtype,
                void* stream, int variant, void* workspace, int64_t workspace_bytes);

/* gemm_bf16_host for 8-bit operands: A, B (both in in_format, one byte per
 * element; lda, ldb in elements, rows multiples of 16 bytes) and C on HOST
 * memory, copied in, multiplied with the automatic variant and C copied back
 * on `stream`, with the device copies, ownership and completion rules of
 * gemm_bf16_host.  Errors as gemm_bf16_host; an unknown in_format ->
 * TCGEMM_ERR_INVALID_ARG. */
int gemm_fp8_host(int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda,
                  const void* B, int64_t ldb,
                  void* C, int64_t ldc,
                  float alpha, float beta, int out_dtype, int in_format, void* stream);



/* Operand types of gemm_quant_i8. */
typedef enum {
    TCGEMM_IN_BF16 = 0,
    TCGEMM_IN_E4M3 = 1,
    TCGEMM_IN_E5M2 = 2
} tcgemm_in_t;

/* GEMM with the quantising epilogue of the "DeepGEMM" article, section 6.2
 * (the next layer wants int8 input: y = round(x * scale + zero_point), with
 * one scale per row -- per token -- done in the GEMM's epilogue instead of a
 * second pass over the fp32 result):
 *
 *   x[i,j] = act( alpha * sum_k A[i,k] B[k,j] + bias[j] )          (fp32)
 *   Q[i,j] = saturate_int8( rne( fmaf(x[i,j], row_scale[i], zero_point) ) )
 *
 * rne rounds to nearest with ties to even; saturation clamps to [-128, 127];
 * a NaN gives 0.  The article gives the formula and the per-row scale; the
 * zero point's granularity (one integer), the rounding (ties to even) and the
 * saturation are this library's readings.
 *
 * A, B: in_type (tcgemm_in_t) operands in the layouts of gemm_bf16 / gemm_fp8
 * (lda, ldb in elements, rows multiples of 16 bytes).
 * Q: int8, column-major M x N, Q[i,j] at ((int8_t*)Q)[j*ldq + i], ldq >= M and
 *    a multiple of 16; written only (there is no beta).
 * bias, bias_dtype, activation: as gemm_bf16_bias_act (TCGEMM_BIAS_NONE and
 *    TCGEMM_ACT_NONE for none).
 * row_scale: M fp32 device values, 16-byte aligned, not overlapping Q.
 * variant: 0 (by shape), TCGEMM_VARIANT_2CTA, _2CTA_W256, _1CTA_N64 or
 *    _SWAP_N64 (the others -> TCGEMM_ERR_INVALID_ARG).
 * Errors: an unknown in_type, a NULL row_scale -> TCGEMM_ERR_INVALID_ARG; a
 * misaligned row_scale -> TCGEMM_ERR_ALIGNMENT; otherwise as gemm_bf16_bias_act. */
int gemm_quant_i8(int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda,
                  const void* B, int64_t ldb, int in_type,
                  void* Q, int64_t ldq, float alpha,
                  const void* bias, int bias_dtype, int activation,
                  const float* row_scale, int zero_point,
                  void* stream, int variant);

/* Storage order of an operand (gemm_bf16_layout). */
typedef enum {
    TCGEMM_ROW_MAJOR = 0,
    TCGEMM_COL_MAJOR = 1
} tcgemm_layout_t;

/* The bf16 GEMM with each operand in either storage order (the work log's
 * layout, "实验设置", is A row-major and B column-major; the other three are
 * the same product with an operand stored transposed):
 *   A row-major:    A[i,k] at A[i*lda + k], lda >= K   (K contiguous)
 *   A column-major: A[i,k] at A[k*lda + i], lda >= M   (M contiguous)
 *   B column-major: B[k,j] at B[j*ldb + k], ldb >= K   (K contiguous)
 *   B row-major:    B[k,j] at B[k*ldb + j], ldb >= N   (N contiguous)
 * C is column-major as in gemm_bf16.  An operand with its M or N index
 * contiguous is loaded by TMA in 64 x 64 boxes and read by the tensor cores
 * as an MN-major operand (the transpose bits of the MMA's instruction
 * descriptor); nothing is transposed in memory.  Variants as
 * gemm_bf16_variant; an unknown layout is TCGEMM_ERR_INVALID_ARG.  Other
 * rules and errors as gemm_bf16_variant. */
int gemm_bf16_layout(int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, int a_layout,
                     const void* B, int64_t ldb, int b_layout,
                     void* C, int64_t ldc,
                     float alpha, float beta, int out_dtype, void* stream, int variant);

/* tcgemm_plan for bf16 (in_kind 0) or 8-bit (in_kind 1) operands and the
 * operand layouts of gemm_bf16_layout (a_layout TCGEMM_ROW_MAJOR and b_layout
 * TCGEMM_COL_MAJOR are gemm_bf16's): a k-block holds 64 bf16 or 128 8-bit
 * values, which changes the k-block count and the stream-K choice, and a
 * row-major B takes 256-wide pair tiles.  Host only. */
int tcgemm_plan_kind(int64_t M, int64_t N, int64_t K, int variant, int in_kind, int a_layout, int b_layout,
                     int num_sms, int64_t* out);

/* Autotuning (the work log attributes its remaining per-shape gaps to the
 * lack of it): time every kernel variant built for this problem on the
 * caller's buffers and remember the fastest.  Every later call for the same
 * device, M, N, K, operand type (tcgemm_in_t), operand layouts
 * (tcgemm_layout_t; gemm_bf16's are TCGEMM_ROW_MAJOR A and TCGEMM_COL_MAJOR
 * B), output type (fp32 or bf16) and beta == 0 or not that asks for the
 * automatic choice (variant 0) then uses it.  Each candidate runs once, then
 * `iters` (1..1000) times, each call between its own pair of CUDA events on
 * `stream`; with flush_bytes > 0 the device buffer `flush` is written
 * (cudaMemsetAsync, untimed) before every timed call, so that a buffer
 * larger than L2 makes the timing that of a cold call (NULL / 0: back-to-back
 * calls, operands partly in L2).  The call synchronises the stream, so it
 * cannot be captured in a CUDA graph.  C is
 * overwritten (with beta != 0 it accumulates): its contents afterwards are
 * undefined.  Writes the chosen variant to *best_variant and, if best_us is
 * not NULL, its mean time in microseconds.  Errors: bad arguments ->
 * TCGEMM_ERR_INVALID_ARG; a failed timed call -> TCGEMM_ERR_CUDA; a device
 * timeout in the timed runs -> TCGEMM_ERR_TIMEOUT. */
int tcgemm_autotune(int64_t M, int64_t N, int64_t K,
                    const void* A, int64_t lda, int a_layout,
                    const void* B, int64_t ldb, int b_layout, int in_type,
                    void* C, int64_t ldc, float alpha, float beta, int out_dtype,
                    int iters, void* flush, int64_t flush_bytes, void* stream,
                    int* best_variant, float* best_us);

/* The variant tcgemm_autotune chose for this problem on the current device,
 * or 0 if none was tuned.  Host only. */
int tcgemm_autotune_lookup(int64_t M, int64_t N, int64_t K, int in_type, int out_dtype, int a_layout,
                           int b_layout, int beta_nonzero);

/* Forget every tuned choice.  Host only. */
void tcgemm_autotune_clear(void);

/* Records `variant` as the tuned choice for this problem on the current
 * device (device 0 when no device is visible), as tcgemm_autotune would — for
 * a choice measured elsewhere; variant 0 removes the entry.  Arguments as
 * tcgemm_autotune_lookup.  A variant not built for that kind of problem (the
 * single-CTA variants 1 and 3 for 8-bit operands or int8 output, variant 3
 * with a column-major A or row-major B, 8-bit operands with those layouts) or
 * a size outside 1..2^31-1 -> TCGEMM_ERR_INVALID_ARG.  Host only. */
int tcgemm_autotune_set(int64_t M, int64_t N, int64_t K, int in_type, int out_dtype, int a_layout, int b_layout,
                        int beta_nonzero, int variant);

/* Writes every tuned choice (all devices) to the text file `path`: a header
 * line, then one line per choice (device ordinal, M, N, K, operand kind and
 * format, output type, A column-major, B row-major, beta != 0, variant).
 * Returns the number of choices written, or -1 if the file cannot be written
 * (tcgemm_last_error says why).  Host only. */
int64_t tcgemm_autotune_save(const char* path);

/* Adds the choices in a file written by tcgemm_autotune_save, replacing any
 * for the same problem; automatic calls use them from then on.  Returns the
 * number read, or -1 (nothing added) if the file cannot be read, lacks the
 * header or holds a line that is not a valid choice.  Choices are keyed by
 * device ordinal: load a table on the kind of GPU it was measured on.  Host
 * only. */
int64_t tcgemm_autotune_load(const char* path);

/* Size in bytes of gemm_bf16_noalloc's fixed scratch array.  Host only. */
int64_t tcgemm_noalloc_scratch_bytes(void);

/* 1 if gemm_bf16_noalloc's scratch array holds what the plan of this problem
 * needs on a device with `num_sms` SMs (the test that entry point applies
 * before launching; plans without a split need none), 0 if the call would be
 * refused, -1 on bad arguments.  Host only; needs no GPU. */
int tcgemm_noalloc_fits(int64_t M, int64_t N, int64_t K, int variant, int num_sms);

/* Workspace bytes the launch for this shape and variant needs on a device
 * with `num_sms` SMs (0: none).  Host only. */
int64_t tcgemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant, int num_sms);

/* The variant gemm_bf16 would run for this shape on a device with `num_sms`
 * streaming multiprocessors.  Host only; needs no GPU. */
int tcgemm_pick_variant(int64_t M, int64_t N, int64_t K, int num_sms);

/* Host-only description of the launch gemm_bf16_variant would make, for tests
 * and tools: out[0] = grid size (CTAs), out[1] = CTAs per cluster, out[2] =
 * tile rows (tiles_m), out[3] = tile columns (tiles_n), out[4] = tile height,
 * out[5] = tile width, out[6] = k-blocks per tile, out[7] = dynamic shared
 * memory bytes, out[8] = tiles computed whole, out[9] = tiles of the last
 * round shared out by stream-K, out[10] = their k-blocks in total, out[11] =
 * workspace bytes, out[12] = tile
 * band height of the visiting order, out[13] = variant, out[14] = CTAs per
 * MMA (cta_group), out[15], out[16] = rows and columns of the unit grid the
 * visiting order walks (the tile grid), out[17] =
 * 1 when stream-K is used, out[18] = rows of the MMA's A operand loaded per
 * CTA (64 for M <= 64 with variant 4, the chosen r for variant 8, else 128),
 * out[19] = 1 when the launch computes the transposed product (variants 6, 7
 * and 8; then out[2..] describe C^T),
 * out[20] = CTAs of a cluster that split each tile's k-blocks (2 for
 * variant 7, else 1), out[21] = the visiting order: 0 for the grouped band
 * order, k > 0 for the Hilbert curve over the enclosing 2^k x 2^k square
 * (environment TCGEMM_ORDER=grouped or =hilbert overrides the default).
 * `out` must hold 22 values.  Returns TCGEMM_OK or TCGEMM_ERR_INVALID_ARG.  Needs no
 * GPU. */
int tcgemm_plan(int64_t M, int64_t N, int64_t K, int variant, int num_sms, int64_t* out);

/* The same description for the current device, using its actual number of
 * SMs and of clusters that can be resident at once (what gemm_bf16_variant
 * itself uses).  Needs a supported GPU. */
int tcgemm_plan_device(int64_t M, int64_t N, int64_t K, int variant, int64_t* out);

/* Current device: out[0] = SMs, out[1] = CTA pairs that can be resident at
 * once with this library's kernels, out[2] = 0 (unused), out[3] = device
 * ordinal.  `out` must hold 4 values.  Needs a supported GPU. */
int tcgemm_device_info(int64_t* out);

/* The work units cluster `cluster` runs under the host plan of tcgemm_plan
 * (host copy of the device iterator): for unit i, out[7i..7i+6] = unit index
 * in visiting order, first and one-past-last k-block, workspace slot (-1 for
 * a whole tile), stream-K tile index (-1 for round-robin tiles), piece index
 * and number of pieces of that tile.  Writes at most max_units units and
 * returns how many there are (-1 on bad arguments).  Needs no GPU. */
int tcgemm_units(int64_t M, int64_t N, int64_t K, int variant, int num_sms, int cluster, int max_units,
                 int32_t* out);

/* Grouped band order of the persistent kernels (host copy of the device
 * function; the work log's "调度与 L2 缓存"): writes the tile row and column
 * of order index t = 0..count-1 into tm[t], tn[t]; consecutive indices run
 * down a band of group_m tile rows, then one tile column right.  Needs no
 * GPU. */
int tcgemm_tile_order(int tiles_m, int tiles_n, int group_m, int64_t count, int32_t* tm, int32_t* tn);

/* The Hilbert order of the work log's "内核 11：希尔伯特曲线" (host copy of the
 * device function): the tiles_m x tiles_n tiles in the order the Hilbert
 * curve over the enclosing 2^k x 2^k square visits them, cells outside the
 * grid skipped; tile row and column of order index t = 0..count-1 into
 * tm[t], tn[t] (count <= tiles_m * tiles_n).  Returns TCGEMM_OK or
 * TCGEMM_ERR_INVALID_ARG.  Needs no GPU. */
int tcgemm_tile_order_hilbert(int tiles_m, int tiles_n, int64_t count, int32_t* tm, int32_t* tn);

/* Human-readable name of a status code (static string). */
const char* tcgemm_status_string(int status);

/* Detail of the last failed call on this host thread (static per-thread
 * buffer, empty when there was none). */
const char* tcgemm_last_error(void);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns TCGEMM_ERR_TIMEOUT if a kernel gave up a wait since
 * the last check (*where_out, if not NULL, receives the role that timed out:
 * 1 producer, 2 MMA, 3 epilogue, 4 drain, 5 self test), TCGEMM_ERR_CUDA if the
 * synchronisation failed, else TCGEMM_OK. */
int tcgemm_check_device_status(void* stream, uint32_t* where_out);

/* Launches a one-thread kernel that waits on a barrier nothing arrives on and
 * gives up after `timeout_ns` nanoseconds, then returns
 * tcgemm_check_device_status() — TCGEMM_ERR_TIMEOUT when the hang guard
 * works.  Touches no user memory. */
int tcgemm_selftest_timeout(void* stream, uint64_t timeout_ns);

/* Self test of the GEMM's own give-up path (the hang guard inside the
 * kernels, not the one-thread wait of tcgemm_selftest_timeout).  Runs
 * C = A*B (alpha 1, beta 0, fp32 output, the layouts and rules of gemm_bf16)
 * with kernel variant `variant` (1, 2, 4 or 5: the plain-product kernels,
 * no split of K) while the TMA producer of CTA 0 withholds the arrival and
 * the loads of its first k-block, so that the MMA thread's wait for that
 * stage runs out after `timeout_ns` (in (0, 10 s]).  The waiting roles give
 * up, every CTA drains its own copies and MMAs, frees its TMEM and exits;
 * the call synchronizes `stream` and returns what tcgemm_check_device_status
 * reports: TCGEMM_ERR_TIMEOUT when the path works (the status word is then
 * cleared and the context stays usable).  C is left unspecified.  Other
 * errors: TCGEMM_ERR_INVALID_ARG for another variant, non-positive sizes or
 * a limit out of range; as gemm_bf16 otherwise.  No counterpart on the
 * pages: it exists to test the bounded waits. */
int tcgemm_selftest_withheld_load(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                  int64_t ldb, void* C, int64_t ldc, int variant, uint64_t timeout_ns,
                                  void* stream);

/* Number of kernels this library has launched in this process. */
uint64_t tcgemm_launch_count(void);

/* Library version: major*10000 + minor*100 + patch. */
int tcgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_H */
