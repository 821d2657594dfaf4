/*
 * sq.h -- absmax-scaled quantization and scaled low-precision GEMM on GB300
 * (sm_103a).  C ABI of libsq.so.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers (cudaMalloc / torch memory on the
 *    current device) unless a parameter says otherwise.  The caller owns every
 *    buffer; the library never allocates or frees device memory, never reads a
 *    device scalar on the host and never synchronises the stream on these
 *    paths.  Work is enqueued on `stream` (NULL = the legacy default stream) and
 *    runs on the device that is current when the call is made.
 *  - Matrices are row-major and packed unless a leading dimension is given:
 *    "A[M,K]" means element (i,k) sits at A[i*K + k].
 *  - A call validates its arguments first and returns SQ_ERR_INVALID_ARG,
 *    SQ_ERR_UNSUPPORTED or SQ_ERR_ALIGNMENT without enqueuing anything when a
 *    check fails.  A launch failure returns SQ_ERR_CUDA.  Errors raised inside
 *    a kernel (a bounded wait that ran out) are recorded on the device and read
 *    back by sq_get_last_device_error().
 *  - Inputs are finite.  Results for NaN or infinite inputs are unspecified.
 *  - Calls that share a workspace must not overlap on the GPU (use one
 *    workspace per stream).
 *
 * Sources (the three pages on the subject):
 *  [P2] POPCORNBENCH "Kimi-K2.6 l2_p13" trace: the INT8 fake-quant formula
 *       (amax = max|x| floored at 1e-8, scale = amax/127,
 *       q = clamp(round(x/scale), -127, 127)) and its rounding discussion
 *       (torch.round rounds halves to even, so roundf is wrong).
 *  [P1] scmp_kernels README, SC quickstart and sc_matmul API: per-row and
 *       per-head ("per_head requires 3D") granularity, C = a @ b.T with float32
 *       in and out.
 *  [P3] AstrAI astrai/extension/ops/fp8.py: module docstring (scales are
 *       quantization steps divided out, x8 = x / scale; amax is returned),
 *       custom::fp8_quantize (bf16 in, fused amax), custom::fp8_gemm
 *       (a @ b * (sa * sb), FP32 accumulation, BF16 out), the fmt map
 *       (0 = E4M3, 1 = E5M2) and the commit notes (last-block amax epilogue,
 *       NT forward; dX and dW read transposed operands).
 */
#ifndef SQ_H_
#define SQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* sq_stream;

typedef enum {
    SQ_OK = 0,
    SQ_ERR_INVALID_ARG = 1,    /* a size, pointer, dtype, fmt or layout is invalid      */
    SQ_ERR_UNSUPPORTED = 2,    /* valid but not implemented here (e.g. shape limits)     */
    SQ_ERR_ALIGNMENT = 3,      /* a pointer or leading dimension breaks the 16-B rules  */
    SQ_ERR_CUDA = 4,           /* the CUDA runtime reported an error                     */
    SQ_ERR_DEVICE_TIMEOUT = 5  /* a kernel's bounded wait ran out (kernel returned early) */
} sq_status;

typedef enum { SQ_F32 = 0, SQ_BF16 = 1 } sq_dtype;

/* Matches the fmt integers of [P3] (_FMT_TO_INT). */
typedef enum { SQ_FMT_E4M3 = 0, SQ_FMT_E5M2 = 1 } sq_fp8_fmt;

/* GEMM operand layouts (all row-major):
 *   SQ_NT: A[M,K], B[N,K], C = A * B^T   (forward, X * W^T)
 *   SQ_NN: A[M,K], B[K,N], C = A * B     (dX = G * W)
 *   SQ_TN: A[K,M], B[K,N], C = A^T * B   (dW = G^T * X)                        */
typedef enum { SQ_NT = 0, SQ_NN = 1, SQ_TN = 2 } sq_layout;

/* Bias of the fused linear forward. */
typedef enum { SQ_BIAS_NONE = 0, SQ_BIAS_BF16 = 1, SQ_BIAS_FP8 = 2 } sq_bias_kind;

/* Gradients the fused linear backward computes (bit mask, [P3] masks). */
typedef enum { SQ_GRAD_INPUT = 1, SQ_GRAD_WEIGHT = 2, SQ_GRAD_BIAS = 4 } sq_grad_mask;

/* Human-readable name of a status code (static storage, never NULL). */
const char* sq_status_string(sq_status s);

/* Bytes of workspace that sq_quantize_fp8 needs.  The caller allocates it once
 * per stream, 16-byte aligned, and zeroes it once (cudaMemset to 0); every
 * completed call leaves it zeroed again, so no per-call memset is needed. */
size_t sq_workspace_bytes(void);

/*
 * Per-row symmetric INT8 quantization  [P2 formula; P1 per_row / per_head].
 *
 *   amax_r = max_k |x[r,k]|,  s_r = fl32(max(amax_r, 1e-8f) / 127),
 *   q[r,k] = clamp(rne(fl32(x[r,k] / s_r)), -127, 127)
 *
 * with one IEEE float32 division per element and ties rounded to even.
 * Per-head quantization of a (H, N, D) tensor is this call with rows = H*N,
 * cols = D.
 *
 *   x       [rows, cols] with row stride `ld` elements (ld >= cols); float32
 *           (dtype SQ_F32) or bf16 (SQ_BF16).
 *   q       [rows, cols] int8, packed (row stride cols).
 *   scales  [rows] float32.
 * rows == 0 or cols == 0 is a no-op (returns SQ_OK; cols == 0 with rows > 0
 * writes nothing).  Any alignment works; 16-byte aligned rows (x, q 16-B
 * aligned, ld*elemsize and cols multiples of 16) take the vectorised path.
 */
sq_status sq_quantize_rowwise_i8(const void* x, int dtype, int64_t rows, int64_t cols,
                                 int64_t ld, int8_t* q, float* scales, sq_stream stream);

/*
 * Per-tensor FP8 quantization of bf16 with the amax fused in  [P3
 * custom::fp8_quantize; commit notes: the last block to finish completes the
 * amax in the same launch].
 *
 *   x8[i] = enc_fmt(fl32(x[i] / *scale))   (RNE, saturating to +-448 / +-57344)
 *   *amax = max_i |x[i]|                  (raw, no floor; 0 for numel == 0)
 *
 *   x_bf16     [numel] bf16, 16-byte aligned.
 *   scale      device pointer to one float32, the quantization step (> 0).
 *   fmt        SQ_FMT_E4M3 or SQ_FMT_E5M2.
 *   x8         [numel] FP8 codes (uint8), 16-byte aligned.
 *   amax       device pointer to one float32, written by the call.
 *   workspace  sq_workspace_bytes() bytes, zeroed once by the caller.
 */
sq_status sq_quantize_fp8(const uint16_t* x_bf16, int64_t numel, const float* scale, int fmt,
                          uint8_t* x8, float* amax, void* workspace, sq_stream stream);

/*
 * sq_quantize_fp8 on several tensors in one launch  [P3 linear_forward_fp8 /
 * linear_backward_fp8: each operand is quantized with its own step and its
 * amax returned; one launch serves them all].
 *
 *   count        1 .. 4 tensors.
 *   x_bf16[t], numel[t], scale[t], x8[t], amax[t]
 *                tensor t's arguments as in sq_quantize_fp8: device pointers
 *                (x and x8 16-byte aligned), passed in host arrays of count
 *                entries that the call reads before it returns.
 *   fmt          SQ_FMT_E4M3 or SQ_FMT_E5M2, for every tensor.
 *   workspace    sq_workspace_bytes() bytes, zeroed once by the caller; every
 *                completed call leaves it zero.
 * Each tensor's codes and amax are those sq_quantize_fp8 gives it alone.
 * Tensors must not overlap.  Errors: SQ_ERR_INVALID_ARG for a count outside
 * 1 .. 4, a NULL array or entry, or a negative numel; SQ_ERR_ALIGNMENT as in
 * sq_quantize_fp8.
 */
sq_status sq_quantize_fp8_multi(int count, const uint16_t* const* x_bf16, const int64_t* numel,
                                const float* const* scale, int fmt, uint8_t* const* x8,
                                float* const* amax, void* workspace, sq_stream stream);

/*
 * Per-tensor FP8 quantization with delayed scaling kept in a history ring
 * [P3 linear_forward_fp8 / linear_backward_fp8 ring arguments; commit notes:
 * the quantize kernel finishes the ring in its last block, so the next
 * step's scale is published on the device with no extra launch].
 *
 *   ring     float32[hist_len + 2], device: [hist | scale | counter].  The
 *            step used for this call is ring[hist_len].  The counter word
 *            (uint32 bits) must be zero before the first call; every completed
 *            call leaves it zero.
 *   After the codes and the amax are written (as sq_quantize_fp8 does):
 *            hist[idx] = amax;  m = max(hist[0..hist_len));
 *            if m > 0: ring[hist_len] = fl32(fl32(m * 2^margin) / fmt_max)
 *            (fmt_max 448 for E4M3, 57344 for E5M2); else the step is kept.
 *            The pages state no formula; margin > 0 adds headroom and
 *            margin 0 gives the previous-amax / fmt_max delayed recipe.
 *   idx      0 <= idx < hist_len (the caller rolls it, e.g. step % hist_len).
 *   margin   -64 .. 64.
 *   workspace  sq_workspace_bytes() bytes, zeroed once (it holds the running
 *            amax); x_bf16 and x8 16-byte aligned.
 * Calls sharing a ring or a workspace must not overlap on the GPU.
 */
sq_status sq_quantize_fp8_ring(const uint16_t* x_bf16, int64_t numel, int fmt, uint8_t* x8,
                               float* amax, float* ring, int64_t hist_len, int64_t idx, int margin,
                               void* workspace, sq_stream stream);

/*
 * Bytes of workspace that sq_gemm_i8_rowscaled needs for these sizes: the
 * INT8 codes staged as exact 16-bit values for the tensor cores, plus 8 KB in
 * which the staging records bounds on the codes' sums of squares (used to
 * skip the exactness drains when they cannot be needed).
 */
size_t sq_gemm_i8_workspace_bytes(int64_t batch, int64_t M, int64_t N, int64_t K);

/*
 * INT8 GEMM with the per-row x per-row dequantization epilogue  [P1
 * sc_matmul: C = a @ b.T, float32 out, per_row / per_head; P2 codes].
 *
 *   acc[b,i,j] = sum_k A[b,i,k] * B[b,j,k]             (exact, int32)
 *   C[b,i,j]   = fl32(fl32(float(acc) * sA[b*M+i]) * sB[b*N+j])
 *
 *   A        int8 codes, batch b at A + b*strideA, [M,K] packed rows.
 *   B        int8 codes, batch b at B + b*strideB, [N,K] packed rows.
 *            Codes in [-127, 127], as the quantizers produce.  -128 is also
 *            computed exactly, but then K * 128^2 must stay below 2^31.
 *   sA, sB   float32 row scales, [batch*M] and [batch*N].
 *   C        float32, batch b at C + b*strideC, [M,N] packed rows (nullable).
 *   acc_out  int32, same layout as C (nullable).  At least one of C, acc_out.
 *   workspace  sq_gemm_i8_workspace_bytes(batch, M, N, K) bytes, 256-B aligned,
 *              contents need no initialisation.  The call writes the staged
 *              operands and the bounds on their sums of squares there and
 *              reads them back in its last launch, so calls that share a
 *              workspace must not overlap on the GPU.
 * Limits: K a multiple of 16, 1 <= K <= 2^17 (so |acc| < 2^31 for codes in
 * [-127, 127]), strides >= the packed batch sizes; all pointers 16-byte
 * aligned.
 */
sq_status sq_gemm_i8_rowscaled(const int8_t* A, const float* sA, const int8_t* B,
                               const float* sB, int64_t batch, int64_t M, int64_t N, int64_t K,
                               int64_t strideA, int64_t strideB, int64_t strideC, float* C,
                               int32_t* acc_out, void* workspace, size_t workspace_bytes,
                               sq_stream stream);

/*
 * The INT8 GEMM call in two phases, for callers that time or schedule the
 * staging apart from the GEMM.  sq_gemm_i8_rowscaled is exactly
 * sq_gemm_i8_stage followed by sq_gemm_i8_rowscaled_staged on the same
 * workspace and stream, and gives the same bits.
 *
 * sq_gemm_i8_stage writes the codes of A and B (arguments as in
 * sq_gemm_i8_rowscaled) into `workspace` as exact 16-bit values, with the
 * bounds on their sums of squares.
 *
 * sq_gemm_i8_rowscaled_staged runs the GEMM and the dequantization epilogue
 * on a workspace staged earlier in stream order for the same batch, M, N and
 * K, by sq_gemm_i8_stage or by sq_quantize_rowwise_i8_staged (both
 * operands).  The scales and outputs are as in sq_gemm_i8_rowscaled.  A
 * workspace staged once may serve several GEMMs with different scales; the
 * call only reads it.
 */
sq_status sq_gemm_i8_stage(const int8_t* A, const int8_t* B, int64_t batch, int64_t M, int64_t N,
                           int64_t K, int64_t strideA, int64_t strideB, void* workspace,
                           size_t workspace_bytes, sq_stream stream);
sq_status sq_gemm_i8_rowscaled_staged(const float* sA, const float* sB, int64_t batch, int64_t M,
                                      int64_t N, int64_t K, int64_t strideC, float* C,
                                      int32_t* acc_out, const void* workspace,
                                      size_t workspace_bytes, sq_stream stream);

/*
 * Per-row INT8 quantization that also stages the codes for the INT8 GEMM
 * [P2 formula and rounding; P1 per_row / per_head]: the results q and scales
 * of sq_quantize_rowwise_i8 (same arguments, same bits), and besides them
 * the operand's share of an INT8 GEMM workspace, as sq_gemm_i8_stage would
 * write it.  Quantizing A and B this way and then calling
 * sq_gemm_i8_rowscaled_staged gives the bits of sq_gemm_i8_rowscaled on q,
 * with one pass less over the codes.
 *   operand    0: x is A, rows = batch*M; 1: x is B, rows = batch*N.
 *   cols       must equal K.
 *   batch, M, N, K, workspace, workspace_bytes  as in sq_gemm_i8_rowscaled.
 * Calls that share a workspace must not overlap on the GPU.
 */
sq_status sq_quantize_rowwise_i8_staged(const void* x, int dtype, int64_t rows, int64_t cols,
                                        int64_t ld, int8_t* q, float* scales, int operand,
                                        int64_t batch, int64_t M, int64_t N, int64_t K,
                                        void* workspace, size_t workspace_bytes,
                                        sq_stream stream);

/*
 * sq_quantize_rowwise_i8_staged for both operands in one call: A (rows
 * batch*M, row pitch lda elements) and B (rows batch*N, pitch ldb), both of
 * dtype, rows of K elements.  The results are those of the two single calls
 * (operand 0 then 1, same bits); when both operands' rows fit the
 * register-resident kernel they are quantized by one launch.
 *   qa, sa     [batch*M*K] codes and [batch*M] scales of A; qb, sb for B.
 *   batch, M, N, K, workspace, workspace_bytes  as in sq_gemm_i8_rowscaled.
 * Errors as in sq_quantize_rowwise_i8_staged.
 */
sq_status sq_quantize_rowwise_i8_staged_pair(const void* xa, int64_t lda, const void* xb, int64_t ldb,
                                             int dtype, int64_t batch, int64_t M, int64_t N,
                                             int64_t K, int8_t* qa, float* sa, int8_t* qb,
                                             float* sb, void* workspace, size_t workspace_bytes,
                                             sq_stream stream);

/*
 * Row-group symmetric INT8 quantization  [P1 sc_matmul group_a / group_b
 * (row-group size) and per_tensor granularity; P2 formula, which is per
 * tensor].  Consecutive groups of group_rows rows share one scale:
 *
 *   s_g = fl32(max(max|x| over the rows of group g, 1e-8) / 127),
 *   q   = clamp(rne(fl32(x / s_g)), -127, 127)
 *
 * group_rows = 1 is sq_quantize_rowwise_i8; group_rows >= rows is per tensor.
 *   scales    ceil(rows / group_rows) float32.
 *   workspace sq_quantize_grouped_i8_workspace_bytes(rows, group_rows) bytes,
 *             4-byte aligned, no initialisation needed (the call clears the
 *             words it uses with cudaMemsetAsync); unused when group_rows = 1.
 * Other arguments as sq_quantize_rowwise_i8.  Two passes over x (the scale of
 * a group depends on rows that other blocks read).
 */
size_t sq_quantize_grouped_i8_workspace_bytes(int64_t rows, int64_t group_rows);
sq_status sq_quantize_grouped_i8(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                                 int64_t group_rows, int8_t* q, float* scales, void* workspace,
                                 size_t workspace_bytes, sq_stream stream);

/*
 * INT8 GEMM with row-group scales  [P1 sc_matmul group_a / group_b].  As
 * sq_gemm_i8_rowscaled, but the dequantization reads
 *   sA[b*ceil(M/group_a) + i/group_a]  and  sB[b*ceil(N/group_b) + j/group_b];
 * group 1 is per row, group >= M (or N) is per tensor.
 */
sq_status sq_gemm_i8_grouped(const int8_t* A, const float* sA, int64_t group_a, const int8_t* B,
                             const float* sB, int64_t group_b, int64_t batch, int64_t M, int64_t N,
                             int64_t K, int64_t strideA, int64_t strideB, int64_t strideC,
                             float* C, int32_t* acc_out, void* workspace, size_t workspace_bytes,
                             sq_stream stream);

/*
 * Scaled FP8 GEMM  [P3 custom::fp8_gemm: a @ b * (sa * sb), FP32 accumulate,
 * BF16 out; layouts per the commit notes: NT forward, dX and dW].
 *
 *   C[i,j] = bf16_rne(fl32(fl32(acc[i,j] * *sa) * *sb)),  acc in float32
 *
 *   A, B     FP8 codes of the same fmt, laid out per `layout` (see sq_layout).
 *   sa, sb   device pointers to one float32 each (quantization steps).
 *   C_bf16   [M,N] bf16 output, packed rows.
 * Limits: every operand's row length in bytes (K for NT; K and N for NN; M and
 * N for TN) a multiple of 16; pointers 16-byte aligned; M, N, K >= 1.
 */
sq_status sq_gemm_fp8_scaled(const uint8_t* A, const uint8_t* B, const float* sa,
                             const float* sb, int fmt, int layout, int64_t M, int64_t N,
                             int64_t K, uint16_t* C_bf16, sq_stream stream);

/*
 * Two independent scaled FP8 GEMMs in one call  [P3 custom::fp8_gemm; the
 * commit notes' backward, where one quantized gradient G feeds dX = G W (NN)
 * and dW = G^T X (TN)].  Problem i (i = 0, 1) computes exactly what
 *   sq_gemm_fp8_scaled(A[i], B[i], sa[i], sb[i], fmt, layout[i], M[i], N[i],
 *                      K[i], C_bf16[i], stream)
 * computes, with the same arguments, limits and rounding; both share fmt.
 *   A, B, sa, sb, layout, M, N, K, C_bf16   host arrays of two entries each
 *                                            (the pointers in them are device
 *                                            pointers).
 * When the estimate says so, one launch deals the tiles of both problems to
 * every SM (so that a small problem's SMs do not idle while the other runs);
 * otherwise the two run as two launches on the stream.
 * Errors: as sq_gemm_fp8_scaled for each problem, and SQ_ERR_INVALID_ARG when
 * either output overlaps the other problem's operands or output (the
 * problems may run side by side).  Ownership: all buffers are the caller's;
 * the call allocates nothing.
 */
sq_status sq_gemm_fp8_scaled_pair(const uint8_t* const A[2], const uint8_t* const B[2],
                                  const float* const sa[2], const float* const sb[2], int fmt,
                                  const int layout[2], const int64_t M[2], const int64_t N[2],
                                  const int64_t K[2], uint16_t* const C_bf16[2], sq_stream stream);

/*
 * Scaled FP8 GEMM with an FP8 E4M3 output  [P3 custom::fp8_gemm with
 * out_dtype = 1 and mm_fp8(out_dtype="e4m3"): the output is quantized to E4M3
 * with its own step out_scale, for layer-to-layer FP8 pipelines].
 *
 *   C[i,j] = e4m3(fl32(fl32(fl32(acc[i,j] * *sa) * *sb) / *out_scale))
 *
 * with the division rounded as IEEE float32 division and RNE, saturating
 * encoding to +-448.  The pages disagree on whether out_scale multiplies or
 * divides (the adapter's docstring calls it the output quantization step, its
 * CPU path multiplies); this library divides, as for every other step.
 *   out_scale  device pointer to one float32 (> 0).
 *   C_e4m3     [M,N] E4M3 codes (uint8), packed rows, 16-byte aligned.
 * Other arguments and limits as sq_gemm_fp8_scaled.
 */
sq_status sq_gemm_fp8_scaled_e4m3(const uint8_t* A, const uint8_t* B, const float* sa,
                                  const float* sb, int fmt, int layout, int64_t M, int64_t N,
                                  int64_t K, const float* out_scale, uint8_t* C_e4m3,
                                  sq_stream stream);

/*
 * Workspace of the fused linear forward / backward: 256 bytes of quantize and
 * step words and the float32 bias (N).
 * Zero it once (cudaMemset); the calls leave the words they rely on zeroed.
 */
size_t sq_linear_workspace_bytes(int64_t T, int64_t N, int64_t K);

/*
 * Fused FP8 linear forward  [P3 linear_forward_fp8: quantize x and w, FP8
 * GEMM with the bias fused in the epilogue, return (out, x8, w8, amax_x,
 * amax_w); optional rings finish the delayed scaling in the quantize kernels;
 * static weights and bias may arrive pre-quantized].
 *
 *   x8  = enc(x / sx);  w8 = enc(w / sw)  (or w8 = w when w_prequantized)
 *   out[i,j] = bf16(fl32(fl32(fl32(acc[i,j] * sx) * sw) + bias[j]))
 *
 *   x        bf16 [M, K];  w  bf16 [N, K], or FP8 codes [N, K] when
 *            w_prequantized != 0 (then w8 is not written and *amax_w = 0).
 *   bias     nullable per bias_kind: SQ_BIAS_BF16 = bf16 [N]; SQ_BIAS_FP8 =
 *            FP8 codes [N] of fmt, value code * *bias_scale.
 *   sx, sw   device steps; either may be NULL when its ring is given, and
 *            the ring's step slot is then used.
 *   x_ring, w_ring  nullable delayed-scaling rings as in sq_quantize_fp8_ring
 *            (hist, idx, margin alike); the step the quantization used is the
 *            one the GEMM uses, even though the ring publishes the next step.
 *   out      bf16 [M, N];  x8 [M, K];  w8 [N, K];  amax_x, amax_w device floats.
 *   workspace  sq_linear_workspace_bytes(M, N, K) bytes, 256-B aligned,
 *            zeroed once.
 * Limits: K a multiple of 16; pointers 16-byte aligned.
 */
sq_status sq_linear_forward_fp8(const uint16_t* x, int64_t M, int64_t K, const void* w,
                                int w_prequantized, int64_t N, const void* bias, int bias_kind,
                                const float* bias_scale, const float* sx, const float* sw, int fmt,
                                float* x_ring, int64_t x_hist, int64_t x_idx, int x_margin,
                                float* w_ring, int64_t w_hist, int64_t w_idx, int w_margin,
                                uint16_t* out, uint8_t* x8, uint8_t* w8, float* amax_x,
                                float* amax_w, void* workspace, size_t workspace_bytes,
                                sq_stream stream);

/*
 * Fused FP8 linear backward  [P3 linear_backward_fp8: the gradient is
 * quantized once (default E5M2 on the page) and feeds both FP8 products; w and
 * x are quantized to the same fmt; returns (gx, gw, gb, amax_g); masks select
 * the gradients].  For out = x w^T with x [T, K], w [N, K], g = dout [T, N]:
 *
 *   gx = g8 w8  (NN, [T, K]),  gw = g8^T x8  (TN, [N, K]),
 *   gb[j] = bf16(sum_t g[t, j]) (float32 sums over 16 row slabs, added in a
 *   fixed order),  each product scaled and rounded as sq_gemm_fp8_scaled.
 *
 *   masks    SQ_GRAD_INPUT | SQ_GRAD_WEIGHT | SQ_GRAD_BIAS.
 *   sg, sw, sx  device steps (sg may be NULL when g_ring is given).
 *   g8 [T,N], w8 [N,K], x8 [T,K]  caller buffers for the quantized operands
 *            (w8 / x8 needed only for the gradients that use them).
 *   amax_g   device float.  workspace as for the forward.
 * Limits: N and K multiples of 16; pointers 16-byte aligned (gb 4-byte).
 */
sq_status sq_linear_backward_fp8(const uint16_t* g, const uint16_t* x, const uint16_t* w,
                                 int64_t T, int64_t N, int64_t K, int masks, const float* sg,
                                 const float* sw, const float* sx, int fmt, float* g_ring,
                                 int64_t g_hist, int64_t g_idx, int g_margin, uint16_t* gx,
                                 uint16_t* gw, uint16_t* gb, float* amax_g, uint8_t* g8,
                                 uint8_t* w8, uint8_t* x8, void* workspace, size_t workspace_bytes,
                                 sq_stream stream);

/*
 * Diagnostics (no counterpart on the pages): the SM clock that the GEMMs
 * actually run at.  With a buffer set, every later GEMM launch of that kind
 * (FP8 or INT8) on the current device writes, for each of its CTAs below
 * max_ctas, four words at records[4*cta]: the SM cycle counter (clock64) and
 * the global nanosecond timer at the CTA's start and at its end.  The
 * cycles over the nanoseconds are the CTA's mean SM clock.  Each launch
 * overwrites the records of the one before; NULL buffers stop the records.
 * The buffers are device memory of 4 * max_ctas 64-bit words, 8-byte
 * aligned, owned by the caller and read by it after synchronising.
 */
sq_status sq_set_clock_probe(unsigned long long* fp8_records, unsigned long long* i8_records,
                             int max_ctas);

/*
 * Self-test of the failure path every kernel with waits takes: launches one
 * CTA that waits on a barrier phase nothing completes; after limit_ns
 * (1 .. 2e9) the wait gives up, the kernel records SQ_ERR_DEVICE_TIMEOUT in
 * the device error word and returns normally (no trap, the context stays
 * usable).  sq_get_last_device_error() then reports and clears it.  The
 * GEMM kernels' waits behave the same way with a 2 s limit.
 */
sq_status sq_selftest_bounded_wait(uint64_t limit_ns, sq_stream stream);

/*
 * Reads and clears the device-side error word of the current device after
 * synchronising `stream`.  Returns SQ_ERR_DEVICE_TIMEOUT if a kernel gave up
 * on a bounded wait since the last call, SQ_ERR_CUDA on a runtime error,
 * else SQ_OK.
 */
sq_status sq_get_last_device_error(sq_stream stream);

/*
 * INT8 GEMM that allocates nothing: the same computation and results as
 * sq_gemm_i8_rowscaled, but the 16-bit staging copy of A and B lives in a
 * fixed device array inside libsq instead of a caller-provided workspace.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory on the path where they run this GEMM, for
 * example code running inside a host framework or engine that owns the
 * whole device memory pool and hands its plugins only the tensors they
 * operate on, or callers that hold device pointers but no allocator.
 *
 *   Arguments are those of sq_gemm_i8_rowscaled without the workspace.
 *   Limit: the staged operands, (batch*M*K + batch*N*K) * 2 bytes each padded
 *   to 256 B (sq_gemm_i8_workspace_bytes), must fit in
 *   SQ_GEMM_I8_NOALLOC_SCRATCH_BYTES (16 MiB); larger problems return
 *   SQ_ERR_UNSUPPORTED and enqueue nothing.
 *   Memory: every GPU that loads libsq holds the 16 MiB array until the
 *   process exits.  No call makes cudaMalloc, cudaFree or any other
 *   allocating call.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   Sharing: all calls on a device share the one array and it keeps the last
 *   call's contents (each call overwrites what it reads).  Calls that overlap
 *   on the GPU (different streams, or different host threads) race on it and
 *   give wrong results; serialise them on one stream.
 */
#define SQ_GEMM_I8_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
sq_status sq_gemm_i8_rowscaled_noalloc(const int8_t* A, const float* sA, const int8_t* B,
                                       const float* sB, int64_t batch, int64_t M, int64_t N,
                                       int64_t K, int64_t strideA, int64_t strideB,
                                       int64_t strideC, float* C, int32_t* acc_out,
                                       sq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SQ_H_ */
