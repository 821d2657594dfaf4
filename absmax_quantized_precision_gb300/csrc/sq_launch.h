// Host-side launchers behind the C ABI (internal to libsq).  Arguments are
// already validated by the entry points in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sq {

// Bound region of an INT8 GEMM workspace, one per operand: a header word,
// then one slot per CTA of the launch that staged the operand.  The header
// holds the number of slots written (0: no bound recorded) and, in
// kBoundRowNorms, whether each slot is a largest row norm (the sum of a
// row's squared codes) or a largest sum of squared codes over a staged chunk
// of 1024 codes.  Each staging launch writes its header and its slots, so the
// region needs no initialisation.
constexpr int kBoundSlots = 1024;                 // words per operand region
constexpr unsigned kBoundCountMask = 0xFFFFu;
constexpr unsigned kBoundRowNorms = 0x80000000u;

// err_word == nullptr keeps to the kernels without waits.
cudaError_t launch_quantize_rowwise_i8(const void* x, int dtype, int64_t rows, int64_t cols,
                                       int64_t ld, int8_t* q, float* scales, bool vec_ok,
                                       unsigned* err_word, cudaStream_t st, int sms);

// Row groups of group_rows rows share one scale; ws holds ceil(rows/group_rows)
// words (zeroed by the launcher with cudaMemsetAsync).
cudaError_t launch_quantize_grouped_i8(const void* x, int dtype, int64_t rows, int64_t cols,
                                       int64_t ld, int64_t group_rows, int8_t* q, float* scales,
                                       unsigned* ws, bool vec_ok, cudaStream_t st, int sms);

// ring == nullptr: plain per-tensor quantize with step *scale.  Otherwise
// delayed scaling with ring = [hist (hist_len) | scale | counter].
cudaError_t launch_quantize_fp8(const uint16_t* x, int64_t n, const float* scale, int fmt,
                                uint8_t* x8, float* amax, unsigned* ws, float* ring, int hist_len,
                                int ring_idx, int margin, unsigned* err_word, cudaStream_t st,
                                int sms);

// Up to four tensors in one launch, each with its own step and amax; the
// workspace words are shared (amax of tensor t in word 0 or t + 1).
cudaError_t launch_quantize_fp8_multi(int count, const uint16_t* const* x, const int64_t* n,
                                      const float* const* scale, int fmt, uint8_t* const* x8,
                                      float* const* amax, unsigned* ws, unsigned* err_word,
                                      cudaStream_t st, int sms);

// The same with a delayed-scaling ring per tensor (ring[t] nullable; the step
// comes from the ring when scale[t] is null) and, in used[t] (nullable), the
// step each tensor used.  The ticket is workspace word 1.
cudaError_t launch_quantize_fp8_rings(int count, const uint16_t* const* x, const int64_t* n,
                                      const float* const* scale, float* const* ring,
                                      const int* hist, const int* idx, const int* margin,
                                      float* const* used, int fmt, uint8_t* const* x8,
                                      float* const* amax, unsigned* ws, unsigned* err_word,
                                      cudaStream_t st, int sms);

// Staging of the INT8 codes of both GEMM operands as exact fp16 values:
// a16[b][r][k] = a[b*stride_a + r*K + k] (M rows per batch), likewise b16.
// An operand that is contiguous and large takes the bulk pipeline, whose CTAs
// record in its bound region (kBoundSlots words) the largest sum of squared
// codes over any of their 1024-code chunks (the ragged tail counts as one
// chunk); the other operands share one launch of a plain kernel, which marks
// their regions as holding no bound.
cudaError_t launch_i8_to_f16_pair(const int8_t* a, int64_t M, const int8_t* b, int64_t N,
                                  int64_t batch, int64_t K, int64_t stride_a, int64_t stride_b,
                                  uint16_t* a16, uint16_t* b16, unsigned* bound_a,
                                  unsigned* bound_b, unsigned* err_word, cudaStream_t st,
                                  int sms);

// The same for one operand.
cudaError_t launch_i8_to_f16_one(const int8_t* src, int64_t batch, int64_t rows, int64_t K,
                                 int64_t stride, uint16_t* dst, unsigned* bound,
                                 unsigned* err_word, cudaStream_t st, int sms);

// Per-row INT8 quantization that also stages the codes for the GEMM: besides
// q and scales, q16[r*cols + k] = the code as an exact fp16 value, and the
// operand's bound region records the largest row norm (the sum of a row's
// squared codes) per CTA.  Rows packed (ld == cols) in q16.  Shapes that the
// fused kernel does not take go through the plain quantize and
// launch_i8_to_f16_one.
cudaError_t launch_quantize_rowwise_i8_staged(const void* x, int dtype, int64_t rows,
                                              int64_t cols, int64_t ld, int8_t* q,
                                              float* scales, bool vec_ok, uint16_t* q16,
                                              unsigned* bound, unsigned* err_word,
                                              cudaStream_t st, int sms);

// Both INT8 GEMM operands quantized and staged: one launch when both take the
// register-resident kernel, else as two calls of the above.
cudaError_t launch_quantize_rowwise_i8_staged_pair(const void* xa, int64_t rows_a, int64_t lda,
                                                   int8_t* qa, float* sa, bool vec_ok_a,
                                                   uint16_t* a16, unsigned* bound_a, const void* xb,
                                                   int64_t rows_b, int64_t ldb, int8_t* qb, float* sb,
                                                   bool vec_ok_b, uint16_t* b16, unsigned* bound_b,
                                                   int dtype, int64_t cols, unsigned* err_word,
                                                   cudaStream_t st, int sms);

// 0 on success, a cudaError_t otherwise; CUDA_ERROR_* from tensor-map encoding
// is reported as cudaErrorInvalidValue.
// C is bf16 [M,N] when out_scale == nullptr, else E4M3 codes [M,N] with the
// output step *out_scale divided out.
cudaError_t launch_gemm_fp8(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            int fmt, int layout, int M, int N, int K, void* C,
                            const float* out_scale, const float* bias, unsigned* err_word,
                            cudaStream_t st, int sms);

// One problem of a grouped FP8 launch (bf16 output, no bias).
struct Fp8Problem {
    const uint8_t* A;
    const uint8_t* B;
    const float* sa;
    const float* sb;
    int layout;           // 0 NT, 1 NN, 2 TN
    int M, N, K;
    void* C;
};

// Two independent FP8 GEMMs: one launch that deals both problems' tiles to
// every SM when that is estimated faster, else two ordinary launches.
cudaError_t launch_gemm_fp8_pair(const Fp8Problem* q, int fmt, unsigned* err_word, cudaStream_t st,
                                 int sms);

// Linear-layer helpers (linear.cu).
// bias kind 1: bf16 [n] widened; kind 2: FP8 codes of fmt times *step.
cudaError_t launch_bias_to_f32(const void* bias, int kind, int fmt, const float* step, int64_t n,
                               float* out, cudaStream_t st);
// gb[j] = bf16(sum_t g[t*N + j]) (N % 8 == 0), in one launch: fp32 sums
// over row slabs, then the slabs added in a fixed order.
cudaError_t launch_colsum_bf16(const uint16_t* g, int64_t T, int64_t N, uint16_t* gb, cudaStream_t st);

// Scales of row i of A in batch b: sA[b*ceil(M/ga) + i/ga] (ga = 1: per row).
// bound_a / bound_b: the operands' bound regions (nullable: no bound); when
// they prove every partial sum exact in fp32, K runs as one chunk.
cudaError_t launch_gemm_i8(const uint16_t* A16, const uint16_t* B16, const float* sA,
                           const float* sB, int ga, int gb, int batch, int M, int N, int K,
                           int64_t strideC, float* C, int32_t* acc_out, const unsigned* bound_a,
                           const unsigned* bound_b, unsigned* err_word, cudaStream_t st, int sms);

// Diagnostics: where the GEMM launches on the current device record their
// CTAs' clocks (nullable; cap records of 4 words each).
cudaError_t set_gemm_clock_probe(unsigned long long* fp8, unsigned long long* i8, int cap);

// One CTA waits on a barrier phase that never completes, for limit_ns.
cudaError_t launch_selftest_wait(unsigned* err_word, unsigned long long limit_ns, cudaStream_t st);

}  // namespace sq
