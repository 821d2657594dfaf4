// Host-side launchers behind the C ABI (internal to libsq).  Arguments are
// already validated by the entry points in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sq {

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

// Staging of the INT8 codes of both GEMM operands as exact fp16 values:
// a16[b][r][k] = a[b*stride_a + r*K + k] (M rows per batch), likewise b16.
// An operand that is contiguous and large takes the bulk pipeline, whose
// *nparts CTAs each write to parts[cta] the largest sum of squared codes over
// any of their 1024-code chunks (the ragged tail counts as one chunk); the
// other operands share one launch of a plain kernel and report *nparts = 0.
// parts_a and parts_b hold at least 256 words each.
// The *nparts that launch_i8_to_f16_pair reports for one operand of these
// sizes (0: it takes the plain kernel and records no bounds).  Every launch
// that passes an error word takes the bulk pipeline when this is non-zero.
int i8_staging_parts(int64_t batch, int64_t rows, int64_t K, int64_t stride, int sms);

cudaError_t launch_i8_to_f16_pair(const int8_t* a, int64_t M, const int8_t* b, int64_t N,
                                  int64_t batch, int64_t K, int64_t stride_a, int64_t stride_b,
                                  uint16_t* a16, uint16_t* b16, unsigned* parts_a, int* nparts_a,
                                  unsigned* parts_b, int* nparts_b, unsigned* err_word,
                                  cudaStream_t st, int sms);

// 0 on success, a cudaError_t otherwise; CUDA_ERROR_* from tensor-map encoding
// is reported as cudaErrorInvalidValue.
// C is bf16 [M,N] when out_scale == nullptr, else E4M3 codes [M,N] with the
// output step *out_scale divided out.
cudaError_t launch_gemm_fp8(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            int fmt, int layout, int M, int N, int K, void* C,
                            const float* out_scale, const float* bias, unsigned* err_word,
                            cudaStream_t st, int sms);

// Linear-layer helpers (linear.cu).
// bias kind 1: bf16 [n] widened; kind 2: FP8 codes of fmt times *step.
cudaError_t launch_bias_to_f32(const void* bias, int kind, int fmt, const float* step, int64_t n,
                               float* out, cudaStream_t st);
// gb[j] = bf16(sum_t g[t*N + j]): fp32 partial sums over `splits` row slabs in
// `partial` (splits * N floats), then a fixed-order sum of the slabs.
cudaError_t launch_colsum_bf16(const uint16_t* g, int64_t T, int64_t N, int splits,
                               float* partial, uint16_t* gb, cudaStream_t st);

// Scales of row i of A in batch b: sA[b*ceil(M/ga) + i/ga] (ga = 1: per row).
// bound_a / bound_b: the staging launches' parts (nparts 0: not available);
// when they prove every partial sum exact in fp32, K runs as one chunk.
cudaError_t launch_gemm_i8(const uint16_t* A16, const uint16_t* B16, const float* sA,
                           const float* sB, int ga, int gb, int batch, int M, int N, int K,
                           int64_t strideC, float* C, int32_t* acc_out, const unsigned* bound_a,
                           int nparts_a, const unsigned* bound_b, int nparts_b,
                           unsigned* err_word, cudaStream_t st, int sms);

// One CTA waits on a barrier phase that never completes, for limit_ns.
cudaError_t launch_selftest_wait(unsigned* err_word, unsigned long long limit_ns, cudaStream_t st);

}  // namespace sq
