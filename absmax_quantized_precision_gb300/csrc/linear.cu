// Small kernels of the fused FP8 linear layer (AstrAI ops/fp8.py,
// linear_forward_fp8 and linear_backward_fp8): the bias in float32 for the
// GEMM epilogue, and the bias gradient (column sums of the output gradient).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sq_device.cuh"
#include "sq_host.h"
#include "sq_launch.h"

namespace sq {

__global__ void __launch_bounds__(256) bias_to_f32_kernel(const void* __restrict__ bias, int kind,
                                                          int fmt, const float* __restrict__ step,
                                                          int64_t n, float* __restrict__ out) {
    pdl_begin();
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= n) return;
    if (kind == 1) {
        out[j] = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(bias)[j]) << 16);
    } else {
        // FP8 -> f16 is exact (f16 holds every E4M3 and E5M2 value), f16 -> f32 too
        const uint16_t code = static_cast<const uint8_t*>(bias)[j];
        uint32_t h2;
        if (fmt == 0) asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(code));
        else asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(code));
        const float v = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
        out[j] = __fmul_rn(v, *step);
    }
}

cudaError_t launch_bias_to_f32(const void* bias, int kind, int fmt, const float* step, int64_t n,
                               float* out, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    return launch_pdl(bias_to_f32_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st,
                      1u, bias, kind, fmt, step, n, out);
}

// Block (x, s): columns [512x, 512x + 512) (two per thread, one 4-byte load),
// rows of slab s.  partial[s*N + j] = fp32 sum over the slab.
__global__ void __launch_bounds__(256) colsum_partial_kernel(const uint16_t* __restrict__ g,
                                                             int64_t T, int64_t N, int splits,
                                                             float* __restrict__ partial) {
    pdl_begin();
    const int64_t j = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * 2;
    const int s = blockIdx.y;
    const int64_t rows_per = (T + splits - 1) / splits;
    const int64_t t0 = s * rows_per;
    const int64_t t1 = t0 + rows_per < T ? t0 + rows_per : T;
    if (j >= N) return;
    float a0 = 0.0f, a1 = 0.0f;
    for (int64_t t = t0; t < t1; ++t) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(g + t * N + j);
        a0 = __fadd_rn(a0, __uint_as_float(w << 16));
        a1 = __fadd_rn(a1, __uint_as_float(w & 0xFFFF0000u));
    }
    partial[s * N + j] = a0;
    partial[s * N + j + 1] = a1;
}

__global__ void __launch_bounds__(256) colsum_final_kernel(const float* __restrict__ partial,
                                                           int splits, int64_t N,
                                                           uint16_t* __restrict__ gb) {
    pdl_begin();
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= N) return;
    float a = 0.0f;
    for (int s = 0; s < splits; ++s) a = __fadd_rn(a, partial[s * N + j]);
    gb[j] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
}

cudaError_t launch_colsum_bf16(const uint16_t* g, int64_t T, int64_t N, int splits,
                               float* partial, uint16_t* gb, cudaStream_t st) {
    if (N <= 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((N / 2 + 255) / 256), static_cast<unsigned>(splits));
    const cudaError_t e = launch_pdl(colsum_partial_kernel, grid, dim3(256), 0, st, 1u, g, T, N, splits, partial);
    if (e != cudaSuccess) return e;
    const float* cpartial = partial;
    return launch_pdl(colsum_final_kernel, dim3(static_cast<unsigned>((N + 255) / 256)), dim3(256), 0, st,
                      1u, cpartial, splits, N, gb);
}

// Self-test of the bounded waits: one CTA waits for a barrier phase that
// nothing completes; the wait gives up after limit_ns, records the timeout in
// the device error word and the kernel returns normally.
__global__ void selftest_wait_kernel(unsigned* err_word, unsigned long long limit_ns) {
    pdl_begin();
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &abort_flag, err_word, limit_ns);
}

cudaError_t launch_selftest_wait(unsigned* err_word, unsigned long long limit_ns, cudaStream_t st) {
    return launch_pdl(selftest_wait_kernel, dim3(1), dim3(32), 0, st, 1u, err_word, limit_ns);
}

}  // namespace sq
