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

// Bias gradient gb[j] = bf16(sum_t g[t*N + j]) in one launch.  Cluster x
// (kColsumSlabs CTAs along y) owns the columns [128x, 128x + 128); CTA s of
// it sums them over row slab s:
// - each half-warp covers the 128 columns, lane l holding the 8 columns
//   [128x + 8(l % 16), +8) (one 16-byte load per row);
// - row stream q = 2w + l / 16 of warp w adds rows t0 + q, t0 + q + 32, ...
//   in increasing order, eight rows' loads in flight at a time;
// - the CTA adds its 32 row streams' sums in stream order into sums[128].
// After a cluster barrier, CTA s adds, for its 16 columns [128x + 16s, +16),
// the slabs' sums in slab order, read through distributed shared memory, and
// writes the bf16 result.  A second barrier keeps every CTA's sums alive until
// they are read.  The order of every addition is fixed, so the result is the
// same on every call.  N % 8 == 0, g 16-byte aligned.
constexpr int kColsumSlabs = 8;    // CTAs per cluster, one row slab each
constexpr int kColsumWarps = 16;
constexpr int kColsumStreams = 2 * kColsumWarps;   // row streams per CTA
constexpr int kColsumCols = 128;   // columns per cluster
constexpr int kColsumRows = 8;     // rows whose loads a thread keeps in flight
__global__ void __cluster_dims__(1, kColsumSlabs, 1) __launch_bounds__(kColsumWarps * 32)
    colsum_kernel(const uint16_t* __restrict__ g, int64_t T, int64_t N, uint16_t* __restrict__ gb) {
    pdl_begin();
    __shared__ float red[kColsumStreams][kColsumCols];
    __shared__ float sums[kColsumCols];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = 2 * warp + (lane >> 4);              // this thread's row stream
    const int cl = 8 * (lane & 15);                    // its first column in the block
    const int s = blockIdx.y;
    const int64_t rows_per = (T + kColsumSlabs - 1) / kColsumSlabs;
    const int64_t t0 = s * rows_per;
    const int64_t t1 = t0 + rows_per < T ? t0 + rows_per : T;
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kColsumCols + cl;
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.0f;
    auto add = [&](const uint4& v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] = __fadd_rn(a[2 * i], __uint_as_float(w[i] << 16));
            a[2 * i + 1] = __fadd_rn(a[2 * i + 1], __uint_as_float(w[i] & 0xFFFF0000u));
        }
    };
    if (j0 < N) {
        const uint16_t* col = g + j0;
        int64_t t = t0 + q;
        for (; t + (kColsumRows - 1) * kColsumStreams < t1; t += kColsumRows * kColsumStreams) {
            uint4 v[kColsumRows];
#pragma unroll
            for (int r = 0; r < kColsumRows; ++r)
                v[r] = *reinterpret_cast<const uint4*>(col + (t + r * kColsumStreams) * N);
#pragma unroll
            for (int r = 0; r < kColsumRows; ++r) add(v[r]);
        }
        for (; t < t1; t += kColsumStreams) add(*reinterpret_cast<const uint4*>(col + t * N));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[q][cl + i] = a[i];
    __syncthreads();
    if (threadIdx.x < kColsumCols) {
        float sum = red[0][threadIdx.x];
#pragma unroll
        for (int r = 1; r < kColsumStreams; ++r) sum = __fadd_rn(sum, red[r][threadIdx.x]);
        sums[threadIdx.x] = sum;
    }
    cluster_sync_all();   // every slab's sums written and visible in the cluster
    constexpr int kPer = kColsumCols / kColsumSlabs;   // columns each CTA finishes
    if (threadIdx.x < kPer) {
        const int c = kPer * s + static_cast<int>(threadIdx.x);
        const int64_t j = static_cast<int64_t>(blockIdx.x) * kColsumCols + c;
        float sum = 0.0f;
#pragma unroll
        for (int r = 0; r < kColsumSlabs; ++r) {
            float v;
            asm volatile("ld.shared::cluster.f32 %0, [%1];"
                         : "=f"(v)
                         : "r"(cluster_addr(&sums[c], static_cast<uint32_t>(r)))
                         : "memory");
            sum = r == 0 ? v : __fadd_rn(sum, v);
        }
        if (j < N) gb[j] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
    }
    cluster_sync_all();   // no CTA leaves while another reads its sums
}

cudaError_t launch_colsum_bf16(const uint16_t* g, int64_t T, int64_t N, uint16_t* gb, cudaStream_t st) {
    if (N <= 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((N + kColsumCols - 1) / kColsumCols),
                    static_cast<unsigned>(kColsumSlabs));
    return launch_pdl(colsum_kernel, grid, dim3(kColsumWarps * 32), 0, st, 1u, g, T, N, gb);
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
