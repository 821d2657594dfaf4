// Register-only throughput of the warp-level mma.sync instructions (int8 and
// f16 inputs) on the current GPU: the rate an INT8 GEMM built on the legacy
// integer MMA could at best reach, for comparison with the tcgen05 path.
// Built and run by `python bench.py --config legacy_mma`; not part of libsq.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__global__ void s8_loop(int* out, int iters) {
  int d[4][4] = {};
  int a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 ^ 5, a3 = a0 + 7, b0 = a0 * 11, b1 = a0 ^ 9;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[j][0]), "+r"(d[j][1]), "+r"(d[j][2]), "+r"(d[j][3]) : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
  for (int j = 0; j < 4; ++j) s += d[j][0] + d[j][1] + d[j][2] + d[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
__global__ void f16_loop(float* out, int iters) {
  float d[4][4] = {};
  unsigned a0 = 0x3c003c00u, a1 = a0, a2 = a0, a3 = a0, b0 = a0, b1 = a0;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[j][0]), "+f"(d[j][1]), "+f"(d[j][2]), "+f"(d[j][3]) : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0;
  for (int j = 0; j < 4; ++j) s += d[j][0] + d[j][1] + d[j][2] + d[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  int blocks = sms * 4, threads = 256, iters = 20000;
  int* oi; float* of;
  cudaMalloc(&oi, blocks * threads * 4); cudaMalloc(&of, blocks * threads * 4);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  for (int rep = 0; rep < 2; ++rep) {
    s8_loop<<<blocks, threads>>>(oi, iters);
    cudaEventRecord(e0); s8_loop<<<blocks, threads>>>(oi, iters); cudaEventRecord(e1); cudaEventSynchronize(e1);
    float ms; cudaEventElapsedTime(&ms, e0, e1);
    double ops = 2.0 * 16 * 8 * 32 * 4.0 * iters * (blocks * threads / 32);
    if (rep) printf("{\"s8_mma_sync_tops\": %.1f, ", ops / ms / 1e9);
    f16_loop<<<blocks, threads>>>(of, iters);
    cudaEventRecord(e0); f16_loop<<<blocks, threads>>>(of, iters); cudaEventRecord(e1); cudaEventSynchronize(e1);
    cudaEventElapsedTime(&ms, e0, e1);
    ops = 2.0 * 16 * 8 * 16 * 4.0 * iters * (blocks * threads / 32);
    if (rep) printf("\"f16_mma_sync_tflops\": %.1f}\n", ops / ms / 1e9);
  }
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 1;
}
