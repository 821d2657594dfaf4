// C ABI of libsq (declared in include/sq.h): argument checks, per-device
// state, and dispatch to the launchers.  No entry point allocates, frees or
// synchronises on its hot path.
#include <cuda_runtime.h>

#include <mutex>

#include "sq.h"
#include "sq_launch.h"

// Device error word of this library, one per device.
static __device__ unsigned g_sq_device_error = 0;

// Staging scratch of sq_gemm_i8_rowscaled_noalloc.  Every device that loads
// the library holds its own copy until the process exits.  Host code must not
// hand this name to a kernel: on the host it only stands in for the symbol;
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_sq_noalloc_scratch[SQ_GEMM_I8_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    int sms = 0;
    unsigned* err_word = nullptr;
    cudaError_t init_err = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

// SM count and the device address of the error word for the current device.
DeviceState* device_state(cudaError_t* err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    DeviceState& s = g_dev[dev];
    std::call_once(s.once, [&] {
        s.init_err = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev);
        if (s.init_err == cudaSuccess)
            s.init_err = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err_word), g_sq_device_error);
    });
    if (s.init_err != cudaSuccess) {
        *err = s.init_err;
        return nullptr;
    }
    return &s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SQ_OK : SQ_ERR_CUDA; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

}  // namespace

extern "C" {

const char* sq_status_string(sq_status s) {
    switch (s) {
        case SQ_OK: return "SQ_OK";
        case SQ_ERR_INVALID_ARG: return "SQ_ERR_INVALID_ARG: invalid size, pointer, dtype, fmt or layout";
        case SQ_ERR_UNSUPPORTED: return "SQ_ERR_UNSUPPORTED: valid but outside this library's limits";
        case SQ_ERR_ALIGNMENT: return "SQ_ERR_ALIGNMENT: a pointer or row length breaks the 16-byte rule";
        case SQ_ERR_CUDA: return "SQ_ERR_CUDA: the CUDA runtime reported an error";
        case SQ_ERR_DEVICE_TIMEOUT: return "SQ_ERR_DEVICE_TIMEOUT: a kernel gave up on a bounded wait";
    }
    return "SQ_ERR_UNKNOWN";
}

size_t sq_workspace_bytes(void) { return 256; }

sq_status sq_quantize_rowwise_i8(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                                 int8_t* q, float* scales, sq_stream stream) {
    if (dtype != SQ_F32 && dtype != SQ_BF16) return SQ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ld < cols) return SQ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return SQ_OK;
    if (!x || !q || !scales) return SQ_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    const int64_t esz = dtype == SQ_F32 ? 4 : 2;
    const bool vec_ok = aligned16(x) && aligned16(q) && ((ld * esz) % 16 == 0) && (cols % 16 == 0);
    return from_cuda(sq::launch_quantize_rowwise_i8(x, dtype, rows, cols, ld, q, scales, vec_ok,
                                                    ds->err_word,
                                                    reinterpret_cast<cudaStream_t>(stream), ds->sms));
}

sq_status sq_quantize_fp8(const uint16_t* x_bf16, int64_t numel, const float* scale, int fmt,
                          uint8_t* x8, float* amax, void* workspace, sq_stream stream) {
    if (fmt != SQ_FMT_E4M3 && fmt != SQ_FMT_E5M2) return SQ_ERR_INVALID_ARG;
    if (numel < 0 || !scale || !amax || !workspace) return SQ_ERR_INVALID_ARG;
    if (numel > 0 && (!x_bf16 || !x8)) return SQ_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(x8) || !aligned16(workspace)) return SQ_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return from_cuda(sq::launch_quantize_fp8(x_bf16, numel, scale, fmt, x8, amax,
                                             static_cast<unsigned*>(workspace), nullptr, 0, 0, 0,
                                             ds->err_word, reinterpret_cast<cudaStream_t>(stream),
                                             ds->sms));
}

sq_status sq_quantize_fp8_multi(int count, const uint16_t* const* x_bf16, const int64_t* numel,
                                const float* const* scale, int fmt, uint8_t* const* x8,
                                float* const* amax, void* workspace, sq_stream stream) {
    if (fmt != SQ_FMT_E4M3 && fmt != SQ_FMT_E5M2) return SQ_ERR_INVALID_ARG;
    if (count < 1 || count > 4 || !x_bf16 || !numel || !scale || !x8 || !amax || !workspace)
        return SQ_ERR_INVALID_ARG;
    for (int t = 0; t < count; ++t) {
        if (numel[t] < 0 || !scale[t] || !amax[t]) return SQ_ERR_INVALID_ARG;
        if (numel[t] > 0 && (!x_bf16[t] || !x8[t])) return SQ_ERR_INVALID_ARG;
        if (!aligned16(x_bf16[t]) || !aligned16(x8[t])) return SQ_ERR_ALIGNMENT;
    }
    if (!aligned16(workspace)) return SQ_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return from_cuda(sq::launch_quantize_fp8_multi(count, x_bf16, numel, scale, fmt, x8, amax,
                                                   static_cast<unsigned*>(workspace), ds->err_word,
                                                   reinterpret_cast<cudaStream_t>(stream), ds->sms));
}

sq_status sq_quantize_fp8_ring(const uint16_t* x_bf16, int64_t numel, int fmt, uint8_t* x8,
                               float* amax, float* ring, int64_t hist_len, int64_t idx, int margin,
                               void* workspace, sq_stream stream) {
    if (fmt != SQ_FMT_E4M3 && fmt != SQ_FMT_E5M2) return SQ_ERR_INVALID_ARG;
    if (numel < 0 || !amax || !ring || !workspace) return SQ_ERR_INVALID_ARG;
    if (numel > 0 && (!x_bf16 || !x8)) return SQ_ERR_INVALID_ARG;
    if (hist_len < 1 || hist_len > (int64_t(1) << 20) || idx < 0 || idx >= hist_len)
        return SQ_ERR_INVALID_ARG;
    if (margin < -64 || margin > 64) return SQ_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(x8) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(ring) & 3u))
        return SQ_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return from_cuda(sq::launch_quantize_fp8(x_bf16, numel, nullptr, fmt, x8, amax,
                                             static_cast<unsigned*>(workspace), ring,
                                             static_cast<int>(hist_len), static_cast<int>(idx),
                                             margin, ds->err_word,
                                             reinterpret_cast<cudaStream_t>(stream), ds->sms));
}

// fp16 copies of A and B, then the two operands' bound regions
constexpr size_t kI8BoundBytes = 2 * sq::kBoundSlots * sizeof(unsigned);

size_t sq_gemm_i8_workspace_bytes(int64_t batch, int64_t M, int64_t N, int64_t K) {
    if (batch <= 0 || M <= 0 || N <= 0 || K <= 0) return 0;
    const size_t a = static_cast<size_t>(batch) * M * K * 2;
    const size_t b = static_cast<size_t>(batch) * N * K * 2;
    return ((a + 255) & ~static_cast<size_t>(255)) + ((b + 255) & ~static_cast<size_t>(255)) +
           kI8BoundBytes;
}

namespace {

// Where the staged operands and their bounds sit in an INT8 GEMM workspace.
struct I8Workspace {
    uint16_t* A16;
    uint16_t* B16;
    unsigned* bound_a;
    unsigned* bound_b;
};

I8Workspace i8_workspace(void* workspace, int64_t batch, int64_t M, int64_t N, int64_t K) {
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const size_t abytes = (static_cast<size_t>(batch) * M * K * 2 + 255) & ~static_cast<size_t>(255);
    const size_t bbytes = (static_cast<size_t>(batch) * N * K * 2 + 255) & ~static_cast<size_t>(255);
    unsigned* bound_a = reinterpret_cast<unsigned*>(w + abytes + bbytes);
    return I8Workspace{reinterpret_cast<uint16_t*>(w), reinterpret_cast<uint16_t*>(w + abytes),
                       bound_a, bound_a + sq::kBoundSlots};
}

// Checks shared by both phases of the INT8 GEMM: sizes, strides of the int8
// operands and the workspace.
sq_status i8_check_common(int64_t batch, int64_t M, int64_t N, int64_t K, int64_t strideA,
                          int64_t strideB, const void* workspace, size_t workspace_bytes) {
    if (batch < 1 || M < 1 || N < 1 || K < 1) return SQ_ERR_INVALID_ARG;
    if (!workspace) return SQ_ERR_INVALID_ARG;
    if (strideA < M * K || strideB < N * K) return SQ_ERR_INVALID_ARG;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (K > (int64_t(1) << 17)) return SQ_ERR_UNSUPPORTED;
    if (batch > 65535 || M > kMaxDim || N > kMaxDim) return SQ_ERR_UNSUPPORTED;
    if (strideA % 16 != 0 || strideB % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SQ_ERR_ALIGNMENT;
    if (workspace_bytes < sq_gemm_i8_workspace_bytes(batch, M, N, K)) return SQ_ERR_INVALID_ARG;
    const int64_t mt = (M + 127) / 128, nt = (N + 127) / 128;
    if (mt * nt * batch > kMaxDim) return SQ_ERR_UNSUPPORTED;
    return SQ_OK;
}

// Phase 1: the int8 codes of A and B staged as exact fp16 in the workspace,
// with the per-CTA bounds on their sums of squares.
sq_status i8_stage(const int8_t* A, const int8_t* B, int64_t batch, int64_t M, int64_t N,
                   int64_t K, int64_t strideA, int64_t strideB, void* workspace,
                   DeviceState* ds, cudaStream_t st) {
    const I8Workspace w = i8_workspace(workspace, batch, M, N, K);
    return from_cuda(sq::launch_i8_to_f16_pair(A, M, B, N, batch, K, strideA, strideB, w.A16, w.B16,
                                               w.bound_a, w.bound_b, ds->err_word, st, ds->sms));
}

// Phase 2: the GEMM on the staged operands with the dequantization epilogue.
// The staging recorded its bounds (or none) in the workspace.
sq_status i8_gemm_staged(const float* sA, int64_t ga, const float* sB, int64_t gb, int64_t batch,
                         int64_t M, int64_t N, int64_t K, int64_t strideC, float* C,
                         int32_t* acc_out, const void* workspace, DeviceState* ds,
                         cudaStream_t st) {
    if (ga > M) ga = M;
    if (gb > N) gb = N;
    const I8Workspace w = i8_workspace(const_cast<void*>(workspace), batch, M, N, K);
    return from_cuda(sq::launch_gemm_i8(w.A16, w.B16, sA, sB, static_cast<int>(ga),
                                        static_cast<int>(gb), static_cast<int>(batch),
                                        static_cast<int>(M), static_cast<int>(N),
                                        static_cast<int>(K), strideC, C, acc_out, w.bound_a,
                                        w.bound_b, ds->err_word, st, ds->sms));
}

sq_status i8_check_outputs(const float* sA, const float* sB, int64_t M, int64_t N,
                           int64_t strideC, const float* C, const int32_t* acc_out, int64_t ga,
                           int64_t gb) {
    if (!sA || !sB || (!C && !acc_out) || ga < 1 || gb < 1) return SQ_ERR_INVALID_ARG;
    if (strideC < M * N) return SQ_ERR_INVALID_ARG;
    if (!aligned16(C) || !aligned16(acc_out)) return SQ_ERR_ALIGNMENT;
    return SQ_OK;
}

sq_status gemm_i8_common(const int8_t* A, const float* sA, int64_t ga, const int8_t* B,
                         const float* sB, int64_t gb, int64_t batch, int64_t M, int64_t N,
                         int64_t K, int64_t strideA, int64_t strideB, int64_t strideC, float* C,
                         int32_t* acc_out, void* workspace, size_t workspace_bytes,
                         sq_stream stream) {
    sq_status r = i8_check_common(batch, M, N, K, strideA, strideB, workspace, workspace_bytes);
    if (r != SQ_OK) return r;
    if (!A || !B) return SQ_ERR_INVALID_ARG;
    r = i8_check_outputs(sA, sB, M, N, strideC, C, acc_out, ga, gb);
    if (r != SQ_OK) return r;
    if (!aligned16(A) || !aligned16(B)) return SQ_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    r = i8_stage(A, B, batch, M, N, K, strideA, strideB, workspace, ds, st);
    if (r != SQ_OK) return r;
    return i8_gemm_staged(sA, ga, sB, gb, batch, M, N, K, strideC, C, acc_out, workspace, ds, st);
}

}  // namespace

sq_status sq_gemm_i8_stage(const int8_t* A, const int8_t* B, int64_t batch, int64_t M, int64_t N,
                           int64_t K, int64_t strideA, int64_t strideB, void* workspace,
                           size_t workspace_bytes, sq_stream stream) {
    sq_status r = i8_check_common(batch, M, N, K, strideA, strideB, workspace, workspace_bytes);
    if (r != SQ_OK) return r;
    if (!A || !B) return SQ_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B)) return SQ_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return i8_stage(A, B, batch, M, N, K, strideA, strideB, workspace, ds,
                    reinterpret_cast<cudaStream_t>(stream));
}

sq_status sq_gemm_i8_rowscaled_staged(const float* sA, const float* sB, int64_t batch, int64_t M,
                                      int64_t N, int64_t K, int64_t strideC, float* C,
                                      int32_t* acc_out, const void* workspace,
                                      size_t workspace_bytes, sq_stream stream) {
    sq_status r = i8_check_common(batch, M, N, K, M * K, N * K, workspace, workspace_bytes);
    if (r != SQ_OK) return r;
    r = i8_check_outputs(sA, sB, M, N, strideC, C, acc_out, 1, 1);
    if (r != SQ_OK) return r;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return i8_gemm_staged(sA, 1, sB, 1, batch, M, N, K, strideC, C, acc_out, workspace, ds,
                          reinterpret_cast<cudaStream_t>(stream));
}

sq_status sq_quantize_rowwise_i8_staged(const void* x, int dtype, int64_t rows, int64_t cols,
                                        int64_t ld, int8_t* q, float* scales, int operand,
                                        int64_t batch, int64_t M, int64_t N, int64_t K,
                                        void* workspace, size_t workspace_bytes,
                                        sq_stream stream) {
    if (dtype != SQ_F32 && dtype != SQ_BF16) return SQ_ERR_INVALID_ARG;
    if (operand != 0 && operand != 1) return SQ_ERR_INVALID_ARG;
    sq_status r = i8_check_common(batch, M, N, K, M * K, N * K, workspace, workspace_bytes);
    if (r != SQ_OK) return r;
    if (rows != batch * (operand ? N : M) || cols != K || ld < cols) return SQ_ERR_INVALID_ARG;
    if (!x || !q || !scales) return SQ_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    const int64_t esz = dtype == SQ_F32 ? 4 : 2;
    const bool vec_ok = aligned16(x) && aligned16(q) && ((ld * esz) % 16 == 0) && (cols % 16 == 0);
    const I8Workspace w = i8_workspace(workspace, batch, M, N, K);
    return from_cuda(sq::launch_quantize_rowwise_i8_staged(
        x, dtype, rows, cols, ld, q, scales, vec_ok, operand ? w.B16 : w.A16,
        operand ? w.bound_b : w.bound_a, ds->err_word, reinterpret_cast<cudaStream_t>(stream),
        ds->sms));
}

sq_status sq_quantize_rowwise_i8_staged_pair(const void* xa, int64_t lda, const void* xb, int64_t ldb,
                                             int dtype, int64_t batch, int64_t M, int64_t N,
                                             int64_t K, int8_t* qa, float* sa, int8_t* qb,
                                             float* sb, void* workspace, size_t workspace_bytes,
                                             sq_stream stream) {
    if (dtype != SQ_F32 && dtype != SQ_BF16) return SQ_ERR_INVALID_ARG;
    sq_status r = i8_check_common(batch, M, N, K, M * K, N * K, workspace, workspace_bytes);
    if (r != SQ_OK) return r;
    if (lda < K || ldb < K) return SQ_ERR_INVALID_ARG;
    if (!xa || !qa || !sa || !xb || !qb || !sb) return SQ_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    const int64_t esz = dtype == SQ_F32 ? 4 : 2;
    const bool vec_a = aligned16(xa) && aligned16(qa) && ((lda * esz) % 16 == 0) && (K % 16 == 0);
    const bool vec_b = aligned16(xb) && aligned16(qb) && ((ldb * esz) % 16 == 0) && (K % 16 == 0);
    const I8Workspace w = i8_workspace(workspace, batch, M, N, K);
    return from_cuda(sq::launch_quantize_rowwise_i8_staged_pair(
        xa, batch * M, lda, qa, sa, vec_a, w.A16, w.bound_a, xb, batch * N, ldb, qb, sb, vec_b,
        w.B16, w.bound_b, dtype, K, ds->err_word, reinterpret_cast<cudaStream_t>(stream), ds->sms));
}

sq_status sq_gemm_i8_rowscaled(const int8_t* A, const float* sA, const int8_t* B, const float* sB,
                               int64_t batch, int64_t M, int64_t N, int64_t K, int64_t strideA,
                               int64_t strideB, int64_t strideC, float* C, int32_t* acc_out,
                               void* workspace, size_t workspace_bytes, sq_stream stream) {
    return gemm_i8_common(A, sA, 1, B, sB, 1, batch, M, N, K, strideA, strideB, strideC, C,
                          acc_out, workspace, workspace_bytes, stream);
}

sq_status sq_gemm_i8_grouped(const int8_t* A, const float* sA, int64_t group_a, const int8_t* B,
                             const float* sB, int64_t group_b, int64_t batch, int64_t M, int64_t N,
                             int64_t K, int64_t strideA, int64_t strideB, int64_t strideC,
                             float* C, int32_t* acc_out, void* workspace, size_t workspace_bytes,
                             sq_stream stream) {
    return gemm_i8_common(A, sA, group_a, B, sB, group_b, batch, M, N, K, strideA, strideB,
                          strideC, C, acc_out, workspace, workspace_bytes, stream);
}

size_t sq_quantize_grouped_i8_workspace_bytes(int64_t rows, int64_t group_rows) {
    if (rows <= 0 || group_rows <= 0) return 0;
    const size_t ng = static_cast<size_t>((rows + group_rows - 1) / group_rows);
    return (ng * 4 + 255) & ~static_cast<size_t>(255);
}

sq_status sq_quantize_grouped_i8(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                                 int64_t group_rows, int8_t* q, float* scales, void* workspace,
                                 size_t workspace_bytes, sq_stream stream) {
    if (dtype != SQ_F32 && dtype != SQ_BF16) return SQ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ld < cols || group_rows < 1) return SQ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return SQ_OK;
    if (!x || !q || !scales) return SQ_ERR_INVALID_ARG;
    if (group_rows > rows) group_rows = rows;
    if (group_rows > 1 && (!workspace ||
                           workspace_bytes < sq_quantize_grouped_i8_workspace_bytes(rows, group_rows)))
        return SQ_ERR_INVALID_ARG;
    if (group_rows > 1 && (reinterpret_cast<uintptr_t>(workspace) & 3u)) return SQ_ERR_ALIGNMENT;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    const int64_t esz = dtype == SQ_F32 ? 4 : 2;
    const bool vec_ok = aligned16(x) && aligned16(q) && ((ld * esz) % 16 == 0) && (cols % 16 == 0);
    return from_cuda(sq::launch_quantize_grouped_i8(x, dtype, rows, cols, ld, group_rows, q, scales,
                                                    static_cast<unsigned*>(workspace), vec_ok,
                                                    reinterpret_cast<cudaStream_t>(stream),
                                                    ds->sms));
}

namespace {

// The argument checks of one scaled FP8 GEMM.
sq_status check_gemm_fp8(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                         int fmt, int layout, int64_t M, int64_t N, int64_t K, const void* C) {
    if (fmt != SQ_FMT_E4M3 && fmt != SQ_FMT_E5M2) return SQ_ERR_INVALID_ARG;
    if (layout != SQ_NT && layout != SQ_NN && layout != SQ_TN) return SQ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return SQ_ERR_INVALID_ARG;
    if (!A || !B || !sa || !sb || !C) return SQ_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return SQ_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return SQ_ERR_ALIGNMENT;
    // TMA row pitches must be multiples of 16 bytes
    if (layout == SQ_NT && K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (layout == SQ_NN && (K % 16 != 0 || N % 16 != 0)) return SQ_ERR_ALIGNMENT;
    if (layout == SQ_TN && (M % 16 != 0 || N % 16 != 0)) return SQ_ERR_ALIGNMENT;
    if (((M + 127) / 128) * ((N + 127) / 128) > kMaxDim) return SQ_ERR_UNSUPPORTED;
    return SQ_OK;
}

sq_status gemm_fp8_common(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                          int fmt, int layout, int64_t M, int64_t N, int64_t K, void* C,
                          const float* out_scale, sq_stream stream) {
    const sq_status r = check_gemm_fp8(A, B, sa, sb, fmt, layout, M, N, K, C);
    if (r != SQ_OK) return r;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return from_cuda(sq::launch_gemm_fp8(A, B, sa, sb, fmt, layout, static_cast<int>(M),
                                         static_cast<int>(N), static_cast<int>(K), C, out_scale,
                                         nullptr, ds->err_word,
                                         reinterpret_cast<cudaStream_t>(stream), ds->sms));
}

}  // namespace

sq_status sq_gemm_fp8_scaled(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                             int fmt, int layout, int64_t M, int64_t N, int64_t K,
                             uint16_t* C_bf16, sq_stream stream) {
    return gemm_fp8_common(A, B, sa, sb, fmt, layout, M, N, K, C_bf16, nullptr, stream);
}

// Whether the byte ranges [p, p + a) and [q, q + b) meet.
bool overlaps(const void* p, int64_t a, const void* q, int64_t b) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(p), y = reinterpret_cast<uintptr_t>(q);
    return x < y + static_cast<uint64_t>(b) && y < x + static_cast<uint64_t>(a);
}

sq_status sq_gemm_fp8_scaled_pair(const uint8_t* const A[2], const uint8_t* const B[2],
                                  const float* const sa[2], const float* const sb[2], int fmt,
                                  const int layout[2], const int64_t M[2], const int64_t N[2],
                                  const int64_t K[2], uint16_t* const C_bf16[2], sq_stream stream) {
    if (!A || !B || !sa || !sb || !layout || !M || !N || !K || !C_bf16) return SQ_ERR_INVALID_ARG;
    for (int i = 0; i < 2; ++i) {
        const sq_status r = check_gemm_fp8(A[i], B[i], sa[i], sb[i], fmt, layout[i], M[i], N[i], K[i],
                                           C_bf16[i]);
        if (r != SQ_OK) return r;
    }
    // the problems run side by side: an output may meet no operand and not
    // the other output
    for (int i = 0; i < 2; ++i) {
        const int j = 1 - i;
        const int64_t c_bytes = M[i] * N[i] * 2;
        if (overlaps(C_bf16[i], c_bytes, A[j], M[j] * K[j]) ||
            overlaps(C_bf16[i], c_bytes, B[j], N[j] * K[j]) ||
            overlaps(C_bf16[i], c_bytes, C_bf16[j], M[j] * N[j] * 2))
            return SQ_ERR_INVALID_ARG;
    }
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    sq::Fp8Problem q[2];
    for (int i = 0; i < 2; ++i)
        q[i] = sq::Fp8Problem{A[i], B[i], sa[i], sb[i], layout[i], static_cast<int>(M[i]),
                              static_cast<int>(N[i]), static_cast<int>(K[i]), C_bf16[i]};
    return from_cuda(sq::launch_gemm_fp8_pair(q, fmt, ds->err_word,
                                              reinterpret_cast<cudaStream_t>(stream), ds->sms));
}

sq_status sq_gemm_fp8_scaled_e4m3(const uint8_t* A, const uint8_t* B, const float* sa,
                                  const float* sb, int fmt, int layout, int64_t M, int64_t N,
                                  int64_t K, const float* out_scale, uint8_t* C_e4m3,
                                  sq_stream stream) {
    if (!out_scale) return SQ_ERR_INVALID_ARG;
    return gemm_fp8_common(A, B, sa, sb, fmt, layout, M, N, K, C_e4m3, out_scale, stream);
}

// ---------------------------------------------------------------- linear layer
namespace {

// workspace: [0, 256) quantize words (amax bits, ticket) and step slots;
// then the float32 bias (N).
constexpr size_t kLinStepX = 64, kLinStepW = 68, kLinStepG = 72, kLinSinkW = 80, kLinSinkX = 84;

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Quantize one operand: with a ring, the step used (sx, or the ring's slot)
// is first copied to `used`, because the quantize publishes the next step
// into the ring's slot when it finishes.  Returns the step pointer that the
// GEMM must read.
// An operand's step: given (step), or from its delayed-scaling ring.
sq_status check_operand(const float* step, const float* ring, int64_t hist, int64_t idx, int margin) {
    if (!step && !ring) return SQ_ERR_INVALID_ARG;
    if (ring && (hist < 1 || hist > (int64_t(1) << 20) || idx < 0 || idx >= hist || margin < -64 ||
                 margin > 64 || (reinterpret_cast<uintptr_t>(ring) & 3u)))
        return SQ_ERR_INVALID_ARG;
    return SQ_OK;
}

// The operands of one linear call, quantized in one launch.  An operand
// without a given step takes the one its ring holds; the kernel writes that
// step into the operand's slot in the workspace, so the GEMM uses the step
// the quantization used although the ring then publishes the next one.
struct LinQuant {
    int count = 0;
    const uint16_t* x[4];
    int64_t n[4];
    const float* scale[4];
    float* ring[4];
    int hist[4], idx[4], margin[4];
    float* used[4];
    uint8_t* x8[4];
    float* amax[4];

    // the step the GEMM should use for the operand just added
    const float* add(const uint16_t* xp, int64_t np, const float* step, float* rg, int64_t h,
                     int64_t i, int mg, uint8_t* x8p, float* am, float* slot) {
        const int t = count++;
        x[t] = xp;
        n[t] = np;
        scale[t] = step;
        ring[t] = rg;
        hist[t] = static_cast<int>(h);
        idx[t] = static_cast<int>(i);
        margin[t] = mg;
        used[t] = step ? nullptr : slot;
        x8[t] = x8p;
        amax[t] = am;
        return step ? step : slot;
    }

    sq_status launch(int fmt, unsigned* qws, unsigned* err_word, cudaStream_t st, int sms) const {
        return from_cuda(sq::launch_quantize_fp8_rings(count, x, n, scale, ring, hist, idx, margin,
                                                       used, fmt, x8, amax, qws, err_word, st, sms));
    }
};

}  // namespace

size_t sq_linear_workspace_bytes(int64_t T, int64_t N, int64_t K) {
    (void)T;
    (void)K;
    if (N <= 0) return 0;
    return 256 + align256(static_cast<size_t>(N) * 4);
}

sq_status sq_linear_forward_fp8(const uint16_t* x, int64_t M, int64_t K, const void* w,
                                int w_prequantized, int64_t N, const void* bias, int bias_kind,
                                const float* bias_scale, const float* sx, const float* sw, int fmt,
                                float* x_ring, int64_t x_hist, int64_t x_idx, int x_margin,
                                float* w_ring, int64_t w_hist, int64_t w_idx, int w_margin,
                                uint16_t* out, uint8_t* x8, uint8_t* w8, float* amax_x,
                                float* amax_w, void* workspace, size_t workspace_bytes,
                                sq_stream stream) {
    if (fmt != SQ_FMT_E4M3 && fmt != SQ_FMT_E5M2) return SQ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return SQ_ERR_INVALID_ARG;
    if (!x || !w || !out || !x8 || !amax_x || !amax_w || !workspace) return SQ_ERR_INVALID_ARG;
    if (!w_prequantized && !w8) return SQ_ERR_INVALID_ARG;
    if (bias_kind != SQ_BIAS_NONE && bias_kind != SQ_BIAS_BF16 && bias_kind != SQ_BIAS_FP8)
        return SQ_ERR_INVALID_ARG;
    if (bias_kind != SQ_BIAS_NONE && !bias) return SQ_ERR_INVALID_ARG;
    if (bias_kind == SQ_BIAS_FP8 && !bias_scale) return SQ_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return SQ_ERR_UNSUPPORTED;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned16(x8) || !aligned16(w8) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SQ_ERR_ALIGNMENT;
    if (workspace_bytes < sq_linear_workspace_bytes(M, N, K)) return SQ_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    unsigned* qws = reinterpret_cast<unsigned*>(wsb);
    float* bias32 = reinterpret_cast<float*>(wsb + 256);
    sq_status r = check_operand(sx, x_ring, x_hist, x_idx, x_margin);
    if (r != SQ_OK) return r;
    if (w_prequantized) {
        if (!sw) return SQ_ERR_INVALID_ARG;
    } else {
        r = check_operand(sw, w_ring, w_hist, w_idx, w_margin);
        if (r != SQ_OK) return r;
    }
    // x and (unless it comes quantized) w in one launch
    LinQuant lq;
    const float* sx_g = lq.add(x, M * K, sx, x_ring, x_hist, x_idx, x_margin, x8, amax_x,
                               reinterpret_cast<float*>(wsb + kLinStepX));
    const float* sw_g = sw;
    const uint8_t* wq = w8;
    if (w_prequantized) {
        wq = static_cast<const uint8_t*>(w);
        if (cudaMemsetAsync(amax_w, 0, sizeof(float), st) != cudaSuccess) return SQ_ERR_CUDA;
    } else {
        sw_g = lq.add(static_cast<const uint16_t*>(w), N * K, sw, w_ring, w_hist, w_idx, w_margin,
                      w8, amax_w, reinterpret_cast<float*>(wsb + kLinStepW));
    }
    r = lq.launch(fmt, qws, ds->err_word, st, ds->sms);
    if (r != SQ_OK) return r;
    const float* bias_f = nullptr;
    if (bias_kind != SQ_BIAS_NONE) {
        e = sq::launch_bias_to_f32(bias, bias_kind, fmt, bias_scale, N, bias32, st);
        if (e != cudaSuccess) return SQ_ERR_CUDA;
        bias_f = bias32;
    }
    return from_cuda(sq::launch_gemm_fp8(x8, wq, sx_g, sw_g, fmt, SQ_NT, static_cast<int>(M),
                                         static_cast<int>(N), static_cast<int>(K), out, nullptr,
                                         bias_f, ds->err_word, st, ds->sms));
}

sq_status sq_linear_backward_fp8(const uint16_t* g, const uint16_t* x, const uint16_t* w,
                                 int64_t T, int64_t N, int64_t K, int masks, const float* sg,
                                 const float* sw, const float* sx, int fmt, float* g_ring,
                                 int64_t g_hist, int64_t g_idx, int g_margin, uint16_t* gx,
                                 uint16_t* gw, uint16_t* gb, float* amax_g, uint8_t* g8,
                                 uint8_t* w8, uint8_t* x8, void* workspace, size_t workspace_bytes,
                                 sq_stream stream) {
    const bool want_gx = masks & SQ_GRAD_INPUT, want_gw = masks & SQ_GRAD_WEIGHT,
               want_gb = masks & SQ_GRAD_BIAS;
    if (fmt != SQ_FMT_E4M3 && fmt != SQ_FMT_E5M2) return SQ_ERR_INVALID_ARG;
    if (T < 1 || N < 1 || K < 1 || (masks & ~7)) return SQ_ERR_INVALID_ARG;
    if (!g || !amax_g || !g8 || !workspace) return SQ_ERR_INVALID_ARG;
    if (want_gx && (!w || !sw || !w8 || !gx)) return SQ_ERR_INVALID_ARG;
    if (want_gw && (!x || !sx || !x8 || !gw)) return SQ_ERR_INVALID_ARG;
    if (want_gb && !gb) return SQ_ERR_INVALID_ARG;
    if (T > kMaxDim || N > kMaxDim || K > kMaxDim) return SQ_ERR_UNSUPPORTED;
    if (N % 16 != 0 || K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (!aligned16(g) || !aligned16(x) || !aligned16(w) || !aligned16(gx) || !aligned16(gw) ||
        !aligned16(g8) || !aligned16(w8) || !aligned16(x8) ||
        (reinterpret_cast<uintptr_t>(gb) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SQ_ERR_ALIGNMENT;
    if (workspace_bytes < sq_linear_workspace_bytes(T, N, K)) return SQ_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    unsigned* qws = reinterpret_cast<unsigned*>(wsb);
    sq_status r = check_operand(sg, g_ring, g_hist, g_idx, g_margin);
    if (r != SQ_OK) return r;
    // one quantization of the gradient, shared by both products, and the
    // operands the asked-for products need, in one launch
    LinQuant lq;
    const float* sg_g = lq.add(g, T * N, sg, g_ring, g_hist, g_idx, g_margin, g8, amax_g,
                               reinterpret_cast<float*>(wsb + kLinStepG));
    if (want_gx)
        lq.add(w, N * K, sw, nullptr, 0, 0, 0, w8, reinterpret_cast<float*>(wsb + kLinSinkW), nullptr);
    if (want_gw)
        lq.add(x, T * K, sx, nullptr, 0, 0, 0, x8, reinterpret_cast<float*>(wsb + kLinSinkX), nullptr);
    r = lq.launch(fmt, qws, ds->err_word, st, ds->sms);
    if (r != SQ_OK) return r;
    if (want_gx && want_gw) {
        // dX[T,K] = G[T,N] W[N,K] (NN) and dW[N,K] = G^T[N,T] X[T,K] (TN, G
        // stored [T,N]): independent products, dealt together
        const sq::Fp8Problem q[2] = {
            {g8, w8, sg_g, sw, SQ_NN, static_cast<int>(T), static_cast<int>(K), static_cast<int>(N), gx},
            {g8, x8, sg_g, sx, SQ_TN, static_cast<int>(N), static_cast<int>(K), static_cast<int>(T), gw}};
        e = sq::launch_gemm_fp8_pair(q, fmt, ds->err_word, st, ds->sms);
        if (e != cudaSuccess) return SQ_ERR_CUDA;
    } else if (want_gx) {
        // dX[T,K] = G[T,N] W[N,K]  (NN)
        e = sq::launch_gemm_fp8(g8, w8, sg_g, sw, fmt, SQ_NN, static_cast<int>(T),
                                static_cast<int>(K), static_cast<int>(N), gx, nullptr, nullptr,
                                ds->err_word, st, ds->sms);
        if (e != cudaSuccess) return SQ_ERR_CUDA;
    } else if (want_gw) {
        // dW[N,K] = G^T[N,T] X[T,K]  (TN, G stored [T,N])
        e = sq::launch_gemm_fp8(g8, x8, sg_g, sx, fmt, SQ_TN, static_cast<int>(N),
                                static_cast<int>(K), static_cast<int>(T), gw, nullptr, nullptr,
                                ds->err_word, st, ds->sms);
        if (e != cudaSuccess) return SQ_ERR_CUDA;
    }
    if (want_gb) {
        e = sq::launch_colsum_bf16(g, T, N, gb, st);
        if (e != cudaSuccess) return SQ_ERR_CUDA;
    }
    return SQ_OK;
}

namespace {

// Device address of g_sq_noalloc_scratch for the current device, looked up
// once per device (with that device current) on the first no-alloc call.
struct NoAllocState {
    std::once_flag once;
    void* scratch = nullptr;
    cudaError_t err = cudaSuccess;
};
NoAllocState g_noalloc[kMaxDevices];

}  // namespace

sq_status sq_gemm_i8_rowscaled_noalloc(const int8_t* A, const float* sA, const int8_t* B,
                                       const float* sB, int64_t batch, int64_t M, int64_t N,
                                       int64_t K, int64_t strideA, int64_t strideB,
                                       int64_t strideC, float* C, int32_t* acc_out,
                                       sq_stream stream) {
    if (batch < 1 || M < 1 || N < 1 || K < 1) return SQ_ERR_INVALID_ARG;
    if (!A || !B || !sA || !sB || (!C && !acc_out)) return SQ_ERR_INVALID_ARG;
    if (strideA < M * K || strideB < N * K || strideC < M * N) return SQ_ERR_INVALID_ARG;
    if (K % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (K > (int64_t(1) << 17)) return SQ_ERR_UNSUPPORTED;
    if (batch > 65535 || M > kMaxDim || N > kMaxDim) return SQ_ERR_UNSUPPORTED;
    // the staged copies must fit the fixed scratch array (checked before any
    // product that could overflow: each factor is below 2^31 here)
    if (static_cast<double>(batch) * (static_cast<double>(M) + static_cast<double>(N)) *
            static_cast<double>(K) * 2.0 > static_cast<double>(SQ_GEMM_I8_NOALLOC_SCRATCH_BYTES))
        return SQ_ERR_UNSUPPORTED;
    const size_t need = sq_gemm_i8_workspace_bytes(batch, M, N, K);
    if (need > SQ_GEMM_I8_NOALLOC_SCRATCH_BYTES) return SQ_ERR_UNSUPPORTED;
    if (strideA % 16 != 0 || strideB % 16 != 0) return SQ_ERR_ALIGNMENT;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(acc_out))
        return SQ_ERR_ALIGNMENT;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return SQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SQ_ERR_UNSUPPORTED;
    NoAllocState& na = g_noalloc[dev];
    std::call_once(na.once, [&] {
        na.err = cudaGetSymbolAddress(&na.scratch, g_sq_noalloc_scratch);
    });
    if (na.err != cudaSuccess || !na.scratch) return SQ_ERR_CUDA;
    // the rest is the workspace entry point with the scratch array as workspace
    return sq_gemm_i8_rowscaled(A, sA, B, sB, batch, M, N, K, strideA, strideB, strideC, C,
                                acc_out, na.scratch, SQ_GEMM_I8_NOALLOC_SCRATCH_BYTES, stream);
}

sq_status sq_set_clock_probe(unsigned long long* fp8_records, unsigned long long* i8_records,
                             int max_ctas) {
    if (max_ctas < 0 || ((fp8_records || i8_records) && max_ctas == 0)) return SQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(fp8_records) | reinterpret_cast<uintptr_t>(i8_records)) & 7u)
        return SQ_ERR_ALIGNMENT;
    return from_cuda(sq::set_gemm_clock_probe(fp8_records, i8_records, max_ctas));
}

sq_status sq_selftest_bounded_wait(uint64_t limit_ns, sq_stream stream) {
    if (limit_ns == 0 || limit_ns > 2000000000ull) return SQ_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    DeviceState* ds = device_state(&e);
    if (!ds) return from_cuda(e);
    return from_cuda(sq::launch_selftest_wait(ds->err_word, limit_ns,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

sq_status sq_get_last_device_error(sq_stream stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return SQ_ERR_CUDA;
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_sq_device_error, sizeof(word));
    if (e != cudaSuccess) return SQ_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_sq_device_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return SQ_ERR_CUDA;
        return SQ_ERR_DEVICE_TIMEOUT;
    }
    return SQ_OK;
}

}  // extern "C"
