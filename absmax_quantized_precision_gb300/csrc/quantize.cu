// Quantize kernels (HBM-bound): per-row symmetric INT8 and per-tensor FP8
// with the amax fused in.
//
// INT8 (POPCORNBENCH "Kimi-K2.6 l2_p13" trace, reference-model analysis and
// rounding discussion; per-row / per-head granularity of the scmp_kernels
// README): s = max(amax_row, 1e-8) / 127, q = clamp(rne(x / s), -127, 127),
// with the quotient rounded exactly as IEEE float32 division rounds it (via
// __fdiv_rn, or the FMA-corrected reciprocal product below where that is
// provably the same float) and round-half-even (__float2int_rn), never a
// plain reciprocal multiply or roundf.
//
// FP8 (AstrAI ops/fp8.py, custom::fp8_quantize and the commit notes): x8 =
// fp8(x / scale), the quotient rounded as IEEE division rounds it, then
// round-to-nearest-even and saturation to the largest
// finite value (cvt.rn.satfinite), amax = max|x| folded in by the last block
// to finish (threadfence + ticket counter), so no second launch and no
// per-call memset: the last block also resets the two workspace words.
#include <cuda_bf16.h>

#include <cstdint>
#include <cstring>

#include "sq_device.cuh"
#include "sq_host.h"
#include "sq_launch.h"

namespace sq {

// ================================================================== INT8 rows
template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    __device__ static float load1(const float* p) { return *p; }
};
template <>
struct Elem<uint16_t> {   // bf16 bit patterns; widening is exact
    static constexpr int kPerVec = 8;
    __device__ static float load1(const uint16_t* p) {
        return __uint_as_float(static_cast<uint32_t>(*p) << 16);
    }
};

// The INT8 quotient only matters where |x/s| >= 1/2; with s in [2^-34, 2^40]
// (s >= 1e-8/127 > 2^-34 always) those quotients and their residuals stay in
// the normal range, and |x/s| <= 128 rules out overflow.
constexpr float kRecipHi = 0x1p40f;

__device__ __forceinline__ int8_t clamp_i8(int n) {
    n = n > 127 ? 127 : (n < -127 ? -127 : n);
    return static_cast<int8_t>(n);
}

__device__ __forceinline__ int8_t encode_i8(float x, float s) {
    return clamp_i8(__float2int_rn(__fdiv_rn(x, s)));
}

__device__ __forceinline__ float row_scale(float amax) {
    return __fdiv_rn(fmaxf(amax, 1e-8f), 127.0f);
}

// ---- one 16-byte input vector at a time (8 bf16 or 4 f32 values)
// |x| max folded into a running maximum.  bf16 values are compared as bf16
// (sign bits cleared, then a packed max): comparisons are exact, so widening
// the result afterwards gives the f32 maximum.  NaN lanes lose to numbers, as
// with fmaxf.
template <typename T>
struct AbsMax;
template <>
struct AbsMax<float> {
    float m = 0.0f;
    __device__ __forceinline__ void add(const uint4& v) {
        m = fmaxf(fmaxf(m, fabsf(__uint_as_float(v.x))), fabsf(__uint_as_float(v.y)));
        m = fmaxf(fmaxf(m, fabsf(__uint_as_float(v.z))), fabsf(__uint_as_float(v.w)));
    }
    __device__ __forceinline__ float value() const { return m; }
};
template <>
struct AbsMax<uint16_t> {
    uint32_t m = 0u;   // two bf16 lanes
    __device__ __forceinline__ static uint32_t max2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ __forceinline__ void add(const uint4& v) {
        const uint32_t a = max2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
        const uint32_t b = max2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
        m = max2(m, max2(a, b));
    }
    __device__ __forceinline__ float value() const {
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
    }
};

// Code of x for a scale in the reciprocal range, as the low byte of a word.
// RNE(t) for |t| < 2^22 is what adding 1.5 * 2^23 leaves in the low bits (the
// sum's ulp is 1 and RN breaks ties to even), and its low byte is the
// two's-complement code.  No clamp is needed: s = RN(m/127) with every
// |x| <= m bounds |x/s| by 127 / (1 - 2^-24) < 127.5, so RNE already lands in
// [-127, 127].
__device__ __forceinline__ uint32_t code_word(float x, float s, float y) {
    return __float_as_uint(__fadd_rn(div_rn_recip(x, s, y), 12582912.0f));
}
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Codes of one 16-byte input vector: pack() returns them as packed bytes
// (4 for float, 8 for bf16), store() writes them at dst (aligned to their
// size), and stage() also writes them as exact fp16 values at dst16 and adds
// their squares to sq.  FAST: s <= kRecipHi.
template <typename T>
struct Codes;
template <>
struct Codes<float> {
    template <bool FAST>
    __device__ __forceinline__ static uint32_t pack(const uint4& v, float s, float y) {
        const float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                            __uint_as_float(v.w)};
        if (FAST)
            return pack_low_bytes(code_word(f[0], s, y), code_word(f[1], s, y), code_word(f[2], s, y),
                                  code_word(f[3], s, y));
        return pack_low_bytes(static_cast<uint8_t>(encode_i8(f[0], s)),
                              static_cast<uint8_t>(encode_i8(f[1], s)),
                              static_cast<uint8_t>(encode_i8(f[2], s)),
                              static_cast<uint8_t>(encode_i8(f[3], s)));
    }
    template <bool FAST>
    __device__ __forceinline__ static void store(const uint4& v, float s, float y, int8_t* dst) {
        *reinterpret_cast<uint32_t*>(dst) = pack<FAST>(v, s, y);
    }
    template <bool FAST>
    __device__ __forceinline__ static void stage(const uint4& v, float s, float y, int8_t* dst,
                                                 uint16_t* dst16, int& sq) {
        const uint32_t w = pack<FAST>(v, s, y);
        *reinterpret_cast<uint32_t*>(dst) = w;
        *reinterpret_cast<uint2*>(dst16) = i8x4_to_f16x4(w);
        sq = __dp4a(static_cast<int>(w), static_cast<int>(w), sq);
    }
};
template <>
struct Codes<uint16_t> {
    template <bool FAST>
    __device__ __forceinline__ static void store(const uint4& v, float s, float y, int8_t* dst) {
        *reinterpret_cast<uint2*>(dst) = pack<FAST>(v, s, y);
    }
    template <bool FAST>
    __device__ __forceinline__ static void stage(const uint4& v, float s, float y, int8_t* dst,
                                                 uint16_t* dst16, int& sq) {
        const uint2 w = pack<FAST>(v, s, y);
        *reinterpret_cast<uint2*>(dst) = w;
        *reinterpret_cast<uint4*>(dst16) = i8x8_to_f16x8(w);
        sq = __dp4a(static_cast<int>(w.x), static_cast<int>(w.x), sq);
        sq = __dp4a(static_cast<int>(w.y), static_cast<int>(w.y), sq);
    }
    template <bool FAST>
    __device__ __forceinline__ static uint2 pack(const uint4& v, float s, float y) {
        const uint32_t src[4] = {v.x, v.y, v.z, v.w};
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(src[i] << 16);
            const float hi = __uint_as_float(src[i] & 0xFFFF0000u);
            if (FAST) {
                c[2 * i] = code_word(lo, s, y);
                c[2 * i + 1] = code_word(hi, s, y);
            } else {
                c[2 * i] = static_cast<uint8_t>(encode_i8(lo, s));
                c[2 * i + 1] = static_cast<uint8_t>(encode_i8(hi, s));
            }
        }
        return make_uint2(pack_low_bytes(c[0], c[1], c[2], c[3]), pack_low_bytes(c[4], c[5], c[6], c[7]));
    }
};

// A group of TPR threads owns one row, held in registers (VPT 16-byte vectors
// per thread).  Rows must start 16-byte aligned and cols be a multiple of 16.
// STAGE: the codes are also written as exact fp16 values at q16 (rows
// packed) for the INT8 GEMM, and the operand's bound region is marked as
// holding no bound.
// A second operand with the same row length may follow in the same launch
// (rows2 > 0): its rows come after the first operand's in the deal.
template <typename T>
struct RowOperand {
    const T* x;
    int64_t rows, ld;
    int8_t* q;
    float* scales;
    uint16_t* q16;
    unsigned* bound;
};

template <typename T, int TPR, int VPT, bool STAGE>
__global__ void __launch_bounds__(256) quant_row_i8_vec(const RowOperand<T> o1, const RowOperand<T> o2,
                                                        int64_t cols) {
    pdl_begin();
    if (STAGE && blockIdx.x == 0 && threadIdx.x == 0) {
        *o1.bound = 0u;
        if (o2.rows > 0) *o2.bound = 0u;
    }
    const int64_t rows = o1.rows + o2.rows;
    constexpr int EPV = Elem<T>::kPerVec;
    constexpr int RPB = 256 / TPR;
    __shared__ float red[8];
    const int g = threadIdx.x / TPR;
    const int lg = threadIdx.x % TPR;
    const int64_t nvec = cols / EPV;
    for (int64_t row0 = static_cast<int64_t>(blockIdx.x) * RPB; row0 < rows;
         row0 += static_cast<int64_t>(gridDim.x) * RPB) {
        const int64_t rowd = row0 + g;   // in the deal: the first operand's rows, then the second's
        const bool live = rowd < rows;
        const bool second = rowd >= o1.rows;
        const int64_t row = second ? rowd - o1.rows : rowd;
        const T* x = second ? o2.x : o1.x;
        const int64_t ld = second ? o2.ld : o1.ld;
        int8_t* q = second ? o2.q : o1.q;
        float* scales = second ? o2.scales : o1.scales;
        uint16_t* q16 = second ? o2.q16 : o1.q16;
        uint4 raw[VPT];                 // the row stays packed: 4 registers per 16 bytes
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t vi = lg + static_cast<int64_t>(i) * TPR;
            raw[i] = (live && vi < nvec) ? ld_stream_v4(x + row * ld + vi * EPV) : make_uint4(0, 0, 0, 0);
        }
        AbsMax<T> am;
#pragma unroll
        for (int i = 0; i < VPT; ++i) am.add(raw[i]);
        float m = am.value();
        if (TPR <= 32) {
#pragma unroll
            for (int o = TPR / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        } else {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            __syncthreads();   // previous row's readers of red[] are done
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
            __syncthreads();
            m = red[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
        }
        const float s = row_scale(m);
        const bool fast = s <= kRecipHi;   // s >= kRecipLo always
        const float y = __frcp_rn(s);
        if (live) {
            if (lg == 0) scales[row] = s;
            int sq = 0;   // unused: this path records no bound
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int64_t vi = lg + static_cast<int64_t>(i) * TPR;
                if (vi >= nvec) continue;
                const int64_t o = row * cols + vi * EPV;
                if (STAGE) {
                    if (fast) Codes<T>::template stage<true>(raw[i], s, y, q + o, q16 + o, sq);
                    else Codes<T>::template stage<false>(raw[i], s, y, q + o, q16 + o, sq);
                } else {
                    if (fast) Codes<T>::template store<true>(raw[i], s, y, q + o);
                    else Codes<T>::template store<false>(raw[i], s, y, q + o);
                }
            }
        }
    }
}

// Any alignment, any row length: one CTA per row, two passes over the row
// (the second pass is served from L2).
template <typename T>
__global__ void __launch_bounds__(256) quant_row_i8_scalar(const T* __restrict__ x, int64_t rows,
                                                           int64_t cols, int64_t ld,
                                                           int8_t* __restrict__ q,
                                                           float* __restrict__ scales) {
    pdl_begin();
    __shared__ float red[8];
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const T* xr = x + row * ld;
        float m = 0.0f;
        for (int64_t k = threadIdx.x; k < cols; k += blockDim.x)
            m = fmaxf(m, fabsf(Elem<T>::load1(xr + k)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        __syncthreads();
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        m = red[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
        const float s = row_scale(m);
        if (threadIdx.x == 0) scales[row] = s;
        for (int64_t k = threadIdx.x; k < cols; k += blockDim.x)
            q[row * cols + k] = encode_i8(Elem<T>::load1(xr + k), s);
    }
}

// Rows of 2-16 KB with enough rows to fill the GPU: persistent CTAs of 256
// threads walk rows blockIdx.x, +gridDim.x, ...; the next row is fetched into
// the other half of a 2 x 16 KB shared-memory buffer with cp.async while the
// current one is quantized, so every CTA always has a row in flight.  The
// row is read from shared memory twice (absmax, then codes); codes go to
// global memory directly.  Needs 16-byte aligned rows and cols % 16 == 0.
constexpr int kPfRowBytes = 16384;

template <typename T>
__global__ void __launch_bounds__(256) quant_row_i8_pf(const T* __restrict__ x, int64_t rows,
                                                       int64_t cols, int64_t ld,
                                                       int8_t* __restrict__ q,
                                                       float* __restrict__ scales) {
    pdl_begin();
    constexpr int EPV = Elem<T>::kPerVec;
    __shared__ __align__(16) uint8_t buf[2][kPfRowBytes];
    __shared__ float red[8];
    const int nvec = static_cast<int>(cols / EPV);          // 16-byte vectors per row
    const int64_t G = gridDim.x;
    const int t = threadIdx.x;
    auto fetch = [&](int64_t row, int b) {
        const T* src = x + row * ld;
        for (int vi = t; vi < nvec; vi += 256) cp_async16(&buf[b][vi * 16], src + vi * EPV);
        cp_async_commit();
    };
    int64_t row = blockIdx.x;
    if (row < rows) fetch(row, 0);
    for (int i = 0; row < rows; ++i, row += G) {
        const int b = i & 1;
        if (row + G < rows) fetch(row + G, b ^ 1);
        else cp_async_commit();                 // keep one group per iteration
        cp_async_wait<1>();                     // this row's copies are done
        __syncthreads();
        AbsMax<T> am;
        for (int vi = t; vi < nvec; vi += 256) am.add(*reinterpret_cast<const uint4*>(&buf[b][vi * 16]));
        float m = am.value();
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((t & 31) == 0) red[t >> 5] = m;
        __syncthreads();
        m = red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
        const float s = row_scale(m);
        const bool fast = s <= kRecipHi;
        const float y = __frcp_rn(s);
        if (t == 0) scales[row] = s;
        int8_t* qr = q + row * cols;
        if (fast) {
            for (int vi = t; vi < nvec; vi += 256)
                Codes<T>::template store<true>(*reinterpret_cast<const uint4*>(&buf[b][vi * 16]), s, y,
                                  qr + vi * EPV);
        } else {
            for (int vi = t; vi < nvec; vi += 256)
                Codes<T>::template store<false>(*reinterpret_cast<const uint4*>(&buf[b][vi * 16]), s, y,
                                   qr + vi * EPV);
        }
        __syncthreads();                        // buffer b and red[] are free again
    }
    cp_async_wait<0>();
}

// quant_row_i8_pf that also stages the codes for the INT8 GEMM: every code
// is written a second time as an exact fp16 value (q16, rows packed), and
// each CTA records in the operand's bound region the largest row norm (sum
// of squared codes) over its rows; block 0 writes the region's header.
template <typename T>
__global__ void __launch_bounds__(256) quant_row_i8_stage_pf(const T* __restrict__ x, int64_t rows,
                                                             int64_t cols, int64_t ld,
                                                             int8_t* __restrict__ q,
                                                             float* __restrict__ scales,
                                                             uint16_t* __restrict__ q16,
                                                             unsigned* __restrict__ bound) {
    pdl_begin();
    constexpr int EPV = Elem<T>::kPerVec;
    __shared__ __align__(16) uint8_t buf[2][kPfRowBytes];
    __shared__ float red[8];
    __shared__ int red_sq[8];
    const int nvec = static_cast<int>(cols / EPV);          // 16-byte vectors per row
    const int64_t G = gridDim.x;
    const int t = threadIdx.x;
    unsigned row_max = 0u;                                   // thread 0: largest row norm
    auto fetch = [&](int64_t row, int b) {
        const T* src = x + row * ld;
        for (int vi = t; vi < nvec; vi += 256) cp_async16(&buf[b][vi * 16], src + vi * EPV);
        cp_async_commit();
    };
    int64_t row = blockIdx.x;
    if (row < rows) fetch(row, 0);
    for (int i = 0; row < rows; ++i, row += G) {
        const int b = i & 1;
        if (row + G < rows) fetch(row + G, b ^ 1);
        else cp_async_commit();                 // keep one group per iteration
        cp_async_wait<1>();                     // this row's copies are done
        __syncthreads();
        AbsMax<T> am;
        for (int vi = t; vi < nvec; vi += 256) am.add(*reinterpret_cast<const uint4*>(&buf[b][vi * 16]));
        float m = am.value();
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((t & 31) == 0) red[t >> 5] = m;
        __syncthreads();
        m = red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
        const float s = row_scale(m);
        const bool fast = s <= kRecipHi;
        const float y = __frcp_rn(s);
        if (t == 0) scales[row] = s;
        int8_t* qr = q + row * cols;
        uint16_t* q16r = q16 + row * cols;
        int sq = 0;                             // <= 127^2 * cols < 2^31 (cols <= 8192)
        if (fast) {
            for (int vi = t; vi < nvec; vi += 256)
                Codes<T>::template stage<true>(*reinterpret_cast<const uint4*>(&buf[b][vi * 16]), s, y,
                                               qr + vi * EPV, q16r + vi * EPV, sq);
        } else {
            for (int vi = t; vi < nvec; vi += 256)
                Codes<T>::template stage<false>(*reinterpret_cast<const uint4*>(&buf[b][vi * 16]), s, y,
                                                qr + vi * EPV, q16r + vi * EPV, sq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if ((t & 31) == 0) red_sq[t >> 5] = sq;
        __syncthreads();                        // buffer b, red[] and red_sq[] are complete
        if (t == 0) {
            // red_sq is next written after two more barriers of the next row
            int rs = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) rs += red_sq[w];
            row_max = max(row_max, static_cast<unsigned>(rs));
        }
    }
    cp_async_wait<0>();
    if (t == 0) {
        bound[1 + blockIdx.x] = row_max;
        if (blockIdx.x == 0) bound[0] = static_cast<unsigned>(gridDim.x) | kBoundRowNorms;
    }
}

template <typename T, int TPR, int VPT, bool STAGE>
static cudaError_t launch_row_vec(const RowOperand<T>& o1, const RowOperand<T>& o2, int64_t cols,
                                  cudaStream_t st, int sms) {
    constexpr int RPB = 256 / TPR;
    int64_t blocks = (o1.rows + o2.rows + RPB - 1) / RPB;
    const int64_t cap = static_cast<int64_t>(sms) * 64;
    if (blocks > cap) blocks = cap;
    return launch_pdl(quant_row_i8_vec<T, TPR, VPT, STAGE>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                      0, st, 1u, o1, o2, cols);
}

// The register-resident shapes by row length (nvec 16-byte vectors per row),
// for one operand or two with the same row length (o2.rows > 0); false if
// the row is too long for them.
template <typename T, bool STAGE>
static bool launch_row_vec_any(const RowOperand<T>& o1, const RowOperand<T>& o2, int64_t cols,
                               cudaStream_t st, int sms, cudaError_t* e) {
    const int64_t nvec = cols / Elem<T>::kPerVec;
    if (nvec <= 16) *e = launch_row_vec<T, 16, 1, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 32) *e = launch_row_vec<T, 32, 1, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 64) *e = launch_row_vec<T, 32, 2, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 128) *e = launch_row_vec<T, 32, 4, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 256) *e = launch_row_vec<T, 32, 8, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 512) *e = launch_row_vec<T, 256, 2, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 1024) *e = launch_row_vec<T, 256, 4, STAGE>(o1, o2, cols, st, sms);
    else if (nvec <= 2048) *e = launch_row_vec<T, 256, 8, STAGE>(o1, o2, cols, st, sms);
    else return false;
    return true;
}

template <typename T>
static bool launch_row_vec_one(const T* x, int64_t rows, int64_t cols, int64_t ld, int8_t* q,
                               float* scales, uint16_t* q16, unsigned* bound, bool stage,
                               cudaStream_t st, int sms, cudaError_t* e) {
    const RowOperand<T> o1{x, rows, ld, q, scales, q16, bound};
    const RowOperand<T> none{nullptr, 0, 0, nullptr, nullptr, nullptr, nullptr};
    return stage ? launch_row_vec_any<T, true>(o1, none, cols, st, sms, e)
                 : launch_row_vec_any<T, false>(o1, none, cols, st, sms, e);
}

template <typename T>
static cudaError_t launch_row(const T* x, int64_t rows, int64_t cols, int64_t ld, int8_t* q,
                              float* scales, bool vec_ok, unsigned* err_word, cudaStream_t st,
                              int sms) {
    (void)err_word;
    const int64_t row_bytes = cols * static_cast<int64_t>(sizeof(T));
    if (vec_ok && row_bytes >= 2048 && row_bytes <= kPfRowBytes && rows >= 2 * sms) {
        int64_t blocks = rows;
        const int64_t cap = static_cast<int64_t>(sms) * 6;
        if (blocks > cap) blocks = cap;
        return launch_pdl(quant_row_i8_pf<T>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1u, x,
                          rows, cols, ld, q, scales);
    }
    if (vec_ok) {
        cudaError_t e = cudaSuccess;
        if (launch_row_vec_one<T>(x, rows, cols, ld, q, scales, nullptr, nullptr, false, st, sms, &e))
            return e;
    }
    int64_t blocks = rows;
    const int64_t cap = static_cast<int64_t>(sms) * 64;
    if (blocks > cap) blocks = cap;
    return launch_pdl(quant_row_i8_scalar<T>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1u, x,
                      rows, cols, ld, q, scales);
}

cudaError_t launch_quantize_rowwise_i8(const void* x, int dtype, int64_t rows, int64_t cols,
                                       int64_t ld, int8_t* q, float* scales, bool vec_ok,
                                       unsigned* err_word, cudaStream_t st, int sms) {
    if (dtype == 0)
        return launch_row<float>(static_cast<const float*>(x), rows, cols, ld, q, scales, vec_ok,
                                 err_word, st, sms);
    return launch_row<uint16_t>(static_cast<const uint16_t*>(x), rows, cols, ld, q, scales, vec_ok,
                                err_word, st, sms);
}

// Inputs of both operands up to this size are quantized by one launch.
constexpr int64_t kPairFusedMaxBytes = int64_t(16) << 20;

// Whether the quantize-and-stage of `rows` rows takes the row pipeline.
static bool stage_takes_pipeline(int dtype, int64_t rows, int64_t cols, bool vec_ok, int sms) {
    const int64_t row_bytes = cols * (dtype == 0 ? 4 : 2);
    return vec_ok && row_bytes >= 2048 && row_bytes <= kPfRowBytes && rows >= 2 * sms;
}

cudaError_t launch_quantize_rowwise_i8_staged(const void* x, int dtype, int64_t rows,
                                              int64_t cols, int64_t ld, int8_t* q,
                                              float* scales, bool vec_ok, uint16_t* q16,
                                              unsigned* bound, unsigned* err_word,
                                              cudaStream_t st, int sms) {
    if (stage_takes_pipeline(dtype, rows, cols, vec_ok, sms)) {
        int64_t blocks = rows;
        int64_t cap = static_cast<int64_t>(sms) * 6;
        if (cap > kBoundSlots - 1) cap = kBoundSlots - 1;
        if (blocks > cap) blocks = cap;
        if (dtype == 0)
            return launch_pdl(quant_row_i8_stage_pf<float>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                              0, st, 1u, static_cast<const float*>(x), rows, cols, ld, q, scales, q16,
                              bound);
        return launch_pdl(quant_row_i8_stage_pf<uint16_t>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                          0, st, 1u, static_cast<const uint16_t*>(x), rows, cols, ld, q, scales, q16,
                          bound);
    }
    cudaError_t e = cudaSuccess;
    if (vec_ok) {
        const bool done = dtype == 0
            ? launch_row_vec_one<float>(static_cast<const float*>(x), rows, cols, ld, q, scales, q16,
                                        bound, true, st, sms, &e)
            : launch_row_vec_one<uint16_t>(static_cast<const uint16_t*>(x), rows, cols, ld, q, scales,
                                           q16, bound, true, st, sms, &e);
        if (done) return e;
    }
    // other shapes: the plain quantize, then the staging of its codes
    e = launch_quantize_rowwise_i8(x, dtype, rows, cols, ld, q, scales, vec_ok, err_word, st, sms);
    if (e != cudaSuccess) return e;
    return launch_i8_to_f16_one(q, 1, rows, cols, rows * cols, q16, bound, err_word, st, sms);
}

cudaError_t launch_quantize_rowwise_i8_staged_pair(const void* xa, int64_t rows_a, int64_t lda,
                                                   int8_t* qa, float* sa, bool vec_ok_a,
                                                   uint16_t* a16, unsigned* bound_a, const void* xb,
                                                   int64_t rows_b, int64_t ldb, int8_t* qb, float* sb,
                                                   bool vec_ok_b, uint16_t* b16, unsigned* bound_b,
                                                   int dtype, int64_t cols, unsigned* err_word,
                                                   cudaStream_t st, int sms) {
    // Both operands' rows in one launch of the register-resident kernel when
    // each would take it alone, or when their inputs are small (the row
    // pipeline pays off on large operands; on small ones a launch saved is
    // worth more); otherwise one launch (or two) per operand.
    const int64_t in_bytes = (rows_a + rows_b) * cols * (dtype == 0 ? 4 : 2);
    if (vec_ok_a && vec_ok_b &&
        ((!stage_takes_pipeline(dtype, rows_a, cols, true, sms) &&
          !stage_takes_pipeline(dtype, rows_b, cols, true, sms)) ||
         in_bytes <= kPairFusedMaxBytes)) {
        cudaError_t e = cudaSuccess;
        bool done;
        if (dtype == 0) {
            const RowOperand<float> oa{static_cast<const float*>(xa), rows_a, lda, qa, sa, a16, bound_a};
            const RowOperand<float> ob{static_cast<const float*>(xb), rows_b, ldb, qb, sb, b16, bound_b};
            done = launch_row_vec_any<float, true>(oa, ob, cols, st, sms, &e);
        } else {
            const RowOperand<uint16_t> oa{static_cast<const uint16_t*>(xa), rows_a, lda, qa, sa, a16, bound_a};
            const RowOperand<uint16_t> ob{static_cast<const uint16_t*>(xb), rows_b, ldb, qb, sb, b16, bound_b};
            done = launch_row_vec_any<uint16_t, true>(oa, ob, cols, st, sms, &e);
        }
        if (done) return e;
    }
    const cudaError_t e = launch_quantize_rowwise_i8_staged(xa, dtype, rows_a, cols, lda, qa, sa, vec_ok_a,
                                                            a16, bound_a, err_word, st, sms);
    if (e != cudaSuccess) return e;
    return launch_quantize_rowwise_i8_staged(xb, dtype, rows_b, cols, ldb, qb, sb, vec_ok_b, b16,
                                             bound_b, err_word, st, sms);
}

// ================================================================== INT8 row groups
// Row-group quantization (scmp_kernels README group_a / group_b, per_tensor;
// the POPCORNBENCH trace's per-tensor fake-quant): consecutive groups of
// group_rows rows share s_g = max(amax_g, 1e-8) / 127.  Two passes, since a
// group's scale depends on rows other CTAs read: (1) amax per group into a
// zeroed workspace word (atomicMax on the bits; every warp owns a contiguous
// run of rows and flushes once per group it touches), (2) encode.  Both
// passes give each row to one warp; 16-byte vector access when rows allow it.
template <typename T, bool VEC>
__device__ __forceinline__ float row_absmax_warp(const T* xr, int64_t cols, int lane) {
    constexpr int EPV = Elem<T>::kPerVec;
    float m = 0.0f;
    if (VEC) {
        const int64_t nvec = cols / EPV;
        AbsMax<T> am;
        for (int64_t vi = lane; vi < nvec; vi += 32) am.add(ld_stream_v4(xr + vi * EPV));
        m = am.value();
    } else {
        for (int64_t k = lane; k < cols; k += 32) m = fmaxf(m, fabsf(Elem<T>::load1(xr + k)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(256) group_absmax_kernel(const T* __restrict__ x, int64_t rows,
                                                           int64_t cols, int64_t ld,
                                                           int64_t group_rows,
                                                           unsigned* __restrict__ amax_bits) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t per = (rows + nwarps - 1) / nwarps;
    const int64_t r0 = warp * per;
    const int64_t r1 = r0 + per < rows ? r0 + per : rows;
    int64_t gcur = -1;
    float mcur = 0.0f;
    for (int64_t r = r0; r < r1; ++r) {
        const int64_t g = r / group_rows;
        if (g != gcur) {
            if (gcur >= 0 && lane == 0) atomicMax(&amax_bits[gcur], __float_as_uint(mcur));
            gcur = g;
            mcur = 0.0f;
        }
        mcur = fmaxf(mcur, row_absmax_warp<T, VEC>(x + r * ld, cols, lane));
    }
    if (gcur >= 0 && lane == 0) atomicMax(&amax_bits[gcur], __float_as_uint(mcur));
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(256) group_encode_kernel(const T* __restrict__ x, int64_t rows,
                                                           int64_t cols, int64_t ld,
                                                           int64_t group_rows,
                                                           const unsigned* __restrict__ amax_bits,
                                                           int8_t* __restrict__ q,
                                                           float* __restrict__ scales) {
    pdl_begin();
    constexpr int EPV = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += nwarps) {
        const int64_t g = r / group_rows;
        const float s = row_scale(__uint_as_float(amax_bits[g]));
        const bool fast = s <= kRecipHi;
        const float y = __frcp_rn(s);
        if (lane == 0 && r == g * group_rows) scales[g] = s;
        const T* xr = x + r * ld;
        int8_t* qr = q + r * cols;
        if (VEC) {
            const int64_t nvec = cols / EPV;
            if (fast) {
                for (int64_t vi = lane; vi < nvec; vi += 32)
                    Codes<T>::template store<true>(ld_stream_v4(xr + vi * EPV), s, y, qr + vi * EPV);
            } else {
                for (int64_t vi = lane; vi < nvec; vi += 32)
                    Codes<T>::template store<false>(ld_stream_v4(xr + vi * EPV), s, y, qr + vi * EPV);
            }
        } else {
            for (int64_t k = lane; k < cols; k += 32) qr[k] = encode_i8(Elem<T>::load1(xr + k), s);
        }
    }
}

template <typename T>
static cudaError_t launch_grouped(const T* x, int64_t rows, int64_t cols, int64_t ld,
                                  int64_t group_rows, int8_t* q, float* scales, unsigned* ws,
                                  bool vec_ok, cudaStream_t st, int sms) {
    const int64_t ngroups = (rows + group_rows - 1) / group_rows;
    cudaError_t e = cudaMemsetAsync(ws, 0, static_cast<size_t>(ngroups) * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks));
    const unsigned* cws = ws;
    if (vec_ok) {
        e = launch_pdl(group_absmax_kernel<T, true>, grid, dim3(256), 0, st, 1u, x, rows, cols, ld,
                       group_rows, ws);
        if (e != cudaSuccess) return e;
        return launch_pdl(group_encode_kernel<T, true>, grid, dim3(256), 0, st, 1u, x, rows, cols, ld,
                          group_rows, cws, q, scales);
    }
    e = launch_pdl(group_absmax_kernel<T, false>, grid, dim3(256), 0, st, 1u, x, rows, cols, ld,
                   group_rows, ws);
    if (e != cudaSuccess) return e;
    return launch_pdl(group_encode_kernel<T, false>, grid, dim3(256), 0, st, 1u, x, rows, cols, ld,
                      group_rows, cws, q, scales);
}

cudaError_t launch_quantize_grouped_i8(const void* x, int dtype, int64_t rows, int64_t cols,
                                       int64_t ld, int64_t group_rows, int8_t* q, float* scales,
                                       unsigned* ws, bool vec_ok, cudaStream_t st, int sms) {
    if (group_rows == 1)
        return launch_quantize_rowwise_i8(x, dtype, rows, cols, ld, q, scales, vec_ok, nullptr, st,
                                          sms);
    if (dtype == 0)
        return launch_grouped<float>(static_cast<const float*>(x), rows, cols, ld, group_rows, q,
                                     scales, ws, vec_ok, st, sms);
    return launch_grouped<uint16_t>(static_cast<const uint16_t*>(x), rows, cols, ld, group_rows, q,
                                    scales, ws, vec_ok, st, sms);
}

// ================================================================== FP8 tensor

// 8 bf16 (one 16-B word) -> 8 FP8 codes (one 8-B word); m = running max|x|.
template <int FMT, bool FAST>
__device__ __forceinline__ uint2 fp8_encode8(const uint4& a, float s, float y, float& m) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t o[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float f[4];
        f[0] = __uint_as_float(w[2 * i] << 16);
        f[1] = __uint_as_float(w[2 * i] & 0xFFFF0000u);
        f[2] = __uint_as_float(w[2 * i + 1] << 16);
        f[3] = __uint_as_float(w[2 * i + 1] & 0xFFFF0000u);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) t[e] = FAST ? fp8_quotient(f[e], s, y) : __fdiv_rn(f[e], s);
        o[i] = fp8x2<FMT>(t[0], t[1]) | (fp8x2<FMT>(t[2], t[3]) << 16);
    }
    return make_uint2(o[0], o[1]);
}

// Streaming pipeline, one per warp: persistent CTAs of kFWarps warps, and
// every warp streams its own chunks of kFChunk bf16 (2 KB in, 1 KB of codes
// out) with no CTA-wide barrier inside the loop.  Lane 0 keeps kFStages input
// chunks in flight in the warp's shared-memory ring with bulk copies
// (cp.async.bulk, completion on the warp's own mbarriers, bounded waits) and
// writes each chunk's codes back with a bulk store from one of two output
// buffers; every lane converts 32 elements per chunk (four 16-B pieces, lane-
// contiguous, so no bank conflicts).  Chunks are dealt round-robin over all
// warps of the grid.  The ragged tail (< one chunk) is done by block 0 with
// plain loads and stores.
//
// Plain mode (no ring): the step is *scale; ws = [amax bits of tensor 0 |
// ticket | amax bits of tensors 1-3].
// Ring mode: delayed scaling with ring = [hist (hist_len) | scale | counter]
// (the AstrAI commit notes' scale ring): the step is *scale if given, else
// ring[hist_len], and the last block records the amax in hist[ring_idx],
// takes the max over the window and publishes the next step
// fl32(fl32(max * 2^margin) / fmt_max) in ring[hist_len] (kept as it was
// when the window max is 0) -- no extra launch.  A launch of one tensor with
// a ring takes the ring's counter word as its ticket; several tensors take
// ws word 1, each with its own ring or none.  Every launch leaves its ticket
// and the amax words at zero.
// One CTA of 24 warps per SM, two 2 KB stages per warp: 96 KB of loads in
// flight per SM.  Measured on GB300 against 8-32 warps per SM, 0.5-4 KB
// chunks and 2-6 stages, this was the fastest shape for both operands of
// the large workload.
constexpr int kFWarps = 24;
constexpr int kFChunk = 1024;
constexpr int kFStages = 2;
constexpr int kFWarpBytes = kFStages * kFChunk * 2 + 2 * kFChunk;
constexpr int kFMaxTensors = 4;   // tensors one launch quantizes
constexpr int kQSmem = kFWarps * kFWarpBytes + kFWarps * kFStages * 8 + 128;

// The tensors of one launch (1 to kFMaxTensors, each with its own step and
// amax) and their chunks' place in the sequence the warps are dealt:
// tensor t owns chunks [first[t], first[t + 1]); the unused entries of
// `first` hold INT64_MAX, so that the owner of a chunk is a count of
// comparisons.  A tensor with a delayed-scaling ring (ring[t] non-null)
// takes its step from the ring when scale[t] is null, and the last block
// updates its ring; used[t] (nullable) receives the step the tensor used,
// written by block 0.
struct Fp8Set {
    const uint16_t* x[kFMaxTensors];
    uint8_t* x8[kFMaxTensors];
    const float* scale[kFMaxTensors];
    float* amax[kFMaxTensors];
    int64_t n[kFMaxTensors];
    int64_t first[kFMaxTensors + 1];
    float* ring[kFMaxTensors];
    int hist[kFMaxTensors], ridx[kFMaxTensors], margin[kFMaxTensors];
    float* used[kFMaxTensors];
    int count;
};

// The workspace word that accumulates tensor t's amax bits (word 1 is the
// ticket of plain mode).
__device__ __forceinline__ int amax_word(int t) { return t == 0 ? 0 : t + 1; }

// MULTI = false: one tensor (set.count == 1), every chunk its own.
template <int FMT, bool MULTI>
__global__ void __launch_bounds__(kFWarps * 32) quant_fp8_kernel(const __grid_constant__ Fp8Set set,
                                                                 unsigned* __restrict__ ws,
                                                                 unsigned* counter, unsigned* err_word) {
    extern __shared__ uint8_t qsmem_raw[];
    uint8_t* qsmem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(qsmem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* in_buf = qsmem + warp * kFWarpBytes;              // kFStages x 2 KB
    uint8_t* out_buf = in_buf + kFStages * kFChunk * 2;        // 2 x 1 KB
    const int nwarps = static_cast<int>(blockDim.x >> 5);    // kFWarps, or fewer for small tensors
    uint64_t* full = reinterpret_cast<uint64_t*>(qsmem + nwarps * kFWarpBytes) + warp * kFStages;
    __shared__ float red[kFMaxTensors][kFWarps];
    __shared__ int is_last;
    __shared__ float s_amax[kFMaxTensors];
    __shared__ int abort_flag;
    // running max|x| per tensor
    float m0 = 0.0f, m1 = 0.0f, m2 = 0.0f, m3 = 0.0f;
    static_assert(kFMaxTensors == 4, "one running maximum per tensor below");

    const int64_t nfull = set.first[set.count];
    const int64_t GW = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t count = gw < nfull ? (nfull - gw + GW - 1) / GW : 0;
    // chunk c of the dealt sequence: its tensor, and its first element there
    auto owner = [&](int64_t c) {
        if (!MULTI) return 0;
        return static_cast<int>(c >= set.first[1]) + static_cast<int>(c >= set.first[2]) +
               static_cast<int>(c >= set.first[3]);
    };
    auto src = [&](int64_t c) {
        const int t = owner(c);
        return set.x[t] + (c - set.first[t]) * kFChunk;
    };
    if (threadIdx.x == 0) abort_flag = 0;
    if (lane == 0) {
        for (int k = 0; k < kFStages; ++k) mbar_init(&full[k], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // The barrier set-up above touches no global memory, so it overlaps the
    // previous kernel's tail; global memory is accessed only from here on.
    pdl_begin();
    if (lane == 0) {
        for (int64_t k = 0; k < count && k < kFStages; ++k) {
            mbar_arrive_expect_tx(&full[k], kFChunk * 2);
            bulk_load(in_buf + k * kFChunk * 2, src(gw + k * GW), kFChunk * 2, &full[k]);
        }
    }
    // The steps are read only now, so their memory latency overlaps that of
    // the first chunks (bulk_load's memory clobber keeps the reads below them).
    float sv[kFMaxTensors], yv[kFMaxTensors];
    bool fv[kFMaxTensors];
#pragma unroll
    for (int t = 0; t < kFMaxTensors; ++t) {
        sv[t] = (t == 0 || (MULTI && t < set.count))
                    ? (set.scale[t] ? *set.scale[t] : set.ring[t][set.hist[t]])
                    : 1.0f;
        yv[t] = __frcp_rn(sv[t]);
        fv[t] = sv[t] >= 0x1p-40f && sv[t] <= 0x1p40f;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
#pragma unroll
        for (int t = 0; t < kFMaxTensors; ++t)
            if (t < set.count && set.used[t]) *set.used[t] = sv[t];
    }
    int64_t i = 0;
    for (; i < count; ++i) {
        const int stage = static_cast<int>(i % kFStages);
        const int ob = static_cast<int>(i & 1);
        int ok = 1;
        if (lane == 0) {
            ok = mbar_wait(&full[stage], static_cast<uint32_t>((i / kFStages) & 1), &abort_flag, err_word);
            if (i >= 2) bulk_wait_read<1>();   // the store from out_buf[ob] two chunks ago is read
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();                          // orders lane 0's wait before the other lanes' reads
        if (!ok) break;
        const int64_t c = gw + i * GW;
        const int t = owner(c);
        const float s = t == 0 ? sv[0] : t == 1 ? sv[1] : t == 2 ? sv[2] : sv[3];
        const float y = t == 0 ? yv[0] : t == 1 ? yv[1] : t == 2 ? yv[2] : yv[3];
        const bool fast = t == 0 ? fv[0] : t == 1 ? fv[1] : t == 2 ? fv[2] : fv[3];
        const uint8_t* in = in_buf + stage * kFChunk * 2;
        uint8_t* out = out_buf + ob * kFChunk;
        uint4 a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a[k] = *reinterpret_cast<const uint4*>(in + (k * 32 + lane) * 16);
        float mc = 0.0f;
        if (fast) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint2*>(out + (k * 32 + lane) * 8) = fp8_encode8<FMT, true>(a[k], s, y, mc);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint2*>(out + (k * 32 + lane) * 8) = fp8_encode8<FMT, false>(a[k], s, y, mc);
        }
        m0 = t == 0 ? fmaxf(m0, mc) : m0;
        m1 = t == 1 ? fmaxf(m1, mc) : m1;
        m2 = t == 2 ? fmaxf(m2, mc) : m2;
        m3 = t == 3 ? fmaxf(m3, mc) : m3;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            bulk_store(set.x8[t] + (c - set.first[t]) * kFChunk, out, kFChunk);
            bulk_commit();
            if (i + kFStages < count) {
                mbar_arrive_expect_tx(&full[stage], kFChunk * 2);
                bulk_load(in_buf + stage * kFChunk * 2, src(c + kFStages * GW), kFChunk * 2, &full[stage]);
            }
        }
    }
    if (lane == 0) {
        if (i < count) {
            // gave up on a wait: let the loads already issued land before exiting
            for (int64_t j = i; j < count && j < i + kFStages; ++j)
                mbar_wait_drain(&full[j % kFStages], static_cast<uint32_t>((j / kFStages) & 1));
            bulk_wait_all();
        } else {
            // Only the stores' shared-memory reads are waited for: their
            // global writes complete before the grid does, and nothing in
            // this launch reads the codes.
            bulk_wait_read<0>();
        }
    }
    // ragged tails, fewer than kFChunk elements each: block 0
    if (blockIdx.x == 0) {
#pragma unroll
        for (int t = 0; t < (MULTI ? kFMaxTensors : 1); ++t) {
            if (t >= set.count) break;
            const uint16_t* x = set.x[t];
            uint8_t* x8 = set.x8[t];
            const float s = sv[t], y = yv[t];
            const bool fast = fv[t];
            float mt = 0.0f;
            for (int64_t e = (set.n[t] / kFChunk) * kFChunk + threadIdx.x; e < set.n[t]; e += blockDim.x) {
                const float f = __uint_as_float(static_cast<uint32_t>(x[e]) << 16);
                mt = fmaxf(mt, fabsf(f));
                const float q = fast ? fp8_quotient(f, s, y) : __fdiv_rn(f, s);
                x8[e] = static_cast<uint8_t>(fp8x2<FMT>(q, 0.0f) & 0xFFu);
            }
            m0 = t == 0 ? fmaxf(m0, mt) : m0;
            m1 = t == 1 ? fmaxf(m1, mt) : m1;
            m2 = t == 2 ? fmaxf(m2, mt) : m2;
            m3 = t == 3 ? fmaxf(m3, mt) : m3;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        if (MULTI) {
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
            m3 = fmaxf(m3, __shfl_xor_sync(0xffffffffu, m3, o));
        }
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = m0;
        red[1][threadIdx.x >> 5] = m1;
        red[2][threadIdx.x >> 5] = m2;
        red[3][threadIdx.x >> 5] = m3;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // max|x| >= 0, so the float order equals the unsigned order of the
        // bits.  The ticket is an acquire-release add: its release orders this
        // block's maxima before the ticket, and the last block's acquire
        // orders its read of the combined maxima after every other block's
        // release (all tickets are one chain of read-modify-writes).
        for (int t = 0; t < set.count; ++t) {
            float bm = red[t][0];
            for (int w = 1; w < nwarps; ++w) bm = fmaxf(bm, red[t][w]);
            red_max_relaxed_gpu(&ws[amax_word(t)], __float_as_uint(bm));
        }
        const unsigned ticket = atom_add_acq_rel_gpu(counter, 1u);
        is_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;          // uniform across the block
    if (threadIdx.x == 0) {
        // every other block's maxima are visible (ordered by the ticket), and
        // no block of this launch touches the words any more: a read and a
        // plain reset do what an exchange would, without waiting for it.
        // All words are read before any store, so the reads share one round
        // trip.
        constexpr int kT = MULTI ? kFMaxTensors : 1;
        unsigned bits[kT];
#pragma unroll
        for (int t = 0; t < kT; ++t) bits[t] = t < set.count ? ld_relaxed_gpu(&ws[amax_word(t)]) : 0u;
#pragma unroll
        for (int t = 0; t < kT; ++t) {
            if (t < set.count) {
                const float a = __uint_as_float(bits[t]);
                ws[amax_word(t)] = 0u;
                *set.amax[t] = a;
                s_amax[t] = a;
            }
        }
    }
    // delayed-scaling rings: hist[idx] = amax, the window's max, the next
    // step; all rings at once, so that their reads share one round trip
    constexpr int kR = MULTI ? kFMaxTensors : 1;
    bool any_ring = false;
#pragma unroll
    for (int t = 0; t < kR; ++t) any_ring |= t < set.count && set.ring[t] != nullptr;
    if (any_ring) {                    // uniform across the block
        __syncthreads();               // s_amax
        float wm[kR];
#pragma unroll
        for (int t = 0; t < kR; ++t) {
            wm[t] = 0.0f;
            if (t < set.count && set.ring[t]) {
                const float a = s_amax[t];
                for (int j = threadIdx.x; j < set.hist[t]; j += blockDim.x)
                    wm[t] = fmaxf(wm[t], j == set.ridx[t] ? a : set.ring[t][j]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm[t] = fmaxf(wm[t], __shfl_xor_sync(0xffffffffu, wm[t], o));
            if ((threadIdx.x & 31) == 0) red[t][threadIdx.x >> 5] = wm[t];
        }
        __syncthreads();
        if (threadIdx.x == 0) {
#pragma unroll
            for (int t = 0; t < kR; ++t) {
                float* ring = set.ring[t];
                if (t >= set.count || !ring) continue;
                float m = red[t][0];
                for (int w = 1; w < nwarps; ++w) m = fmaxf(m, red[t][w]);
                ring[set.ridx[t]] = s_amax[t];
                if (m > 0.0f) {
                    const float fmax_v = FMT == 0 ? 448.0f : 57344.0f;
                    ring[set.hist[t]] = __fdiv_rn(ldexpf(m, set.margin[t]), fmax_v);
                }
            }
        }
    }
    // every ticket of this launch is taken; the next launch on the stream
    // starts after this one completes
    if (threadIdx.x == 0) *counter = 0u;
}

template <int FMT, bool MULTI>
static cudaError_t launch_fp8_fmt(const Fp8Set& set, unsigned* ws, unsigned* counter,
                                  unsigned* err_word, cudaStream_t st, int sms) {
    const cudaError_t attr =
        set_max_dynamic_smem(reinterpret_cast<const void*>(quant_fp8_kernel<FMT, MULTI>), kQSmem);
    if (attr != cudaSuccess) return attr;
    const int64_t nfull = set.first[set.count];
    // Small tensors (under one chunk per warp of a full grid) run CTAs of 8
    // warps, several per SM, which start faster than one 24-warp CTA per SM.
    const int warps = nfull < static_cast<int64_t>(sms) * kFWarps ? 8 : kFWarps;
    const int smem = warps * kFWarpBytes + warps * kFStages * 8 + 128;
    int64_t blocks = (nfull + warps - 1) / warps;
    if (blocks < 1) blocks = 1;
    const int64_t cap = static_cast<int64_t>(sms) * (warps == kFWarps ? 1 : 3);
    if (blocks > cap) blocks = cap;
    return launch_pdl(quant_fp8_kernel<FMT, MULTI>, dim3(static_cast<unsigned>(blocks)), dim3(warps * 32),
                      static_cast<size_t>(smem), st, 1u, set, ws, counter, err_word);
}

static Fp8Set make_set(int count, const uint16_t* const* x, const int64_t* n,
                       const float* const* scale, uint8_t* const* x8, float* const* amax) {
    Fp8Set set;
    memset(&set, 0, sizeof(set));
    set.count = count;
    set.first[0] = 0;
    for (int t = 0; t < kFMaxTensors; ++t) {
        if (t < count) {
            set.x[t] = x[t];
            set.x8[t] = x8[t];
            set.scale[t] = scale[t];
            set.amax[t] = amax[t];
            set.n[t] = n[t];
            set.first[t + 1] = set.first[t] + n[t] / kFChunk;
        } else {
            set.first[t + 1] = INT64_MAX;
        }
    }
    return set;
}

static cudaError_t launch_set(const Fp8Set& set, int fmt, unsigned* ws, unsigned* counter,
                              unsigned* err_word, cudaStream_t st, int sms) {
    if (set.count == 1) {
        if (fmt == 0) return launch_fp8_fmt<0, false>(set, ws, counter, err_word, st, sms);
        return launch_fp8_fmt<1, false>(set, ws, counter, err_word, st, sms);
    }
    if (fmt == 0) return launch_fp8_fmt<0, true>(set, ws, counter, err_word, st, sms);
    return launch_fp8_fmt<1, true>(set, ws, counter, err_word, st, sms);
}

cudaError_t launch_quantize_fp8_multi(int count, const uint16_t* const* x, const int64_t* n,
                                      const float* const* scale, int fmt, uint8_t* const* x8,
                                      float* const* amax, unsigned* ws, unsigned* err_word,
                                      cudaStream_t st, int sms) {
    return launch_quantize_fp8_rings(count, x, n, scale, nullptr, nullptr, nullptr, nullptr, nullptr,
                                     fmt, x8, amax, ws, err_word, st, sms);
}

cudaError_t launch_quantize_fp8_rings(int count, const uint16_t* const* x, const int64_t* n,
                                      const float* const* scale, float* const* ring,
                                      const int* hist, const int* idx, const int* margin,
                                      float* const* used, int fmt, uint8_t* const* x8,
                                      float* const* amax, unsigned* ws, unsigned* err_word,
                                      cudaStream_t st, int sms) {
    if (count < 1 || count > kFMaxTensors) return cudaErrorInvalidValue;
    Fp8Set set = make_set(count, x, n, scale, x8, amax);
    for (int t = 0; t < count; ++t) {
        set.ring[t] = ring ? ring[t] : nullptr;
        set.hist[t] = hist ? hist[t] : 0;
        set.ridx[t] = idx ? idx[t] : 0;
        set.margin[t] = margin ? margin[t] : 0;
        set.used[t] = used ? used[t] : nullptr;
    }
    return launch_set(set, fmt, ws, ws + 1, err_word, st, sms);
}

cudaError_t launch_quantize_fp8(const uint16_t* x, int64_t n, const float* scale, int fmt,
                                uint8_t* x8, float* amax, unsigned* ws, float* ring, int hist_len,
                                int ring_idx, int margin, unsigned* err_word, cudaStream_t st,
                                int sms) {
    Fp8Set set = make_set(1, &x, &n, &scale, &x8, &amax);
    set.ring[0] = ring;
    set.hist[0] = hist_len;
    set.ridx[0] = ring_idx;
    set.margin[0] = margin;
    // one tensor with a ring: the ticket is the ring's counter word
    unsigned* counter = ring ? reinterpret_cast<unsigned*>(ring + hist_len + 1) : ws + 1;
    return launch_set(set, fmt, ws, counter, err_word, st, sms);
}

}  // namespace sq
