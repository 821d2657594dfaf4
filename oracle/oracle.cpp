// CPU oracle for absmax-scaled quantization and the scaled low-precision GEMMs.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load this library.  It is deliberately
// plain and slow: every step is the written-out definition, with no blocking,
// fusion or reordering beyond what the definition states.  It shares no code,
// header, table or helper with the CUDA library.
//
// What it follows (sources are the three pages on the subject):
//  * INT8 symmetric quantization, "POPCORNBENCH Kimi-K2.6 l2_p13" trace,
//    reference-model analysis (amax = max|x| floored at 1e-8, scale = amax/127,
//    q = clamp(round(x/scale), -127, 127)) and its rounding discussion
//    (torch.round rounds halves to even: 0.5->0, 1.5->2, 2.5->2, -0.5->0,
//    -1.5->-2, -2.5->-2).  Applied per row ("per_row" granularity of the
//    scmp_kernels README, SC quickstart); per head = per row within each head.
//  * FP8 per-tensor quantization, AstrAI ops/fp8.py, module docstring and the
//    CPU kernel of custom::fp8_quantize: x8 = fp8(float(x) / scale), amax =
//    max|x|.  The scale is a quantization step that is divided out.
//  * FP8 GEMM, AstrAI ops/fp8.py, CPU kernel of custom::fp8_gemm:
//    out = bf16(float(a) @ float(b) * sa * sb).
// Readings where the pages are silent (all listed in the design notes):
//  * x/scale is one IEEE float32 division, rounded to nearest even.
//  * FP8 encoding rounds to nearest even and saturates to the largest finite
//    value (E4M3 +-448, E5M2 +-57344); subnormals are kept; codes follow the
//    OCP 8-bit floating point definition (E4M3 has no infinity, NaN = S.1111.111;
//    E5M2 infinity = S.11111.00, NaN = S.11111.xx with xx != 0).
//  * The returned FP8 amax is the raw max|x| (no floor).
//  * INT8 dequantization is (float(acc) * sA[i]) * sB[j], each product rounded
//    to float32, left to right.
//  * FP8 GEMM reference: the sum of decoded products in fp64, then * sa * sb in
//    fp64; the bf16 value reported is RNE(fl32(fl32(fl32(ref) * sa) * sb)).
//
// Build: g++ -O2 -std=c++17 -fopenmp -ffp-contract=off (no -ffast-math), so
// float expressions are evaluated one IEEE operation at a time.

#include <omp.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------- bits
float f32_from_bits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t bits_of_f32(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

// bf16 -> f32 is exact: the 16 stored bits are the top half of the f32.
float bf16_widen(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

// f32 -> bf16, round to nearest, ties to even (NaN stays NaN).
uint16_t bf16_round(float f) {
    uint32_t u = bits_of_f32(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;
    return (uint16_t)keep;
}

// ---------------------------------------------------------------- FP8 formats
struct Fp8 {
    int mbits;        // stored mantissa bits
    int ebits;        // exponent bits
    int bias;
    bool has_inf;     // E5M2 has infinities, E4M3 (fn) does not
    uint8_t max_code; // largest finite magnitude code
};
const Fp8 kE4M3 = {3, 4, 7, false, 0x7E};   // 1.110b * 2^8  = 448
const Fp8 kE5M2 = {2, 5, 15, true, 0x7B};   // 1.11b  * 2^15 = 57344

const Fp8* fmt_of(int fmt) { return fmt == 0 ? &kE4M3 : (fmt == 1 ? &kE5M2 : nullptr); }

bool code_is_nan(uint8_t c, const Fp8& f) {
    int e = (c >> f.mbits) & ((1 << f.ebits) - 1);
    int m = c & ((1 << f.mbits) - 1);
    int emax_field = (1 << f.ebits) - 1;
    if (f.has_inf) return e == emax_field && m != 0;
    return e == emax_field && m == (1 << f.mbits) - 1;
}

double decode(uint8_t c, const Fp8& f) {
    int s = c >> 7;
    int e = (c >> f.mbits) & ((1 << f.ebits) - 1);
    int m = c & ((1 << f.mbits) - 1);
    int emax_field = (1 << f.ebits) - 1;
    double v;
    if (code_is_nan(c, f)) return std::nan("");
    if (f.has_inf && e == emax_field) v = INFINITY;
    else if (e == 0) v = std::ldexp((double)m, 1 - f.bias - f.mbits);           // subnormal
    else v = std::ldexp((double)((1 << f.mbits) + m), e - f.bias - f.mbits);    // normal
    return s ? -v : v;
}

// Bit-level encoder: round the float32 magnitude to the nearest multiple of
// the FP8 unit in the last place at its exponent (ties to even), carry into
// the exponent, then saturate anything above the largest finite value.
uint8_t encode(float t, const Fp8& f) {
    uint32_t u = bits_of_f32(t);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint8_t)(sign | 0x7F);          // NaN -> NaN
    if (a == 0x7F800000u) return (uint8_t)(sign | f.max_code);   // inf saturates
    uint32_t E = a >> 23;
    if (E == 0) return sign;   // zero or f32 subnormal (< 2^-126): rounds to 0
    int e = (int)E - 127;
    uint64_t sig = (a & 0x7FFFFFu) | 0x800000u;   // value = sig * 2^(e-23)
    const int emin = 1 - f.bias;
    int shift = (e >= emin) ? (23 - f.mbits) : (23 - f.mbits + (emin - e));
    uint64_t q;
    if (shift >= 40) {
        q = 0;
    } else {
        q = sig >> shift;
        uint64_t rem = sig & ((1ull << shift) - 1);
        uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (q & 1))) q += 1;
    }
    int be;
    uint32_t mant;
    const uint64_t one = 1ull << f.mbits;
    if (e >= emin) {
        if (q == 2 * one) { q = one; e += 1; }
        be = e + f.bias;
        mant = (uint32_t)(q - one);
    } else {
        if (q == one) { be = 1; mant = 0; }
        else { be = 0; mant = (uint32_t)q; }
    }
    const int emax_field = (1 << f.ebits) - 1;
    uint32_t code = ((uint32_t)be << f.mbits) | mant;
    bool over;
    if (f.has_inf) over = be >= emax_field;
    else over = be > emax_field || (be == emax_field && mant == (uint32_t)(one - 1));
    if (over || code > f.max_code) code = f.max_code;
    return (uint8_t)(sign | code);
}

// Nearest integer, halves to even, for |t| < 2^31, written out from the
// definition (not rint): truncate, then look at the fractional part.
int32_t round_half_even(float t) {
    int64_t i = (int64_t)t;             // truncation toward zero (exact)
    float frac = t - (float)i;          // exact: same binade or below
    if (t >= 0.0f) {
        if (frac > 0.5f) return (int32_t)(i + 1);
        if (frac == 0.5f) return (int32_t)(i + (i & 1));
        return (int32_t)i;
    }
    if (frac < -0.5f) return (int32_t)(i - 1);
    if (frac == -0.5f) return (int32_t)(i - (i & 1));
    return (int32_t)i;
}

float load_elem(const void* x, int dtype, int64_t idx) {
    if (dtype == 0) return ((const float*)x)[idx];
    return bf16_widen(((const uint16_t*)x)[idx]);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- codec
double or_fp8_decode(uint8_t code, int fmt) {
    const Fp8* f = fmt_of(fmt);
    return f ? decode(code, *f) : std::nan("");
}

int or_fp8_encode_array(const float* t, int64_t n, int fmt, uint8_t* out) {
    const Fp8* f = fmt_of(fmt);
    if (!f || n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = encode(t[i], *f);
    return 0;
}

int or_fp8_code_is_nan(uint8_t code, int fmt) {
    const Fp8* f = fmt_of(fmt);
    return f ? (int)code_is_nan(code, *f) : -1;
}

int32_t or_round_half_even(float t) { return round_half_even(t); }

uint16_t or_bf16_round(float f) { return bf16_round(f); }

// ---------------------------------------------------------------- quantize
// Per-row symmetric INT8.  x: rows x cols, row stride ld elements, dtype
// 0 = float32, 1 = bf16 bits.  q: rows x cols packed (row stride cols).
int or_quantize_rowwise_i8(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                           int8_t* q, float* scales) {
    if (rows < 0 || cols < 0 || ld < cols || (dtype != 0 && dtype != 1)) return -1;
    const float floor_amax = 1e-8f;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < cols; ++k) {
            float a = std::fabs(load_elem(x, dtype, r * ld + k));
            if (a > amax) amax = a;
        }
        float a = amax < floor_amax ? floor_amax : amax;
        float s = a / 127.0f;
        scales[r] = s;
        for (int64_t k = 0; k < cols; ++k) {
            float t = load_elem(x, dtype, r * ld + k) / s;
            int32_t n = round_half_even(t);
            if (n > 127) n = 127;
            if (n < -127) n = -127;
            q[r * cols + k] = (int8_t)n;
        }
    }
    return 0;
}

// Row-group symmetric INT8 (scmp_kernels README: group_a / group_b row-group
// sizes; per_tensor granularity; the POPCORNBENCH trace's per-tensor formula):
// rows are split into consecutive groups of group_rows rows (the last may be
// shorter); each group g has s_g = fl32(max(max|x| over the group, 1e-8)/127)
// and q = clamp(rne(fl32(x / s_g)), -127, 127).  group_rows = 1 is per row;
// group_rows >= rows is per tensor.  scales: ceil(rows / group_rows) floats.
int or_quantize_grouped_i8(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                           int64_t group_rows, int8_t* q, float* scales) {
    if (rows < 0 || cols < 0 || ld < cols || group_rows < 1 || (dtype != 0 && dtype != 1))
        return -1;
    const int64_t ngroups = (rows + group_rows - 1) / group_rows;
    const float floor_amax = 1e-8f;
    for (int64_t g = 0; g < ngroups; ++g) {
        const int64_t r0 = g * group_rows;
        const int64_t r1 = r0 + group_rows < rows ? r0 + group_rows : rows;
        float amax = 0.0f;
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t k = 0; k < cols; ++k) {
                float a = std::fabs(load_elem(x, dtype, r * ld + k));
                if (a > amax) amax = a;
            }
        float a = amax < floor_amax ? floor_amax : amax;
        float s = a / 127.0f;
        scales[g] = s;
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t k = 0; k < cols; ++k) {
                float t = load_elem(x, dtype, r * ld + k) / s;
                int32_t n = round_half_even(t);
                if (n > 127) n = 127;
                if (n < -127) n = -127;
                q[r * cols + k] = (int8_t)n;
            }
    }
    return 0;
}

// Per-tensor FP8 quantize of bf16 input with the scale divided out; returns
// the raw amax = max|x| through *amax.
int or_quantize_fp8(const uint16_t* x, int64_t n, float scale, int fmt, uint8_t* x8,
                    float* amax) {
    const Fp8* f = fmt_of(fmt);
    if (!f || n < 0) return -1;
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = bf16_widen(x[i]);
        float a = std::fabs(v);
        if (a > m) m = a;
        x8[i] = encode(v / scale, *f);
    }
    *amax = m;
    return 0;
}

// Delayed scaling with a history ring (AstrAI ops/fp8.py, linear_forward_fp8
// docstring and commit notes: the measured amax lands in hist[idx] and the
// next step's scale is published on the device).  ring = [hist (H) | scale |
// counter]; the scale used for this quantization is ring[H].  After
// quantizing: hist[idx] = amax; m = max(hist); if m > 0 the next step is
// fl32(fl32(m * 2^margin) / fmt_max) (margin adds headroom; the pages give no
// formula -- at margin 0 this is the previous-amax / fmt_max recipe), else
// the scale is left as it was.  The counter slot is not touched.
int or_quantize_fp8_ring(const uint16_t* x, int64_t n, int fmt, uint8_t* x8, float* amax,
                         float* ring, int64_t H, int64_t idx, int margin) {
    const Fp8* f = fmt_of(fmt);
    if (!f || n < 0 || H < 1 || idx < 0 || idx >= H || margin < -64 || margin > 64) return -1;
    const float scale = ring[H];
    int rc = or_quantize_fp8(x, n, scale, fmt, x8, amax);
    if (rc) return rc;
    ring[idx] = *amax;
    float m = 0.0f;
    for (int64_t i = 0; i < H; ++i)
        if (ring[i] > m) m = ring[i];
    if (m > 0.0f) {
        const float fmax_f = (float)decode(f->max_code, *f);
        const float scaled = std::ldexp(m, margin);     // exact: a power-of-two scaling
        ring[H] = scaled / fmax_f;
    }
    return 0;
}

// ---------------------------------------------------------------- GEMMs
// INT8 GEMM, C[b] = A[b] * B[b]^T.  A[b]: M x K (batch stride sA_batch
// elements), B[b]: N x K.  acc is the exact integer sum (int64), checked to
// fit int32.  Output rows: `rows` (n_rows of them, indices into 0..M) or all
// rows when rows == NULL.  acc_out / c_out: [batch][n_rows][N].
// Scales: sa[b*M + i], sb[b*N + j].  Returns 1 if an accumulator left int32.
int or_gemm_i8(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
               int64_t batch, int64_t M, int64_t N, int64_t K,
               int64_t strideA, int64_t strideB,
               const int64_t* rows, int64_t n_rows,
               int32_t* acc_out, float* c_out) {
    if (batch < 0 || M < 0 || N < 0 || K < 0) return -1;
    if (!rows) n_rows = M;
    int overflow = 0;
    for (int64_t b = 0; b < batch; ++b) {
#pragma omp parallel for schedule(static) reduction(| : overflow)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t i = rows ? rows[r] : r;
            const int8_t* a = A + b * strideA + i * K;
            for (int64_t j = 0; j < N; ++j) {
                const int8_t* bb = B + b * strideB + j * K;
                int64_t acc = 0;
                for (int64_t k = 0; k < K; ++k) acc += (int64_t)a[k] * (int64_t)bb[k];
                if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
                int64_t o = (b * n_rows + r) * N + j;
                if (acc_out) acc_out[o] = (int32_t)acc;
                if (c_out) {
                    float c = (float)(int32_t)acc;
                    c = c * sa[b * M + i];
                    c = c * sb[b * N + j];
                    c_out[o] = c;
                }
            }
        }
    }
    return overflow;
}

// INT8 GEMM with row-group scales: like or_gemm_i8 but the dequantization
// uses sa[b*ceil(M/ga) + i/ga] and sb[b*ceil(N/gb) + j/gb].
int or_gemm_i8_grouped(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                       int64_t ga, int64_t gb, int64_t batch, int64_t M, int64_t N, int64_t K,
                       const int64_t* rows, int64_t n_rows, int32_t* acc_out, float* c_out) {
    if (batch < 0 || M < 0 || N < 0 || K < 0 || ga < 1 || gb < 1) return -1;
    if (!rows) n_rows = M;
    const int64_t Mg = (M + ga - 1) / ga, Ng = (N + gb - 1) / gb;
    int overflow = 0;
    for (int64_t b = 0; b < batch; ++b) {
#pragma omp parallel for schedule(static) reduction(| : overflow)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t i = rows ? rows[r] : r;
            const int8_t* a = A + (b * M + i) * K;
            for (int64_t j = 0; j < N; ++j) {
                const int8_t* bb = B + (b * N + j) * K;
                int64_t acc = 0;
                for (int64_t k = 0; k < K; ++k) acc += (int64_t)a[k] * (int64_t)bb[k];
                if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
                int64_t o = (b * n_rows + r) * N + j;
                if (acc_out) acc_out[o] = (int32_t)acc;
                if (c_out) {
                    float c = (float)(int32_t)acc;
                    c = c * sa[b * Mg + i / ga];
                    c = c * sb[b * Ng + j / gb];
                    c_out[o] = c;
                }
            }
        }
    }
    return overflow;
}

// FP8 GEMM reference.  layout 0 = NT: A[M,K], B[N,K], C = A B^T.
// 1 = NN: A[M,K], B[K,N], C = A B.  2 = TN: A[K,M], B[K,N], C = A^T B.
// All row-major and packed.  ref_out: [n_rows][N] fp64 sum of decoded
// products times sa times sb.  bf16_out (nullable): bf16 bits of
// RNE(fl32(fl32(fl32(sum) * sa) * sb)).
int or_gemm_fp8(const uint8_t* A, const uint8_t* B, int fmt, int layout,
                int64_t M, int64_t N, int64_t K, float sa, float sb,
                const int64_t* rows, int64_t n_rows, double* ref_out, uint16_t* bf16_out) {
    const Fp8* f = fmt_of(fmt);
    if (!f || layout < 0 || layout > 2 || M < 0 || N < 0 || K < 0) return -1;
    if (!rows) n_rows = M;
    double table[256];
    for (int c = 0; c < 256; ++c) table[c] = decode((uint8_t)c, *f);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t a = layout == 2 ? A[k * M + i] : A[i * K + k];
                uint8_t b = layout == 0 ? B[j * K + k] : B[k * N + j];
                sum += table[a] * table[b];
            }
            if (ref_out) ref_out[r * N + j] = sum * (double)sa * (double)sb;
            if (bf16_out) {
                float c = (float)sum;
                c = c * sa;
                c = c * sb;
                bf16_out[r * N + j] = bf16_round(c);
            }
        }
    }
    return 0;
}

// FP8 GEMM with an E4M3 output (AstrAI ops/fp8.py, fp8_gemm with out_dtype 1:
// the output quantized with its own step out_scale, divided out -- the
// adapter's docstring reading; its CPU path multiplies, the pages disagree).
// t_out: fp64 reference (sum * sa * sb) / out_scale; codes_out: E4M3 of
// fl32(fl32(fl32(fl32(sum) * sa) * sb) / out_scale).  Both nullable.
int or_gemm_fp8_e4m3(const uint8_t* A, const uint8_t* B, int fmt, int layout, int64_t M,
                     int64_t N, int64_t K, float sa, float sb, float out_scale,
                     const int64_t* rows, int64_t n_rows, double* t_out, uint8_t* codes_out) {
    const Fp8* f = fmt_of(fmt);
    if (!f || layout < 0 || layout > 2 || M < 0 || N < 0 || K < 0) return -1;
    if (!rows) n_rows = M;
    double table[256];
    for (int c = 0; c < 256; ++c) table[c] = decode((uint8_t)c, *f);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t a = layout == 2 ? A[k * M + i] : A[i * K + k];
                uint8_t b = layout == 0 ? B[j * K + k] : B[k * N + j];
                sum += table[a] * table[b];
            }
            if (t_out) t_out[r * N + j] = sum * (double)sa * (double)sb / (double)out_scale;
            if (codes_out) {
                float c = (float)sum;
                c = c * sa;
                c = c * sb;
                codes_out[r * N + j] = encode(c / out_scale, kE4M3);
            }
        }
    }
    return 0;
}

// FP8 GEMM with the bias added in the epilogue (AstrAI ops/fp8.py,
// linear_forward_fp8: the bias is fused into the GEMM epilogue).  bias_f32 is
// the bias already in float32 (nullable): a bf16 bias widened exactly, or a
// pre-quantized FP8 bias decoded and multiplied by its step (fl32).
// ref_out: fp64 sum * sa * sb + bias; bf16_out: RNE(fl32(fl32(fl32(fl32(sum) *
// sa) * sb) + bias)).
int or_gemm_fp8_bias(const uint8_t* A, const uint8_t* B, int fmt, int layout, int64_t M,
                     int64_t N, int64_t K, float sa, float sb, const float* bias_f32,
                     const int64_t* rows, int64_t n_rows, double* ref_out, uint16_t* bf16_out) {
    const Fp8* f = fmt_of(fmt);
    if (!f || layout < 0 || layout > 2 || M < 0 || N < 0 || K < 0) return -1;
    if (!rows) n_rows = M;
    double table[256];
    for (int c = 0; c < 256; ++c) table[c] = decode((uint8_t)c, *f);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t a = layout == 2 ? A[k * M + i] : A[i * K + k];
                uint8_t b = layout == 0 ? B[j * K + k] : B[k * N + j];
                sum += table[a] * table[b];
            }
            const float bj = bias_f32 ? bias_f32[j] : 0.0f;
            if (ref_out) ref_out[r * N + j] = sum * (double)sa * (double)sb + (double)bj;
            if (bf16_out) {
                float c = (float)sum;
                c = c * sa;
                c = c * sb;
                c = c + bj;
                bf16_out[r * N + j] = bf16_round(c);
            }
        }
    }
    return 0;
}

// Decoded FP8 bias: out[j] = fl32(decode(code[j]) * step).
int or_fp8_bias_to_f32(const uint8_t* codes, int64_t n, int fmt, float step, float* out) {
    const Fp8* f = fmt_of(fmt);
    if (!f || n < 0) return -1;
    for (int64_t j = 0; j < n; ++j) out[j] = (float)decode(codes[j], *f) * step;
    return 0;
}

// Column sums of a bf16 [T, N] matrix in fp64 (the gradient of a bias that
// is broadcast over the T rows).
int or_colsum_bf16(const uint16_t* g, int64_t T, int64_t N, double* out) {
    if (T < 0 || N < 0) return -1;
    for (int64_t j = 0; j < N; ++j) out[j] = 0.0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < N; ++j) out[j] += (double)bf16_widen(g[t * N + j]);
    return 0;
}

// Timing support only: the OpenMP thread count of the loops below.
void or_set_num_threads(int n) {
    if (n > 0) omp_set_num_threads(n);
}

int or_num_threads(void) {
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}

}  // extern "C"
