/*
 * Seeded synthetic inputs for the tests and the benchmark.
 *
 * This file holds no quantization or GEMM arithmetic: it only draws numbers.
 * Both the CPU oracle and the CUDA library receive the arrays it fills, so
 * the two sides see identical inputs.
 *
 * Generator: counter-based.  Element c of the uniform stream of `seed` is
 *   z = splitmix64_mix(base + (c + 1) * GAMMA),  base = splitmix64_mix(seed)
 * with splitmix64 as published by Steele, Lea and Flood ("Fast splittable
 * pseudorandom number generators", OOPSLA 2014; constants of Vigna's
 * splitmix64.c).  u = ((z >> 11) + 0.5) * 2^-53 lies in (0, 1).
 * Normal draws use Box-Muller on the uniform pair (2j, 2j+1): element 2j is
 * r*cos(2*pi*u2), element 2j+1 is r*sin(2*pi*u2), r = sqrt(-2 ln u1).
 * Student-t with integer df d: element i uses normals (d+1)i .. (d+1)i+d,
 * t = Z0 / sqrt((Z1^2 + ... + Zd^2) / d).
 * Values are produced in fp64, then rounded to f32 (round to nearest even)
 * and, for bf16 output, from that f32 to bf16 (round to nearest even).
 * Every element depends only on (seed, index), so a sub-range can be drawn
 * on its own and the thread count does not change the result.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static double uniform01(uint64_t base, uint64_t c) {
    uint64_t z = mix64(base + (c + 1) * GAMMA);
    return ((double)(z >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static double normal_at(uint64_t base, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t j = i >> 1;
    double u1 = uniform01(base, 2 * j);
    double u2 = uniform01(base, 2 * j + 1);
    double r = sqrt(-2.0 * log(u1));
    return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* dist: 0 = normal(mean=p0, std=p1); 1 = p1 * student_t(df=(int)p0).
 * out_kind: 0 = float32, 1 = bf16 bit patterns (uint16).
 * Fills out[0..n) with elements start .. start+n-1 of the stream. */
int synth_fill(uint64_t seed, int dist, double p0, double p1,
               int64_t start, int64_t n, void* out, int out_kind) {
    if (n < 0 || start < 0 || (dist != 0 && dist != 1) || (out_kind != 0 && out_kind != 1))
        return -1;
    int df = (int)p0;
    if (dist == 1 && (df < 1 || df > 64)) return -1;
    const uint64_t base = mix64(seed);
    float* of = (float*)out;
    uint16_t* ob = (uint16_t*)out;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) {
        uint64_t i = (uint64_t)(start + k);
        double v;
        if (dist == 0) {
            v = p0 + p1 * normal_at(base, i);
        } else {
            uint64_t b = (uint64_t)(df + 1) * i;
            double z = normal_at(base, b);
            double chi = 0.0;
            for (int m = 1; m <= df; ++m) {
                double y = normal_at(base, b + (uint64_t)m);
                chi += y * y;
            }
            v = p1 * (z / sqrt(chi / (double)df));
        }
        float f = (float)v;
        if (out_kind == 0) of[k] = f;
        else ob[k] = f32_to_bf16_bits(f);
    }
    return 0;
}

/* The raw uniform stream, exposed so tests can check the generator itself. */
void synth_uniform(uint64_t seed, int64_t start, int64_t n, double* out) {
    const uint64_t base = mix64(seed);
    for (int64_t k = 0; k < n; ++k) out[k] = uniform01(base, (uint64_t)(start + k));
}
