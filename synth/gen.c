/*
 * Seeded synthetic inputs for the RVQ MoE expert FFN.
 *
 * This file holds input generation only: random bytes, normal samples and
 * the fp32 -> bf16 rounding of generated activations.  It contains none of
 * the method's arithmetic (no dequantisation, no lookup tables, no routing,
 * no FFN), so both the CPU oracle and the CUDA path can draw identical inputs
 * from it without sharing any compute code.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used counter-style: output i of a stream
 * with seed S is the SplitMix64 finaliser applied to S + (i + 1) * gamma,
 * which equals the (i+1)-th output of the sequential generator seeded with S.
 * Any index can therefore be generated independently, on any thread.
 *
 * Plain C11, libc + libm only; no architecture-specific code, so x86_64 and
 * aarch64 hosts produce the same bytes.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output number i (0-based) of the SplitMix64 stream seeded with seed. */
uint64_t synth_sm64_at(uint64_t seed, uint64_t i)
{
    return sm64_mix(seed + (i + 1) * SM64_GAMMA);
}

/* Child seed for a named sub-stream (tag) of a parent seed. */
uint64_t synth_derive(uint64_t seed, uint64_t tag)
{
    return sm64_mix(synth_sm64_at(seed, tag) ^ 0xA0761D6478BD642FULL);
}

/* Bytes [first, first + count) of the byte stream of seed: byte b is byte
 * (b mod 8) (little-endian) of output b / 8. */
void synth_bytes(uint64_t seed, uint64_t first, uint64_t count, uint8_t *out)
{
    uint64_t b = first, end = first + count;
    uint8_t *o = out;
    while (b < end && (b & 7u)) {
        *o++ = (uint8_t)(synth_sm64_at(seed, b >> 3) >> (8u * (b & 7u)));
        ++b;
    }
    while (b + 8 <= end) {
        uint64_t v = synth_sm64_at(seed, b >> 3);
        for (int i = 0; i < 8; ++i) o[i] = (uint8_t)(v >> (8 * i));
        o += 8;
        b += 8;
    }
    while (b < end) {
        *o++ = (uint8_t)(synth_sm64_at(seed, b >> 3) >> (8u * (b & 7u)));
        ++b;
    }
}

/* Uniform double in [0, 1) from the top 53 bits of an output. */
static inline double u01(uint64_t v) { return (double)(v >> 11) * 0x1.0p-53; }

/* count samples of N(0, sigma^2), rounded to fp32.  Sample 2p and 2p+1 come
 * from one Box-Muller pair built from outputs 2p and 2p+1 of the stream:
 * r = sqrt(-2 ln(1 - u1)), a = 2 pi u2, samples r cos a and r sin a. */
void synth_normal_f32(uint64_t seed, uint64_t count, double sigma, float *out)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (uint64_t p = 0; 2 * p < count; ++p) {
        double u1 = u01(synth_sm64_at(seed, 2 * p));
        double u2 = u01(synth_sm64_at(seed, 2 * p + 1));
        double r = sqrt(-2.0 * log(1.0 - u1));
        double a = two_pi * u2;
        out[2 * p] = (float)(sigma * r * cos(a));
        if (2 * p + 1 < count) out[2 * p + 1] = (float)(sigma * r * sin(a));
    }
}

/* fp32 -> bf16 bit pattern, round to nearest even (NaN kept quiet). */
uint16_t synth_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void synth_f32_to_bf16_array(const float *in, uint64_t count, uint16_t *out)
{
    for (uint64_t i = 0; i < count; ++i) out[i] = synth_f32_to_bf16(in[i]);
}

/* A seeded permutation of 0..n-1 (Fisher-Yates driven by the stream). */
void synth_permutation(uint64_t seed, int32_t n, int32_t *out)
{
    for (int32_t i = 0; i < n; ++i) out[i] = i;
    for (int32_t i = n - 1; i > 0; --i) {
        uint64_t v = synth_sm64_at(seed, (uint64_t)(n - 1 - i));
        int32_t j = (int32_t)(v % (uint64_t)(i + 1));
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}
