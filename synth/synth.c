/*
 * Seeded synthetic inputs for the lane-structured decoder: FP16 weight
 * tensors, token ids and KV-cache fill values.
 *
 * This file holds no arithmetic of the decode method itself; it only draws
 * random numbers.  Both the CPU oracle and the CUDA engine consume its output
 * (as raw FP16 bit patterns and int32 ids), so the two sides see identical
 * inputs without sharing any computation.
 *
 * Generator: the SplitMix64 sequence (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used counter-style: output i
 * of a stream with key K is mix64(K + (i + 1) * GAMMA).  Every element is a
 * pure function of (seed, stream, index), so the fill is identical for any
 * thread count.  Normals come from the Box-Muller transform on two such
 * outputs.  Values are rounded to FP16 (round to nearest even) by the
 * compiler's _Float16 conversion.
 */
#include <stdint.h>
#include <math.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GAMMA) + (stream + 1) * GAMMA);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GAMMA);
}

static inline uint16_t to_f16_bits(double v) {
    _Float16 h = (_Float16)v;
    uint16_t b;
    __builtin_memcpy(&b, &h, 2);
    return b;
}

/* out[i] = fp16(offset + scale * z_i), z_i ~ N(0, 1), i in [0, n). */
void synth_normal_f16(uint64_t seed, uint64_t stream, double scale, double offset,
                      uint16_t *out, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    const int64_t npair = (n + 1) / 2;
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < npair; ++j) {
        uint64_t a = draw(key, 2 * (uint64_t)j);
        uint64_t b = draw(key, 2 * (uint64_t)j + 1);
        double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
        double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
        double r = sqrt(-2.0 * log(u1));
        double z0 = r * cos(two_pi * u2);
        double z1 = r * sin(two_pi * u2);
        out[2 * j] = to_f16_bits(offset + scale * z0);
        if (2 * j + 1 < n) out[2 * j + 1] = to_f16_bits(offset + scale * z1);
    }
}

/* out[i] = v for every i (used for unit RMSNorm gains). */
void synth_fill_f16(double v, uint16_t *out, int64_t n) {
    uint16_t b = to_f16_bits(v);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = b;
}

/* Uniform token ids in [0, vocab): the high 32 bits scaled by vocab. */
void synth_tokens(uint64_t seed, uint64_t stream, int32_t vocab, int32_t *out, int64_t n) {
    const uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) {
        uint64_t b = draw(key, (uint64_t)i);
        out[i] = (int32_t)(((b >> 32) * (uint64_t)vocab) >> 32);
    }
}
