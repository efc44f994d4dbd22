/*
 * Seeded synthetic inputs for the decode library and its CPU oracle.
 *
 * This module only draws random numbers and encodes them in the weight file
 * formats (F32, F16, Q8_0 blocks).  It holds none of the forward pass's
 * arithmetic, and both the oracle and the CUDA library receive its outputs
 * unchanged.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Value i of stream s under
 * seed k is the (i+1)-th output of SplitMix64 started from
 * key(k, s) = mix(k ^ mix(s + GOLDEN)), so any element can be drawn on its own
 * and the result does not depend on the number of threads.
 * Normals: Box-Muller (cosine branch) from values 2i and 2i+1.
 * Bounded integers: the high 32 bits times the range, shifted right by 32.
 * FP16 encoding: the compiler's _Float16 conversion (IEEE round to nearest even).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t key_of(uint64_t seed, uint64_t stream) { return mix(seed ^ mix(stream + GOLDEN)); }
static inline uint64_t draw(uint64_t key, uint64_t i) { return mix(key + (i + 1) * GOLDEN); }

static inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t a = draw(key, 2 * i), b = draw(key, 2 * i + 1);
    double u1 = (double)((a >> 11) + 1) * 0x1.0p-53;   /* (0, 1] */
    double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline uint16_t to_f16_bits(float v) {
    _Float16 h = (_Float16)v;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

/* Value i of the SplitMix64 sequence whose state starts at `state` (the
 * published generator itself, so that it can be checked against its
 * reference outputs); value i of stream s under seed k is this sequence at
 * state key(k, s). */
uint64_t syn_splitmix64_at(uint64_t state, uint64_t i) { return draw(state, i); }
uint64_t syn_draw(uint64_t seed, uint64_t stream, uint64_t i) { return draw(key_of(seed, stream), i); }
double syn_normal_at(uint64_t seed, uint64_t stream, uint64_t i) { return normal_at(key_of(seed, stream), i); }

/* out[i] = (float)(mean + std * N_i) */
void syn_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, float *out) {
    uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (float)(mean + std * normal_at(key, (uint64_t)i));
}

/* out[i] = f16((float)(mean + std * N_i)) */
void syn_normal_f16(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, uint16_t *out) {
    uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = to_f16_bits((float)(mean + std * normal_at(key, (uint64_t)i)));
}

/* out[i] uniform over the integers lo..hi */
void syn_uniform_i32(uint64_t seed, uint64_t stream, int64_t n, int32_t lo, int32_t hi, int32_t *out) {
    uint64_t key = key_of(seed, stream), range = (uint64_t)((int64_t)hi - lo + 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (int32_t)(lo + (int64_t)(((draw(key, (uint64_t)i) >> 32) * range) >> 32));
}

/* Q8_0 blocks (34 bytes: little-endian FP16 scale, then 32 signed bytes):
 * scale = f16((float)(|N| * dstd / 127)) from stream 2s, quants uniform over
 * -127..127 from stream 2s+1 (element index = block*32 + j). */
void syn_q8_0(uint64_t seed, uint64_t stream, int64_t nblocks, double dstd, uint8_t *out) {
    uint64_t ks = key_of(seed, 2 * stream), kq = key_of(seed, 2 * stream + 1);
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; b++) {
        uint8_t *blk = out + b * 34;
        uint16_t d = to_f16_bits((float)(fabs(normal_at(ks, (uint64_t)b)) * dstd / 127.0));
        blk[0] = (uint8_t)(d & 0xff);
        blk[1] = (uint8_t)(d >> 8);
        for (int j = 0; j < 32; j++) {
            uint64_t h = draw(kq, (uint64_t)(b * 32 + j));
            blk[2 + j] = (uint8_t)(int8_t)(-127 + (int64_t)(((h >> 32) * 255u) >> 32));
        }
    }
}
