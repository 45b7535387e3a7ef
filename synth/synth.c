/*
 * synth.c -- seeded synthetic inputs for the radix-sort workloads.
 *
 * This file holds no sorting arithmetic.  It only draws keys and payloads that
 * the CUDA library and the CPU oracle both consume, so that the two sides see
 * exactly the same bytes.  Every draw comes from SplitMix64 (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) used
 * as a counter-based generator: draw i of a stream with seed s is
 * mix(s + (i + 1) * GOLDEN_GAMMA), which equals the i-th output of the
 * sequential generator started at state s.
 *
 * All functions write into caller-owned host memory and return 0 on success.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t sm64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Draw i of the stream with seed s. */
static inline uint64_t sm64_at(uint64_t s, uint64_t i)
{
    return sm64_mix(s + (i + 1) * GOLDEN_GAMMA);
}

/* Uniform double in [0, 1) from the top 53 bits of a draw. */
static inline double unit_open1(uint64_t x) { return (double)(x >> 11) * 0x1.0p-53; }

/* Uniform double in (0, 1] (never zero, for the logarithm of Box-Muller). */
static inline double unit_open0(uint64_t x) { return (double)((x >> 11) + 1) * 0x1.0p-53; }

/* Lemire's multiply-high reduction of a 64-bit draw to [0, bound). */
static inline uint64_t below(uint64_t x, uint64_t bound)
{
    return (uint64_t)(((unsigned __int128)x * bound) >> 64);
}

void synth_splitmix64(uint64_t* out, size_t n, uint64_t seed)
{
    for (size_t i = 0; i < n; ++i) out[i] = sm64_at(seed, i);
}

/* Keys uniform over all 32 bits: the high half of each draw. */
void synth_u32_uniform(uint32_t* out, size_t n, uint64_t seed)
{
    for (size_t i = 0; i < n; ++i) out[i] = (uint32_t)(sm64_at(seed, i) >> 32);
}

/* Keys uniform over all 64 bits. */
void synth_u64_uniform(uint64_t* out, size_t n, uint64_t seed)
{
    for (size_t i = 0; i < n; ++i) out[i] = sm64_at(seed, i);
}

/* Low-entropy keys: the AND of four uniform 32-bit words, so that each bit
 * is set with probability 1/16. */
void synth_u32_and4(uint32_t* out, size_t n, uint64_t seed)
{
    for (size_t i = 0; i < n; ++i) {
        uint32_t w = 0xFFFFFFFFu;
        for (int j = 0; j < 4; ++j) w &= (uint32_t)(sm64_at(seed, 4 * (uint64_t)i + j) >> 32);
        out[i] = w;
    }
}

/* Keys uniform over `bits` low bits (1..32); used for tie-heavy test inputs. */
void synth_u32_bits(uint32_t* out, size_t n, uint64_t seed, int bits)
{
    uint64_t mask = bits >= 32 ? 0xFFFFFFFFull : ((1ull << bits) - 1);
    for (size_t i = 0; i < n; ++i) out[i] = (uint32_t)((sm64_at(seed, i) >> 32) & mask);
}

/* Spread the low 10 bits of v so that bit b lands at bit 3b. */
static inline uint32_t spread3(uint32_t v)
{
    uint32_t r = 0;
    for (int b = 0; b < 10; ++b) r |= ((v >> b) & 1u) << (3 * b);
    return r;
}

/* 30-bit Morton codes of points uniform in [0,1)^3, each axis quantised to
 * 10 bits as q = min(floor(1024 c), 1023).  Bit 3b+2 holds x's bit b, 3b+1
 * holds y's and 3b holds z's.  Point i uses draws 3i, 3i+1, 3i+2. */
void synth_u32_morton30(uint32_t* out, size_t n, uint64_t seed)
{
    for (size_t i = 0; i < n; ++i) {
        uint32_t q[3];
        for (int a = 0; a < 3; ++a) {
            double c = unit_open1(sm64_at(seed, 3 * (uint64_t)i + a));
            double f = floor(1024.0 * c);
            q[a] = f > 1023.0 ? 1023u : (uint32_t)f;
        }
        out[i] = (spread3(q[0]) << 2) | (spread3(q[1]) << 1) | spread3(q[2]);
    }
}

/* Payload = original index. */
void synth_iota_u32(uint32_t* out, size_t n)
{
    for (size_t i = 0; i < n; ++i) out[i] = (uint32_t)i;
}

/*
 * float32 keys drawn N(0,1) by Box-Muller in double (key i uses draws 2i and
 * 2i+1), rounded to float.  Then `per_special` distinct positions each receive
 * -0.0, +0.0, +Inf, -Inf and the quiet NaN 0x7FC00000, in that order.  The
 * 5*per_special positions are the first entries of a partial Fisher-Yates
 * shuffle of 0..n-1 driven by the stream seed ^ 0xF15E5ull.  `scratch` must
 * hold n uint32 values (the index permutation).
 */
int synth_f32_normal_specials(uint32_t* out_bits, size_t n, uint64_t seed,
                              size_t per_special, uint32_t* scratch)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (size_t i = 0; i < n; ++i) {
        double u1 = unit_open0(sm64_at(seed, 2 * (uint64_t)i));
        double u2 = unit_open1(sm64_at(seed, 2 * (uint64_t)i + 1));
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        float f = (float)z;
        memcpy(&out_bits[i], &f, 4);
    }
    size_t total = 5 * per_special;
    if (total > n) return 1;
    if (total == 0) return 0;
    for (size_t i = 0; i < n; ++i) scratch[i] = (uint32_t)i;
    uint64_t pseed = seed ^ 0xF15E5ull;
    for (size_t j = 0; j < total; ++j) {
        size_t r = j + (size_t)below(sm64_at(pseed, j), (uint64_t)(n - j));
        uint32_t t = scratch[j]; scratch[j] = scratch[r]; scratch[r] = t;
    }
    static const uint32_t specials[5] = {0x80000000u, 0x00000000u, 0x7F800000u,
                                         0xFF800000u, 0x7FC00000u};
    for (size_t j = 0; j < total; ++j) out_bits[scratch[j]] = specials[j / per_special];
    return 0;
}

/*
 * Adversarial float32 bit patterns for edge-case tests: each key is drawn from
 * one of several classes chosen by the draw's low byte -- a boundary-value
 * table (zeros, min/max subnormals, FLT_MIN/FLT_MAX, infinities, quiet and
 * signalling NaNs of both signs with assorted payloads), uniform bit patterns
 * (which include every class) and N(0,1)-like values from a uniform mantissa.
 */
void synth_f32_edge(uint32_t* out_bits, size_t n, uint64_t seed)
{
    static const uint32_t table[] = {
        0x00000000u, 0x80000000u, 0x00000001u, 0x80000001u, 0x007FFFFFu, 0x807FFFFFu,
        0x00800000u, 0x80800000u, 0x7F7FFFFFu, 0xFF7FFFFFu, 0x7F800000u, 0xFF800000u,
        0x7FC00000u, 0xFFC00000u, 0x7F800001u, 0xFF800001u, 0x7FFFFFFFu, 0xFFFFFFFFu,
        0x7FA00000u, 0xFFBFFFFFu, 0x3F800000u, 0xBF800000u, 0x3F800001u, 0xBF800001u};
    const size_t nt = sizeof(table) / sizeof(table[0]);
    for (size_t i = 0; i < n; ++i) {
        uint64_t x = sm64_at(seed, i);
        uint32_t cls = (uint32_t)(x & 0xFF);
        uint32_t hi = (uint32_t)(x >> 32);
        if (cls < 64) {
            out_bits[i] = table[hi % nt];
        } else if (cls < 128) {
            out_bits[i] = hi;
        } else {
            /* sign, exponent in [120, 134), random mantissa */
            uint32_t sign = hi & 0x80000000u;
            uint32_t ex = 120u + ((hi >> 23) % 14u);
            out_bits[i] = sign | (ex << 23) | (hi & 0x007FFFFFu);
        }
    }
}
