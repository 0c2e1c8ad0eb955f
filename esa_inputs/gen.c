/* Counter-based input generator (SplitMix64 + Box-Muller), see __init__.py
 * for the definition. Holds none of the attention method's arithmetic. */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

static inline uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t word(uint64_t key, uint64_t i) { return mix(key + (i + 1) * GAMMA); }

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    b = b + 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

void gen_normal_bf16(uint64_t key, int64_t start, int64_t n, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        uint64_t w1 = word(key, 2 * (uint64_t)(start + i)), w2 = word(key, 2 * (uint64_t)(start + i) + 1);
        double u1 = ((double)(w1 >> 11) + 0.5) * 0x1p-53, u2 = ((double)(w2 >> 11) + 0.5) * 0x1p-53;
        double z = sqrt(-2.0 * log(u1)) * cos(2.0 * 3.14159265358979323846 * u2);
        out[i] = f32_to_bf16_rne((float)z);
    }
}

void gen_int8_uniform(uint64_t key, int64_t start, int64_t n, int8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (int8_t)((int)(word(key, (uint64_t)(start + i)) >> 60) - 8);
}
