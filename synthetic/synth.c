/* Seeded synthetic operands: the fast implementation of the recipe stated in
 * synthetic/__init__.py (splitmix64 -> two uniforms -> Box-Muller -> mean/std
 * -> fp32 -> bf16).  It draws numbers only; nothing here belongs to the fused
 * Linear method.  Built with plain gcc (-O2, no fast-math) so both the x86 and
 * the Arm host produce the same values up to libm's last-ulp behaviour.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ull;

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * 256u + stream);
}

/* Standard normal for element index i of the stream keyed by `key`. */
static inline double normal_at(uint64_t key, int64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
    uint64_t j = (uint64_t)i >> 1;
    uint64_t a = mix64(key + (2u * j + 1u) * GOLDEN);
    uint64_t b = mix64(key + (2u * j + 2u) * GOLDEN);
    double u1 = ((double)(a >> 11) + 1.0) * inv53;
    double u2 = (double)(b >> 11) * inv53;
    double rho = sqrt(-2.0 * log(u1));
    double ang = two_pi * u2;
    return (i & 1) ? rho * sin(ang) : rho * cos(ang);
}

void synth_normal_f64(uint64_t key, int64_t start, int64_t count, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) out[t] = normal_at(key, start + t);
}

void synth_draw_f32(uint64_t key, int64_t start, int64_t count, double mean, double std,
                    float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) out[t] = (float)(mean + std * normal_at(key, start + t));
}

void synth_draw_bf16(uint64_t key, int64_t start, int64_t count, double mean, double std,
                     uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        float f = (float)(mean + std * normal_at(key, start + t));
        uint32_t bits;
        memcpy(&bits, &f, 4);
        bits += ((bits >> 16) & 1u) + 0x7FFFu;
        out[t] = (uint16_t)(bits >> 16);
    }
}
