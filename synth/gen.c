/*
 * Seeded synthetic-input generator shared by the oracle and the CUDA path.
 *
 * It holds none of the model's arithmetic: it only turns (seed, stream, index)
 * into reproducible numbers.  Every value is a pure function of its index, so
 * the fill is order-free and runs in parallel.
 *
 *   u64   = splitmix64 chain over (seed, stream, index)
 *   N(0,1) via Box-Muller on the two 32-bit halves of one u64
 *   bf16  = round-to-nearest-even of the fp32 draw
 *
 * Built as a shared library and called through ctypes (synth/__init__.py).
 */
#include <stdint.h>
#include <math.h>

static inline uint64_t sm64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ULL;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ULL;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBULL;
    return x ^ (x >> 31);
}

static inline uint64_t draw_u64(uint64_t seed, uint64_t stream, uint64_t i) {
    return sm64(sm64(sm64(seed) ^ stream) ^ i);
}

static inline float draw_normal(uint64_t seed, uint64_t stream, uint64_t i) {
    uint64_t h = draw_u64(seed, stream, i);
    double u1 = ((double)(h >> 32) + 0.5) * (1.0 / 4294967296.0);   /* (0,1) */
    double u2 = (double)(h & 0xffffffffULL) * (1.0 / 4294967296.0); /* [0,1) */
    return (float)(sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2));
}

static inline uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    uint32_t bias = 0x7FFFu + ((v.u >> 16) & 1u);
    return (uint16_t)((v.u + bias) >> 16);
}

void synth_fill_normal_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, float std_) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = std_ * draw_normal(seed, stream, (uint64_t)i);
}

void synth_fill_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, float std_) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne(std_ * draw_normal(seed, stream, (uint64_t)i));
}

void synth_round_bf16(const float* in, uint16_t* out, int64_t n) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* Uniform integers in [lo, hi] (inclusive), one per index. */
void synth_fill_randint(int32_t* out, int64_t n, uint64_t seed, uint64_t stream, int32_t lo, int32_t hi) {
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
    for (int64_t i = 0; i < n; ++i)
        out[i] = lo + (int32_t)(draw_u64(seed, stream, (uint64_t)i) % span);
}

/* Raw 64-bit draws (used to build random logits for sampler tests). */
void synth_fill_u64(uint64_t* out, int64_t n, uint64_t seed, uint64_t stream) {
    for (int64_t i = 0; i < n; ++i) out[i] = draw_u64(seed, stream, (uint64_t)i);
}
