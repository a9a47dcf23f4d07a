/*
 * Seeded synthetic inputs shared by the oracle tests, the CUDA-path tests
 * and the benchmark.  This file holds no arithmetic of the decode step: it
 * only turns (seed, tensor id, element index) into numbers.
 *
 * Generator (stated here so that any implementation can reproduce it):
 *   - splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014) used as a counter-based generator: the n-th
 *     64-bit draw of a stream with key K is mix64(K + (n+1)*GAMMA).
 *   - a stream key is mix64(seed ^ mix64(tensor_id*GAMMA + 1)).
 *   - uniforms take the top 53 bits: u = ((r >> 11) + 1) * 2^-53 in (0, 1].
 *   - normals use Box and Muller (1958): element i of a tensor uses the pair
 *     j = i/2, u1 = draw 2j, u2 = draw 2j+1, rad = sqrt(-2 ln u1),
 *     z = rad*cos(2 pi u2) for even i, rad*sin(2 pi u2) for odd i;
 *     the value is (float)(mean + std*z), computed in double.
 *   - token ids are draw(i) mod vocab.
 */
#include <math.h>
#include <stdint.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(seed ^ mix64(tensor_id * SYNTH_GAMMA + 1ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t n) {
    return mix64(key + (n + 1ULL) * SYNTH_GAMMA);
}

static inline double unit_open0(uint64_t r) {
    return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

uint64_t synth_draw_u64(uint64_t seed, uint64_t tensor_id, uint64_t n) {
    return draw(stream_key(seed, tensor_id), n);
}

/* out[k] = mean + std * z(start + k), k in [0, count).  Works pair by pair:
 * both normals of a Box-Muller pair come from one (u1, u2). */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count,
                      double mean, double std, float *out) {
    if (count == 0) return;
    const uint64_t key = stream_key(seed, tensor_id);
    const double two_pi = 6.283185307179586476925286766559;
    const long long j0 = (long long)(start >> 1), j1 = (long long)((start + count - 1) >> 1);
#pragma omp parallel for schedule(static)
    for (long long j = j0; j <= j1; j++) {
        double u1 = unit_open0(draw(key, 2 * (uint64_t)j));
        double u2 = unit_open0(draw(key, 2 * (uint64_t)j + 1));
        double rad = sqrt(-2.0 * log(u1));
        double z[2] = {rad * cos(two_pi * u2), rad * sin(two_pi * u2)};
        for (int e = 0; e < 2; e++) {
            uint64_t i = 2 * (uint64_t)j + (uint64_t)e;
            if (i >= start && i < start + count) out[i - start] = (float)(mean + std * z[e]);
        }
    }
}

/* out[k] = draw(start + k) mod vocab, k in [0, count). */
void synth_tokens_i32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count,
                      uint32_t vocab, int32_t *out) {
    const uint64_t key = stream_key(seed, tensor_id);
    for (uint64_t k = 0; k < count; k++)
        out[k] = (int32_t)(draw(key, start + k) % (uint64_t)vocab);
}
