/*
 * Seeded synthetic input generator shared by the CUDA path's tests/bench and
 * the CPU oracle.  It holds none of the forward pass's arithmetic: it only
 * draws weights, norm scales and token ids.
 *
 * Every tensor is an independent counter-based stream keyed by (seed, tensor
 * id), so any slice of any tensor can be produced on its own, in parallel, in
 * any order, with identical bytes.
 *
 *   mix(z)       SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable
 *                pseudorandom number generators", OOPSLA 2014; constants as
 *                published in Vigna's reference splitmix64.c).
 *   key          mix(seed ^ mix(tensor_id + GOLDEN))
 *   word(c)      mix(key + (c + 1) * GOLDEN)      counter c = 0, 1, 2, ...
 *   normal pair  Box-Muller (1958) on u1 = (word(2j) >> 11 + 1) / 2^53 in (0,1]
 *                and u2 = (word(2j+1) >> 11) / 2^53 in [0,1):
 *                  r = sqrt(-2 ln u1);  z[2j] = r cos(2 pi u2), z[2j+1] = r sin(2 pi u2)
 *                element value = (float)(mean + std * z) computed in double.
 *   uniform int  floor(word(i) * bound / 2^64) (multiply-high), in [0, bound).
 *
 * Built with -ffp-contract=off so that no platform fuses the double products.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix(seed ^ mix(tensor_id + GOLDEN));
}

static inline uint64_t word(uint64_t key, uint64_t c) { return mix(key + (c + 1) * GOLDEN); }

uint64_t synth_word(uint64_t seed, uint64_t tensor_id, uint64_t counter) {
    return word(stream_key(seed, tensor_id), counter);
}

static inline void normal_pair(uint64_t key, uint64_t j, double* z0, double* z1) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = (double)((word(key, 2 * j) >> 11) + 1) * (1.0 / 9007199254740992.0);
    double u2 = (double)(word(key, 2 * j + 1) >> 11) * (1.0 / 9007199254740992.0);
    double r = sqrt(-2.0 * log(u1));
    double a = two_pi * u2;
    *z0 = r * cos(a);
    *z1 = r * sin(a);
}

/* out[i] = mean + std * z[start + i] for i in [0, n). */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n, double mean,
                      double std, float* out) {
    const uint64_t key = stream_key(seed, tensor_id);
    long long npairs = (long long)((start + n + 1) / 2 - start / 2);
    uint64_t j0 = start / 2;
#pragma omp parallel for schedule(static)
    for (long long p = 0; p < npairs; ++p) {
        uint64_t j = j0 + (uint64_t)p;
        double z0, z1;
        normal_pair(key, j, &z0, &z1);
        uint64_t e0 = 2 * j, e1 = 2 * j + 1;
        if (e0 >= start && e0 < start + n) out[e0 - start] = (float)(mean + std * z0);
        if (e1 >= start && e1 < start + n) out[e1 - start] = (float)(mean + std * z1);
    }
}

/* out[i] = uniform integer in [0, bound) for counter start + i. */
void synth_uniform_u32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n, uint32_t bound,
                       uint32_t* out) {
    const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; ++i) {
        uint64_t w = word(key, start + (uint64_t)i);
        out[i] = (uint32_t)(((unsigned __int128)w * bound) >> 64);
    }
}
