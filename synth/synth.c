/*
 * Seeded synthetic inputs: a counter-based generator.
 *
 * This file holds no arithmetic of the MoE method.  It only turns
 * (seed, stream, index) into pseudo-random numbers so that the CPU oracle,
 * the tests and the benchmark can build identical inputs of any size,
 * in any order and on any number of threads.
 *
 *   mix(x)      = the SplitMix64 output function (Steele, Lea and Flood,
 *                 "Fast splittable pseudorandom number generators",
 *                 OOPSLA 2014), gamma 0x9E3779B97F4A7C15.
 *   key         = mix(mix(seed) ^ stream)
 *   bits(i)     = mix(key + i * gamma)
 *   uniform(i)  = ((bits(i) >> 11) + 0.5) * 2^-53          in (0, 1)
 *   normal(i)   = Box-Muller on the pair (uniform(2p), uniform(2p+1)),
 *                 p = i / 2; even i takes the cosine branch, odd i the sine.
 */
#include <math.h>
#include <stdint.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z += SYNTH_GAMMA;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed) ^ stream);
}

static inline double unit_open(uint64_t key, uint64_t i) {
  uint64_t b = mix64(key + i * SYNTH_GAMMA);
  return ((double)(b >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t p = i >> 1;
  double u1 = unit_open(key, 2 * p);
  double u2 = unit_open(key, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

/* out[t] = scale * normal(offset + t), rounded to float, t in [0, n). */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double scale, float* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) out[t] = (float)(scale * normal_at(key, offset + (uint64_t)t));
}

/* out[t] = normal(offset + t) in double. */
void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) out[t] = normal_at(key, offset + (uint64_t)t);
}

/* out[t] = uniform(offset + t) in (0, 1). */
void synth_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) out[t] = unit_open(key, offset + (uint64_t)t);
}
