/*
 * Seeded synthetic inputs for the layer-sliding fine-tuning step.
 *
 * This file holds input generation only: no part of the training step's
 * arithmetic lives here.  Both the CPU oracle's tests and the CUDA path's
 * tests and benchmark draw their inputs from it, so that the two sides see
 * bit-identical weights, tokens and labels.
 *
 * Generator (counter based, so any slice can be drawn independently and in
 * parallel):
 *   key(seed, stream)    = splitmix64(seed ^ splitmix64(stream + 1))
 *   word(seed, stream,i) = splitmix64(key + i)
 *   uniform(i)           = (word >> 11) * 2^-53              in [0, 1)
 *   normal(i)            = Box-Muller over the pair (2*(i/2), 2*(i/2)+1):
 *                          r = sqrt(-2 ln(1 - u0)), phi = 2 pi u1,
 *                          i even -> r cos(phi), i odd -> r sin(phi)
 *   randint(i, n)        = floor(uniform(i) * n)
 * splitmix64 is Steele, Lea and Flood's SplitMix64 finaliser
 * (OOPSLA 2014), with Vigna's published constants.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stddef.h>

/* Worker threads for the generators (the draws do not depend on it). */
void synth_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}

static inline uint64_t sm64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t key_of(uint64_t seed, uint64_t stream) {
  return sm64(seed ^ sm64(stream + 1ULL));
}

static inline double u53(uint64_t w) { return (double)(w >> 11) * 0x1.0p-53; }

/* out[j] = mean + std * normal(offset + j), j in [0, n); float32 output.
 * Each Box-Muller pair is computed once and gives both of its draws. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset,
                      int64_t n, double mean, double std, float* out) {
  if (n <= 0) return;
  const uint64_t key = key_of(seed, stream);
  const double two_pi = 6.283185307179586476925286766559;
  const uint64_t first = offset & ~1ULL, last = offset + (uint64_t)n;  /* [first, last) */
  const int64_t pairs = (int64_t)((last - first + 1ULL) / 2ULL);
#pragma omp parallel for schedule(static)
  for (int64_t q = 0; q < pairs; ++q) {
    const uint64_t p = first + 2ULL * (uint64_t)q;
    double u0 = u53(sm64(key + p));
    double u1 = u53(sm64(key + p + 1ULL));
    double r = sqrt(-2.0 * log(1.0 - u0));
    double ph = two_pi * u1;
    if (p >= offset) out[p - offset] = (float)(mean + std * (r * cos(ph)));
    if (p + 1ULL >= offset && p + 1ULL < last) out[p + 1ULL - offset] = (float)(mean + std * (r * sin(ph)));
  }
}

/* out[j] = floor(uniform(offset + j) * hi), int32 output in [0, hi). */
void synth_randint_i32(uint64_t seed, uint64_t stream, uint64_t offset,
                       int64_t n, int64_t hi, int32_t* out) {
  const uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) {
    double u = u53(sm64(key + offset + (uint64_t)j));
    int64_t v = (int64_t)(u * (double)hi);
    if (v >= hi) v = hi - 1;
    out[j] = (int32_t)v;
  }
}

/* out[j] = uniform(offset + j), float64 output in [0, 1). */
void synth_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset,
                       int64_t n, double* out) {
  const uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) out[j] = u53(sm64(key + offset + (uint64_t)j));
}
