/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * oracle's callers.  It holds none of the attention arithmetic: it only turns
 * (seed, stream, index) into numbers.
 *
 * Generator (counter-based, so any slice can be produced independently and
 * in parallel):
 *   splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014; finaliser constants as published by S. Vigna).
 *   The n-th output of a stream with key K is  mix(K + (n+1) * GAMMA),
 *   exactly the n-th output of the sequential splitmix64 generator seeded
 *   with K.
 *   key(seed, stream) = mix(seed * 0x100 + stream).
 *
 * Normals: Box-Muller on pairs (element 2p uses cos, 2p+1 uses sin) with
 *   u1 = (top 53 bits of draw 2p + 1) * 2^-53  in (0, 1]
 *   u2 = (top 53 bits of draw 2p+1)   * 2^-53  in [0, 1)
 * computed in double, rounded to float, multiplied by `mult` (the configs use
 * 1 or 2, both exact), then rounded to bfloat16 with round-to-nearest-even.
 *
 * Plain C99 + OpenMP; no architecture-specific code, so x86_64 and aarch64
 * builds give the same bits (up to libm's correctly-rounded-in-practice
 * log/sin/cos, which are then rounded twice more).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0x100ull + stream);
}

static inline uint64_t draw(uint64_t key, uint64_t n) {
  return mix64(key + (n + 1ull) * GAMMA);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* Raw 64-bit draws n = start .. start+count-1 of stream (seed, stream). */
void bsgen_u64(uint64_t seed, uint64_t stream, int64_t start, int64_t count,
               uint64_t* out) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = draw(key, (uint64_t)(start + i));
}

/* Uniform doubles in [0, 1): top 53 bits of each draw times 2^-53. */
void bsgen_uniform(uint64_t seed, uint64_t stream, int64_t start, int64_t count,
                   double* out) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i)
    out[i] = (double)(draw(key, (uint64_t)(start + i)) >> 11) * 0x1.0p-53;
}

static inline double normal_at(uint64_t key, uint64_t e) {
  const uint64_t p = e >> 1;
  const double u1 = (double)((draw(key, 2 * p) >> 11) + 1ull) * 0x1.0p-53;
  const double u2 = (double)(draw(key, 2 * p + 1) >> 11) * 0x1.0p-53;
  const double r = sqrt(-2.0 * log(u1));
  const double t = 6.283185307179586476925286766559 * u2;
  return (e & 1ull) ? r * sin(t) : r * cos(t);
}

/* Normal(0,1) * mult, rounded to bf16 (bit patterns), elements start .. start+count-1. */
void bsgen_normal_bf16(uint64_t seed, uint64_t stream, int64_t start, int64_t count,
                       float mult, uint16_t* out) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    float f = (float)normal_at(key, (uint64_t)(start + i));
    out[i] = f32_to_bf16_rne(f * mult);
  }
}

/* Normal(0,1) * mult in double precision (no rounding), for fp64 oracle tests. */
void bsgen_normal_f64(uint64_t seed, uint64_t stream, int64_t start, int64_t count,
                      double mult, double* out) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i)
    out[i] = normal_at(key, (uint64_t)(start + i)) * mult;
}

/* Raw splitmix64 outputs for an explicit key (the n-th output, n = start ..);
   exposed so the tests can check the published splitmix64 sequence. */
void bsgen_splitmix64_raw(uint64_t key, int64_t start, int64_t count, uint64_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = draw(key, (uint64_t)(start + i));
}
