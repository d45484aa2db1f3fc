/*
 * Seeded synthetic inputs for the ring-attention workloads.
 *
 * This file holds random-number generation only: no attention arithmetic.
 * It serves both the fp64 oracle and the GPU library, which share nothing else.
 *
 * Generator (two published methods, written from their definitions):
 *   - SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): the n-th output (n = 0, 1, ...) is
 *     mix(seed + (n + 1) * 0x9E3779B97F4A7C15), where mix is the
 *     xor-shift/multiply finaliser with shifts 30, 27, 31.
 *   - Box-Muller (Box & Muller, 1958): two uniforms u1 in (0,1], u2 in [0,1)
 *     give R = sqrt(-2 ln u1), theta = 2 pi u2, and the normals R cos(theta),
 *     R sin(theta).
 * Element n of a stream uses outputs 2*(n/2) and 2*(n/2)+1; even n takes the
 * cosine branch, odd n the sine branch.  The value is computed in fp64, cast
 * to fp32, then rounded to bf16 with round-to-nearest-even, and finally
 * multiplied by a power-of-two factor (exact in bf16).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* n-th output of the SplitMix64 sequence started from `seed`. */
uint64_t ri_splitmix64(uint64_t seed, uint64_t n) {
  return sm64_mix(seed + (n + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf/nan: not produced */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline double normal_at(uint64_t seed, uint64_t n) {
  const uint64_t p = n >> 1;
  const uint64_t x1 = ri_splitmix64(seed, 2 * p);
  const uint64_t x2 = ri_splitmix64(seed, 2 * p + 1);
  const double u1 = (double)((x1 >> 11) + 1ULL) * 0x1.0p-53; /* (0, 1] */
  const double u2 = (double)(x2 >> 11) * 0x1.0p-53;          /* [0, 1) */
  const double r = sqrt(-2.0 * log(u1));
  const double th = 6.283185307179586476925286766559 * u2;
  return (n & 1) ? r * sin(th) : r * cos(th);
}

typedef struct {
  uint64_t seed, first;
  int64_t count;
  float mult;
  uint16_t *out;
} job_t;

static void *normal_worker(void *arg) {
  job_t *j = (job_t *)arg;
  for (int64_t i = 0; i < j->count; ++i) {
    float f = (float)normal_at(j->seed, j->first + (uint64_t)i);
    uint16_t b = f32_to_bf16_rne(f);
    if (j->mult != 1.0f) {
      uint32_t u = (uint32_t)b << 16;
      float g;
      memcpy(&g, &u, 4);
      b = f32_to_bf16_rne(g * j->mult); /* power of two: exact */
    }
    j->out[i] = b;
  }
  return NULL;
}

/*
 * Fill out[0..count) with bf16 bit patterns of stream elements
 * first .. first+count-1 for `seed`, scaled by `mult` (a power of two).
 * Returns 0 on success.
 */
int ri_normal_bf16(uint64_t seed, uint64_t first, int64_t count, float mult,
                   uint16_t *out, int n_threads) {
  if (count < 0 || (count > 0 && !out)) return 1;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (count < (int64_t)1 << 16) n_threads = 1;
  pthread_t th[256];
  job_t jobs[256];
  int64_t per = (count + n_threads - 1) / n_threads;
  per = (per + 1) & ~(int64_t)1;
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    int64_t lo = (int64_t)t * per;
    if (lo >= count) break;
    int64_t hi = lo + per < count ? lo + per : count;
    jobs[t] = (job_t){seed, first + (uint64_t)lo, hi - lo, mult, out + lo};
    if (n_threads == 1) {
      normal_worker(&jobs[t]);
    } else if (pthread_create(&th[t], NULL, normal_worker, &jobs[t]) != 0) {
      normal_worker(&jobs[t]);
      th[t] = 0;
      jobs[t].count = -1;
    }
    started = t + 1;
  }
  if (n_threads > 1)
    for (int t = 0; t < started; ++t)
      if (jobs[t].count >= 0) pthread_join(th[t], NULL);
  return 0;
}

/* Uniform in [0,1) from output n of the sequence for `seed` (53-bit). */
double ri_uniform(uint64_t seed, uint64_t n) {
  return (double)(ri_splitmix64(seed, n) >> 11) * 0x1.0p-53;
}
