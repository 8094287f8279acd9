/*
 * Seeded synthetic input generator (bulk bf16 normals).
 *
 * This file holds no arithmetic of the fused linear + cross-entropy method: it only
 * draws the hidden states H and head weights W that both the CUDA path and the fp64
 * oracle consume, so that both sides read byte-identical bf16 inputs.
 *
 * Generator: counter-based.  Element k of stream `stream` under seed `seed` is a pure
 * function of (seed, stream, k), so any slice of a tensor (a row range) can be
 * regenerated on its own and threads can split the work without changing the values.
 *   key        = splitmix64(seed ^ splitmix64(stream))
 *   bits(j)    = splitmix64(key + j)            (j = 64-bit counter)
 *   u(j)       = (bits(j) >> 11) * 2^-53        (uniform on [0, 1))
 *   pair p     = Box-Muller on u1 = 1 - u(2p) in (0, 1], u2 = u(2p+1):
 *                r = sqrt(-2 ln u1); x(2p) = r cos(2 pi u2), x(2p+1) = r sin(2 pi u2)
 * splitmix64 is the mixing function published by Steele, Lea and Flood (OOPSLA 2014);
 * Box-Muller is the classical transform (Box and Muller, 1958).
 * The value is scaled by `stddev` in double precision, rounded to float, then to bf16
 * with round-to-nearest-even.  Values are host-side data only.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ULL;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ULL;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBULL;
  return x ^ (x >> 31);
}

static inline double unit_uniform(uint64_t key, uint64_t j) {
  return (double)(splitmix64(key + j) >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf stays inf */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static inline double normal_at(uint64_t key, uint64_t k) {
  uint64_t p = k >> 1;
  double u1 = 1.0 - unit_uniform(key, 2 * p);
  double u2 = unit_uniform(key, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  return (k & 1) ? r * sin(a) : r * cos(a);
}

typedef struct {
  uint16_t* out;
  uint64_t key;
  int64_t begin, end; /* absolute element indices */
  int64_t offset;     /* absolute index of out[0] */
  double stddev;
} job_t;

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t k = j->begin; k < j->end; ++k)
    j->out[k - j->offset] = f32_to_bf16_rne((float)(j->stddev * normal_at(j->key, (uint64_t)k)));
  return 0;
}

/* Fill out[0..count) with elements [offset, offset+count) of the normal stream. */
int synth_normal_bf16(uint16_t* out, int64_t offset, int64_t count, uint64_t seed, uint64_t stream,
                      double stddev, int nthreads) {
  if (count <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  uint64_t key = splitmix64(seed ^ splitmix64(stream));
  pthread_t th[256];
  int joinable[256];
  job_t jobs[256];
  int64_t per = (count + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = offset + (int64_t)t * per;
    int64_t e = b + per;
    if (e > offset + count) e = offset + count;
    if (b >= e) break;
    jobs[t].out = out;
    jobs[t].key = key;
    jobs[t].begin = b;
    jobs[t].end = e;
    jobs[t].offset = offset;
    jobs[t].stddev = stddev;
    joinable[t] = pthread_create(&th[t], 0, run_job, &jobs[t]) == 0;
    if (!joinable[t]) run_job(&jobs[t]);
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (joinable[t]) pthread_join(th[t], 0);
  return 0;
}

/* Uniform doubles on [0, 1) of the same counter stream (used for label draws). */
int synth_uniform_f64(double* out, int64_t offset, int64_t count, uint64_t seed, uint64_t stream) {
  uint64_t key = splitmix64(seed ^ splitmix64(stream));
  for (int64_t k = 0; k < count; ++k) out[k] = unit_uniform(key, (uint64_t)(offset + k));
  return 0;
}
