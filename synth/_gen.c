/*
 * Seeded synthetic inputs: a counter-based generator for weights and token ids.
 *
 * This file holds no arithmetic of the transformer forward pass. It only turns
 * (seed, stream, index) into bits, so that the CPU oracle and the CUDA library
 * can be fed byte-identical inputs.
 *
 * Definition (stated here so that any other implementation can reproduce it):
 *   mix(z)      = splitmix64 finaliser: z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                 z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31.
 *   key(s, t)   = mix(mix(s + G) ^ (t * 0xD1B54A32D192ED03)),  G = 0x9E3779B97F4A7C15
 *   word(k, i)  = mix(k + (i + 1) * G)                          (all mod 2^64)
 *   normal pair j of stream (s, t): z = word(key, j);
 *       u1 = ((z >> 32) + 0.5) / 2^32,  u2 = (z & 0xffffffff) / 2^32,
 *       r = sqrt(-2 ln u1),  element 2j = r cos(2 pi u2),  element 2j+1 = r sin(2 pi u2)
 *     (Box-Muller), times sigma, plus mean, rounded to float32 (nearest),
 *     then to bfloat16 (round to nearest, ties to even).
 *   uniform id i in [0, V): ((word(key, i) >> 32) * V) >> 32.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define STREAM_MUL 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + GOLDEN) ^ (stream * STREAM_MUL));
}

static inline uint64_t word(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint64_t key;
  uint64_t begin, end; /* element range */
  double sigma, mean;
  uint16_t* out_bf16;
  float* out_f32;
} normal_job;

static void normal_range(const normal_job* j) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t e = j->begin;
  while (e < j->end) {
    uint64_t pair = e >> 1;
    uint64_t z = word(j->key, pair);
    double u1 = ((double)(z >> 32) + 0.5) * (1.0 / 4294967296.0);
    double u2 = (double)(z & 0xffffffffULL) * (1.0 / 4294967296.0);
    double r = sqrt(-2.0 * log(u1));
    double v[2] = {r * cos(two_pi * u2), r * sin(two_pi * u2)};
    for (int h = (int)(e & 1); h < 2 && e < j->end; ++h, ++e) {
      float f = (float)(v[h] * j->sigma + j->mean);
      if (j->out_bf16) j->out_bf16[e] = f32_to_bf16_rne(f);
      if (j->out_f32) j->out_f32[e] = f;
    }
  }
}

static void* normal_thread(void* p) {
  normal_range((const normal_job*)p);
  return 0;
}

/* Fill n elements of stream (seed, stream) with N(mean, sigma^2). Either output
 * may be NULL. out_f32 receives the float32 value before bf16 rounding. */
void synth_normal(uint64_t seed, uint64_t stream, uint64_t n, double sigma, double mean,
                  uint16_t* out_bf16, float* out_f32, int n_threads) {
  uint64_t key = synth_key(seed, stream);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 64) n_threads = 64;
  if (n < (1u << 16)) n_threads = 1;
  normal_job jobs[64];
  pthread_t tid[64];
  uint64_t chunk = ((n + n_threads - 1) / n_threads + 1) & ~1ULL; /* even split points */
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    uint64_t b = chunk * t, e = b + chunk;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[t] = (normal_job){key, b, e, sigma, mean, out_bf16, out_f32};
    if (t == 0) continue;
    if (pthread_create(&tid[t], 0, normal_thread, &jobs[t]) != 0) {
      normal_range(&jobs[t]);
      tid[t] = 0;
    }
    started = t;
  }
  normal_range(&jobs[0]);
  for (int t = 1; t <= started; ++t)
    if (tid[t]) pthread_join(tid[t], 0);
}

void synth_uniform_ids(uint64_t seed, uint64_t stream, uint64_t n, uint32_t vocab, int32_t* out) {
  uint64_t key = synth_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)(((word(key, i) >> 32) * (uint64_t)vocab) >> 32);
}

void synth_words(uint64_t seed, uint64_t stream, uint64_t n, uint64_t* out) {
  uint64_t key = synth_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = word(key, i);
}
