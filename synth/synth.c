/*
 * Seeded, counter-based synthetic inputs shared by the oracle and the GPU library.
 *
 * This file holds none of the decoder's arithmetic: it only produces numbers
 * (weights, token ids, cache contents, uniform draws) from a seed and a counter,
 * so that both sides of a comparison can be fed identical bytes.
 *
 * The integer hash and the exact uniform follow "bend-ml-llama 0.2.1.0, main.bend",
 * section "Sampling", definitions hash32 (Chris Wellons' lowbias32) and uniform
 * (top 24 bits of hash32(hash32(seed) + n) times 2^-24).  Normal values are drawn
 * with the Box-Muller transform from two such uniforms, in double precision, then
 * rounded to bf16 (round to nearest, ties to even) or kept as f32.
 *
 * Build: gcc -O2 -fPIC -shared -pthread synth.c -o libsynth.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

uint32_t synth_hash32(uint32_t x) {
  x ^= x >> 16;
  x *= 2146121005u;
  x ^= x >> 15;
  x *= 2221713035u;
  x ^= x >> 16;
  return x;
}

/* 24-bit draw n of a seed, as an integer in [0, 2^24). */
static inline uint32_t draw24(uint32_t seed_h, uint32_t n) {
  return synth_hash32(seed_h + n) >> 8;
}

float synth_uniform(uint32_t seed, uint32_t n) {
  return (float)draw24(synth_hash32(seed), n) * 5.9604644775390625e-8f;
}

void synth_uniforms(uint32_t seed, uint32_t n0, int64_t count, float* out) {
  uint32_t h = synth_hash32(seed);
  for (int64_t i = 0; i < count; ++i)
    out[i] = (float)draw24(h, n0 + (uint32_t)i) * 5.9604644775390625e-8f;
}

/* Token ids in [0, vocab): (draw24 * vocab) >> 24, in 64-bit integers. */
void synth_tokens(uint32_t seed, uint32_t n0, int64_t count, int32_t vocab, int32_t* out) {
  uint32_t h = synth_hash32(seed);
  for (int64_t i = 0; i < count; ++i)
    out[i] = (int32_t)(((uint64_t)draw24(h, n0 + (uint32_t)i) * (uint64_t)vocab) >> 24);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) /* inf / nan */
    return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* Element i of a normal tensor: Box-Muller on draws 2i and 2i+1 of the tensor's seed. */
static inline double normal_at(uint32_t seed_h, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double a = (double)draw24(seed_h, (uint32_t)(2 * i)) * (1.0 / 16777216.0);
  double b = (double)draw24(seed_h, (uint32_t)(2 * i + 1)) * (1.0 / 16777216.0);
  return sqrt(-2.0 * log(1.0 - a)) * cos(two_pi * b);
}

typedef struct {
  uint32_t seed_h;
  uint64_t lo, hi;
  double std, mean;
  int bf16;
  void* out;
} job_t;

static void* normal_job(void* arg) {
  job_t* j = (job_t*)arg;
  if (j->bf16) {
    uint16_t* o = (uint16_t*)j->out;
    for (uint64_t i = j->lo; i < j->hi; ++i)
      o[i] = f32_to_bf16_rne((float)(j->mean + j->std * normal_at(j->seed_h, i)));
  } else {
    float* o = (float*)j->out;
    for (uint64_t i = j->lo; i < j->hi; ++i)
      o[i] = (float)(j->mean + j->std * normal_at(j->seed_h, i));
  }
  return 0;
}

#define SYNTH_MAX_THREADS 64

/*
 * count values of N(mean, std^2) into out (bf16 bits if bf16 != 0, else f32).
 * The tensor seed is hash32(seed ^ tensor_idx); value i uses draws 2i and 2i+1,
 * so the result does not depend on nthreads.
 */
void synth_normal(uint32_t seed, uint32_t tensor_idx, int64_t count, double mean, double std,
                  int32_t bf16, void* out, int32_t nthreads) {
  uint32_t seed_h = synth_hash32(synth_hash32(seed ^ tensor_idx));
  if (nthreads < 1) nthreads = 1;
  if (nthreads > SYNTH_MAX_THREADS) nthreads = SYNTH_MAX_THREADS;
  if (count < 65536) nthreads = 1;
  job_t jobs[SYNTH_MAX_THREADS];
  pthread_t th[SYNTH_MAX_THREADS];
  uint64_t per = ((uint64_t)count + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t lo = per * (uint64_t)t, hi = lo + per;
    if (lo > (uint64_t)count) lo = (uint64_t)count;
    if (hi > (uint64_t)count) hi = (uint64_t)count;
    jobs[t] = (job_t){seed_h, lo, hi, std, mean, bf16, out};
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], 0, normal_job, &jobs[t]) != 0) break;
    started = t;
  }
  normal_job(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) normal_job(&jobs[t]); /* threads that failed to start */
  for (int t = 1; t <= started; ++t) pthread_join(th[t], 0);
}

void synth_const(int64_t count, float value, int32_t bf16, void* out) {
  if (bf16) {
    uint16_t b = f32_to_bf16_rne(value);
    uint16_t* o = (uint16_t*)out;
    for (int64_t i = 0; i < count; ++i) o[i] = b;
  } else {
    float* o = (float*)out;
    for (int64_t i = 0; i < count; ++i) o[i] = value;
  }
}

/*
 * The whole weight blob of a decoder, in the tensor order of the loader in
 * "bend-ml-llama 0.2.1.0, main.bend", section "Loading" (st_nth / t_layer):
 * embedding; for each layer ln1, q, k, v, o, ln2, gate, up, down; final norm;
 * then, for an untied head, the LM head.  Tensor t of layer i has index 1 + 9i + t;
 * the final norm 1 + 9L, the untied head 2 + 9L.  Matrices are N(0, wstd^2), the
 * norm gains are the constant `gain`.
 * dims: d (hidden), qw (query width), kvw (key width), f (MLP inner), L, V, tied.
 * Returns the number of elements written.
 */
int64_t synth_model_blob(int32_t d, int32_t qw, int32_t kvw, int32_t f, int32_t L, int32_t V,
                         int32_t tied, int32_t bf16, uint32_t seed, double wstd, float gain,
                         void* out, int32_t nthreads) {
  const int64_t es = bf16 ? 2 : 4;
  char* p = (char*)out;
  int64_t n = 0;
#define PUT_NORMAL(idx, cnt)                                                       \
  do {                                                                             \
    synth_normal(seed, (uint32_t)(idx), (cnt), 0.0, wstd, bf16, p + n * es, nthreads); \
    n += (cnt);                                                                    \
  } while (0)
#define PUT_GAIN(cnt)                              \
  do {                                             \
    synth_const((cnt), gain, bf16, p + n * es);    \
    n += (cnt);                                    \
  } while (0)
  PUT_NORMAL(0, (int64_t)V * d);
  for (int i = 0; i < L; ++i) {
    int64_t b = 1 + 9 * (int64_t)i;
    PUT_GAIN(d);
    PUT_NORMAL(b + 1, (int64_t)qw * d);
    PUT_NORMAL(b + 2, (int64_t)kvw * d);
    PUT_NORMAL(b + 3, (int64_t)kvw * d);
    PUT_NORMAL(b + 4, (int64_t)d * qw);
    PUT_GAIN(d);
    PUT_NORMAL(b + 6, (int64_t)f * d);
    PUT_NORMAL(b + 7, (int64_t)f * d);
    PUT_NORMAL(b + 8, (int64_t)d * f);
  }
  PUT_GAIN(d);
  if (!tied) PUT_NORMAL(2 + 9 * (int64_t)L, (int64_t)V * d);
#undef PUT_NORMAL
#undef PUT_GAIN
  return n;
}
