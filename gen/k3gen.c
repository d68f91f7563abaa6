/* k3gen.c -- seeded, counter-based synthetic input generator (definition in k3gen.h).
 * Plain C99 + POSIX threads.  Shared by both sides of every comparison; it holds
 * none of the MoE method's arithmetic. */
#include "k3gen.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define K3GEN_GAMMA 0x9E3779B97F4A7C15ull

static uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

static uint64_t base_of(uint64_t seed, uint64_t stream) {
  return mix64(seed * K3GEN_GAMMA + mix64(stream + K3GEN_GAMMA));
}

uint64_t k3gen_draw(uint64_t seed, uint64_t stream, uint64_t n) {
  return mix64(base_of(seed, stream) + (n + 1u) * K3GEN_GAMMA);
}

static double u53_of(uint64_t d) { return (double)(d >> 11) * (1.0 / 9007199254740992.0); }

double k3gen_u53(uint64_t seed, uint64_t stream, uint64_t n) {
  return u53_of(k3gen_draw(seed, stream, n));
}

void k3gen_bytes(uint64_t seed, uint64_t stream, uint64_t first, uint8_t *out, size_t n) {
  const uint64_t b = base_of(seed, stream);
  size_t i = 0;
  while (i < n) {
    const uint64_t pos = first + i;
    const uint64_t d = mix64(b + (pos / 8u + 1u) * K3GEN_GAMMA);
    unsigned j = (unsigned)(pos % 8u);
    if (j == 0 && n - i >= 8) {
      for (unsigned q = 0; q < 8; ++q) out[i + q] = (uint8_t)(d >> (8 * q));
      i += 8;
    } else {
      for (; j < 8 && i < n; ++j, ++i) out[i] = (uint8_t)(d >> (8 * j));
    }
  }
}

void k3gen_uint8_range(uint64_t seed, uint64_t stream, uint64_t first, uint8_t *out, size_t n,
                       int lo, int hi) {
  const uint64_t b = base_of(seed, stream);
  const double span = (double)(hi - lo + 1);
  for (size_t i = 0; i < n; ++i) {
    const uint64_t d = mix64(b + (first + i + 1u) * K3GEN_GAMMA);
    out[i] = (uint8_t)(lo + (int)floor(u53_of(d) * span));
  }
}

static double normal_at(uint64_t b, uint64_t n) {
  const double u1 = 1.0 - u53_of(mix64(b + (2u * n + 1u) * K3GEN_GAMMA));
  const double u2 = u53_of(mix64(b + (2u * n + 2u) * K3GEN_GAMMA));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

void k3gen_normal_f64(uint64_t seed, uint64_t stream, uint64_t first, double *out, size_t n) {
  const uint64_t b = base_of(seed, stream);
  for (size_t i = 0; i < n; ++i) out[i] = normal_at(b, first + i);
}

void k3gen_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, float *out, size_t n,
                      double sigma) {
  const uint64_t b = base_of(seed, stream);
  for (size_t i = 0; i < n; ++i) out[i] = (float)(sigma * normal_at(b, first + i));
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void k3gen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, uint16_t *out, size_t n,
                       double sigma) {
  const uint64_t b = base_of(seed, stream);
  for (size_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne((float)(sigma * normal_at(b, first + i)));
}

void k3gen_uniform_f64(uint64_t seed, uint64_t stream, uint64_t first, double *out, size_t n) {
  const uint64_t b = base_of(seed, stream);
  for (size_t i = 0; i < n; ++i) out[i] = u53_of(mix64(b + (first + i + 1u) * K3GEN_GAMMA));
}

/* ---- per-expert weights, threaded ---- */
typedef struct {
  uint64_t seed;
  int H, I, e0, e1, slo, shi;
  uint8_t *w13c, *w13s, *w2c, *w2s;
  int tid, nthreads;
} expert_job;

static void *expert_worker(void *arg) {
  const expert_job *j = (const expert_job *)arg;
  const size_t n13c = (size_t)2 * j->I * (j->H / 2), n13s = (size_t)2 * j->I * (j->H / 32);
  const size_t n2c = (size_t)j->H * (j->I / 2), n2s = (size_t)j->H * (j->I / 32);
  for (int e = j->e0 + j->tid; e < j->e1; e += j->nthreads) {
    const size_t r = (size_t)(e - j->e0);
    const uint64_t ue = (uint64_t)(uint32_t)e;
    if (j->w13c) k3gen_bytes(j->seed, ((uint64_t)K3GEN_KIND_W13_CODES << 32) | ue, 0, j->w13c + r * n13c, n13c);
    if (j->w13s)
      k3gen_uint8_range(j->seed, ((uint64_t)K3GEN_KIND_W13_SCALES << 32) | ue, 0, j->w13s + r * n13s, n13s,
                        j->slo, j->shi);
    if (j->w2c) k3gen_bytes(j->seed, ((uint64_t)K3GEN_KIND_W2_CODES << 32) | ue, 0, j->w2c + r * n2c, n2c);
    if (j->w2s)
      k3gen_uint8_range(j->seed, ((uint64_t)K3GEN_KIND_W2_SCALES << 32) | ue, 0, j->w2s + r * n2s, n2s,
                        j->slo, j->shi);
  }
  return NULL;
}

int k3gen_experts(uint64_t seed, int H, int I, int e0, int e1, int slo, int shi, uint8_t *w13c,
                  uint8_t *w13s, uint8_t *w2c, uint8_t *w2s, int nthreads) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32 || e0 < 0 || e1 < e0 || slo < 0 || shi > 255 || slo > shi)
    return -1;
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > e1 - e0) nthreads = e1 - e0 > 0 ? e1 - e0 : 1;
  if (nthreads > 256) nthreads = 256;
  expert_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    expert_job j = {seed, H, I, e0, e1, slo, shi, w13c, w13s, w2c, w2s, t, nthreads};
    jobs[t] = j;
  }
  if (nthreads == 1) {
    expert_worker(&jobs[0]);
    return 0;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, expert_worker, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = started; t < nthreads; ++t) expert_worker(&jobs[t]); /* run leftovers inline */
  return 0;
}
