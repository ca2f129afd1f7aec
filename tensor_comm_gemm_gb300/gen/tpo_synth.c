/*
 * Seeded synthetic input generation (host C, threaded).
 *
 * This file draws and rounds random inputs only; it holds none of the
 * tensor-parallel GEMM arithmetic.  It implements exactly the recipe stated in
 * tensor_comm_gemm_gb300/synth.py (splitmix64 counter streams, uniform[-1,1),
 * Box-Muller normals, bf16 round-to-nearest-even, OCP e4m3 round-to-nearest-
 * even with saturation), so that large workloads generate in seconds.  The
 * numpy functions in synth.py are the readable definition; a CPU test checks
 * that the two agree.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

static inline uint16_t f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

static inline uint8_t f32_to_e4m3(float x) {
  uint32_t bits;
  memcpy(&bits, &x, 4);
  uint8_t sign = (uint8_t)((bits >> 31) << 7);
  double a = fabs((double)x);
  int e2;
  (void)frexp(a, &e2);
  int e = e2 - 1;
  if (e < -6) e = -6;
  double q = ldexp(1.0, e - 3);
  double v = nearbyint(a / q) * q; /* default rounding mode: nearest, ties to even */
  if (v > 448.0) v = 448.0;
  uint8_t code;
  if (v < ldexp(1.0, -6)) {
    code = (uint8_t)nearbyint(v / ldexp(1.0, -9));
  } else {
    (void)frexp(v, &e2);
    int ev = e2 - 1;
    int mant = (int)nearbyint(v / ldexp(1.0, ev - 3)) - 8;
    code = (uint8_t)(((ev + 7) << 3) | mant);
  }
  return (uint8_t)(code | sign);
}

typedef struct {
  int kind; /* 0 uniform->bf16, 1 normal->bf16, 2 normal->f32, 3 f32*scale->e4m3 */
  uint64_t key;
  int64_t start, count;
  double sigma;
  float scale;
  const float* in;
  void* out;
} job_t;

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  for (int64_t t = 0; t < j->count; ++t) {
    int64_t i = j->start + t;
    if (j->kind == 0) {
      float u = (float)(draw(j->key, (uint64_t)i) >> 40) * 0x1p-24f;
      ((uint16_t*)j->out)[i] = f32_to_bf16(2.0f * u - 1.0f);
    } else if (j->kind == 1 || j->kind == 2) {
      uint64_t d0 = draw(j->key, 2 * (uint64_t)i), d1 = draw(j->key, 2 * (uint64_t)i + 1);
      double u1 = (double)((d0 >> 11) + 1) * 0x1p-53;
      double u2 = (double)(d1 >> 11) * 0x1p-53;
      double z = sqrt(-2.0 * log(u1)) * cos(2.0 * M_PI * u2);
      float f = (float)(z * j->sigma);
      if (j->kind == 1)
        ((uint16_t*)j->out)[i] = f32_to_bf16(f);
      else
        ((float*)j->out)[i] = f;
    } else {
      float f = j->in[i] * j->scale;
      ((uint8_t*)j->out)[i] = f32_to_e4m3(f);
    }
  }
  return NULL;
}

static int run(job_t proto, int64_t count, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  job_t jobs[256];
  int64_t per = (count + nthreads - 1) / nthreads;
  int used = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t s = (int64_t)t * per;
    if (s >= count) break;
    jobs[t] = proto;
    jobs[t].start = s;
    jobs[t].count = (s + per <= count) ? per : count - s;
    if (pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0) {
      run_job(&jobs[t]);
      th[t] = 0;
    }
    used = t + 1;
  }
  for (int t = 0; t < used; ++t)
    if (th[t]) pthread_join(th[t], NULL);
  return 0;
}

int tpo_synth_uniform_bf16(uint64_t key, int64_t count, uint16_t* out, int nthreads) {
  job_t j = {0, key, 0, 0, 0.0, 0.0f, NULL, out};
  return run(j, count, nthreads);
}

int tpo_synth_normal_bf16(uint64_t key, int64_t count, double sigma, uint16_t* out, int nthreads) {
  job_t j = {1, key, 0, 0, sigma, 0.0f, NULL, out};
  return run(j, count, nthreads);
}

int tpo_synth_normal_f32(uint64_t key, int64_t count, double sigma, float* out, int nthreads) {
  job_t j = {2, key, 0, 0, sigma, 0.0f, NULL, out};
  return run(j, count, nthreads);
}

int tpo_synth_quant_e4m3(const float* in, int64_t count, float scale, uint8_t* out, int nthreads) {
  job_t j = {3, 0, 0, 0, 0.0, scale, in, out};
  return run(j, count, nthreads);
}
