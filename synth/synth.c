/*
 * Seeded synthetic inputs for the layer-staged decoder: weights and token ids.
 *
 * This module is shared by the CPU oracle and the CUDA path as *data*, never as
 * code of the decode step: it draws numbers and encodes them (bf16, int8 with a
 * per-row scale) and holds none of the step's arithmetic (no norm, no GEMV, no
 * attention).
 *
 * Generator (counter based, so any element can be drawn independently and the
 * fill is parallel and order free):
 *   key(seed, stream)  = mix64(seed * 0xD1342543DE82EF95 + mix64(stream))
 *   u64(seed, stream, i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the output function of SplitMix64 (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).
 * Normal draws use the Box-Muller transform in double: pair j of a stream takes
 * u64(2j) and u64(2j+1); element 2j is r*cos(2*pi*u2), element 2j+1 is
 * r*sin(2*pi*u2), r = sqrt(-2 ln u1), u1 in (0, 1], u2 in [0, 1).
 * A weight is w = (float)(stddev * z); its bf16 encoding rounds that float to
 * nearest, ties to even.
 * Symmetric int8 row quantisation of the float draws: s_r = max_k |w_rk| / 127
 * (fp32 division), q = clamp(nearbyint(w / s_r), -127, 127) (fp32 division,
 * ties to even); an all-zero row gets s_r = 0 and q = 0.
 * Token ids: floor(u64 * V / 2^64), i.e. the high word of a 64x64 product.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0xD1342543DE82EF95ull + mix64(stream));
}

static inline uint64_t draw_u64(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
}

/* Element i of the standard-normal stream with key `key`. */
static inline double draw_normal(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  uint64_t a = draw_u64(key, 2 * j), b = draw_u64(key, 2 * j + 1);
  double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
  double u2 = (double)(b >> 11) * 0x1.0p-53;         /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ---- a tiny static-partition parallel for (pthreads) ---- */
typedef void (*range_fn)(void* ctx, uint64_t lo, uint64_t hi);
typedef struct { range_fn fn; void* ctx; uint64_t lo, hi; } job_t;
static void* job_main(void* p) { job_t* j = (job_t*)p; j->fn(j->ctx, j->lo, j->hi); return NULL; }

static int g_threads = 0;
void synth_set_threads(int n) { g_threads = n; }
static int n_threads(void) {
  if (g_threads > 0) return g_threads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n < 1 ? 1 : (n > 64 ? 64 : (int)n);
}

static void par_range(uint64_t n, uint64_t grain, range_fn fn, void* ctx) {
  int t = n_threads();
  if ((uint64_t)t * grain > n) t = (int)(n / grain);
  if (t <= 1) { fn(ctx, 0, n); return; }
  pthread_t th[64];
  job_t jobs[64];
  for (int k = 0; k < t; ++k) {
    jobs[k].fn = fn; jobs[k].ctx = ctx;
    jobs[k].lo = n * (uint64_t)k / (uint64_t)t;
    jobs[k].hi = n * (uint64_t)(k + 1) / (uint64_t)t;
  }
  int started = 0;
  for (int k = 1; k < t; ++k) {
    if (pthread_create(&th[k], NULL, job_main, &jobs[k]) != 0) { job_main(&jobs[k]); th[k] = 0; continue; }
    ++started;
  }
  job_main(&jobs[0]);
  for (int k = 1; k < t; ++k) if (th[k]) pthread_join(th[k], NULL);
  (void)started;
}

/* ---- normal draws ---- */
typedef struct { uint64_t key; double stddev; void* out; } normal_ctx;

static void fill_bf16(void* c, uint64_t lo, uint64_t hi) {
  normal_ctx* x = (normal_ctx*)c;
  uint16_t* o = (uint16_t*)x->out;
  for (uint64_t i = lo; i < hi; ++i) o[i] = f32_to_bf16_rne((float)(x->stddev * draw_normal(x->key, i)));
}
static void fill_f32(void* c, uint64_t lo, uint64_t hi) {
  normal_ctx* x = (normal_ctx*)c;
  float* o = (float*)x->out;
  for (uint64_t i = lo; i < hi; ++i) o[i] = (float)(x->stddev * draw_normal(x->key, i));
}

/* bf16 weights: out[i] = bf16_rne((float)(stddev * N_i)), i in [0, n). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, double stddev, uint16_t* out, uint64_t n) {
  normal_ctx c = {stream_key(seed, stream), stddev, out};
  par_range(n, 1u << 16, fill_bf16, &c);
}

/* fp32 values: out[i] = (float)(mean + stddev * N_i). */
typedef struct { uint64_t key; double mean, stddev; float* out; } affine_ctx;
static void fill_affine(void* c, uint64_t lo, uint64_t hi) {
  affine_ctx* x = (affine_ctx*)c;
  for (uint64_t i = lo; i < hi; ++i) x->out[i] = (float)(x->mean + x->stddev * draw_normal(x->key, i));
}
void synth_normal_f32(uint64_t seed, uint64_t stream, double mean, double stddev, float* out, uint64_t n) {
  affine_ctx c = {stream_key(seed, stream), mean, stddev, out};
  par_range(n, 1u << 16, fill_affine, &c);
}

/* int8 rows: the float draws of (seed, stream) quantised per row (see header). */
typedef struct { uint64_t key; double stddev; uint64_t cols; int8_t* q; float* s; } q8_ctx;
static void fill_q8(void* c, uint64_t lo, uint64_t hi) {
  q8_ctx* x = (q8_ctx*)c;
  float* row = (float*)malloc(sizeof(float) * x->cols);
  for (uint64_t r = lo; r < hi; ++r) {
    float amax = 0.0f;
    for (uint64_t k = 0; k < x->cols; ++k) {
      row[k] = (float)(x->stddev * draw_normal(x->key, r * x->cols + k));
      float a = fabsf(row[k]);
      if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    x->s[r] = s;
    int8_t* q = x->q + r * x->cols;
    for (uint64_t k = 0; k < x->cols; ++k) {
      float v = (s > 0.0f) ? nearbyintf(row[k] / s) : 0.0f;
      if (v > 127.0f) v = 127.0f;
      if (v < -127.0f) v = -127.0f;
      q[k] = (int8_t)v;
    }
  }
  free(row);
}
void synth_normal_q8_rows(uint64_t seed, uint64_t stream, double stddev, uint64_t rows, uint64_t cols,
                          int8_t* q, float* s) {
  q8_ctx c = {stream_key(seed, stream), stddev, cols, q, s};
  par_range(rows, 16, fill_q8, &c);
}

/* Token ids uniform in [0, vocab). */
void synth_tokens(uint64_t seed, uint64_t stream, uint32_t vocab, int32_t* out, uint64_t n) {
  uint64_t key = stream_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) {
    unsigned __int128 p = (unsigned __int128)draw_u64(key, i) * (unsigned __int128)vocab;
    out[i] = (int32_t)(uint64_t)(p >> 64);
  }
}

/* Uniform bf16 values in [-a, a): used only to fill caches for timing. */
typedef struct { uint64_t key; double a; uint16_t* out; } unif_ctx;
static void fill_unif(void* c, uint64_t lo, uint64_t hi) {
  unif_ctx* x = (unif_ctx*)c;
  for (uint64_t i = lo; i < hi; ++i) {
    double u = (double)(draw_u64(x->key, i) >> 11) * 0x1.0p-53;
    x->out[i] = f32_to_bf16_rne((float)(x->a * (2.0 * u - 1.0)));
  }
}
void synth_uniform_bf16(uint64_t seed, uint64_t stream, double a, uint16_t* out, uint64_t n) {
  unif_ctx c = {stream_key(seed, stream), a, out};
  par_range(n, 1u << 16, fill_unif, &c);
}
