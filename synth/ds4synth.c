/*
 * ds4synth.c -- seeded synthetic inputs for the routed MoE FFN of a
 * DeepSeek-V4-Flash-shaped layer.
 *
 * This module only draws random numbers and lays them out as the canonical
 * weight formats' bytes. It holds none of the layer's arithmetic (no
 * dequantisation, no dot products, no routing). Both the CPU oracle and the
 * CUDA library consume what it writes; neither is imported here.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014). Every output block is a pure function of
 * (key, block index), so any slice can be regenerated independently and the
 * work splits across threads without changing a byte.
 *
 * Weight recipes follow the workload descriptions of the DwarfStar MoE
 * layer (routed 2-bit superblocks, Q8_0 shared expert and router):
 *   Q2S  : q uniform in {0..3}, 4-bit scale and 4-bit min uniform,
 *          d and dmin = fp16(|N(0, dsig)|).
 *   Q8_0 : w ~ N(0, sigma) per element; d = fp16(max|w| / 127);
 *          q = clamp(round_half_away(w / d), -127, 127).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* One SplitMix64 step. */
static inline uint64_t sm_next(uint64_t *s) {
  *s += GOLDEN;
  return mix64(*s);
}

/* Stream state for block `idx` of the tensor identified by `key`. */
static inline uint64_t stream_for(uint64_t key, uint64_t idx) {
  return mix64(key ^ mix64(idx * GOLDEN + 0x632BE59BD9B4E019ull));
}

uint64_t ds4s_key(uint64_t seed, uint32_t layer, uint32_t tensor) {
  uint64_t s = mix64(seed + GOLDEN);
  s = mix64(s ^ ((uint64_t)layer << 32 | tensor));
  return s;
}

/* Uniform double in (0, 1]. */
static inline double u01_open0(uint64_t u) {
  return ((double)(u >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}
/* Uniform double in [0, 1). */
static inline double u01(uint64_t u) {
  return (double)(u >> 11) * (1.0 / 9007199254740992.0);
}

/* Two independent N(0,1) draws by the Box-Muller transform. */
static inline void normal2(uint64_t *s, double *a, double *b) {
  double u1 = u01_open0(sm_next(s));
  double u2 = u01(sm_next(s));
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925 * u2;
  *a = r * cos(t);
  *b = r * sin(t);
}

static inline uint16_t to_half(float f) {
  _Float16 h = (_Float16)f; /* IEEE round-to-nearest-even */
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}
static inline float from_half(uint16_t b) {
  _Float16 h;
  memcpy(&h, &b, 2);
  return (float)h;
}

/* ---------------------------------------------------------------------- */
/* A tiny parallel-for over [0, n) in contiguous slices.                   */

typedef void (*range_fn)(int64_t lo, int64_t hi, void *ctx);
typedef struct {
  range_fn fn;
  void *ctx;
  int64_t lo, hi;
} slice_t;

static void *slice_run(void *p) {
  slice_t *s = (slice_t *)p;
  s->fn(s->lo, s->hi, s->ctx);
  return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx) {
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if (n < 4096 || nthreads == 1) {
    fn(0, n, ctx);
    return;
  }
  pthread_t th[256];
  slice_t sl[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  int used = 0;
  for (int t = 0; t < nthreads; t++) {
    int64_t lo = (int64_t)t * per, hi = lo + per;
    if (lo >= n) break;
    if (hi > n) hi = n;
    sl[t] = (slice_t){fn, ctx, lo, hi};
    if (pthread_create(&th[t], NULL, slice_run, &sl[t]) != 0) {
      slice_run(&sl[t]);
      th[t] = 0;
    }
    used = t + 1;
  }
  for (int t = 0; t < used; t++)
    if (th[t]) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------------- */
/* 2-bit superblock (84 bytes): sm[16] | qs[64] | fp16 d | fp16 dmin.       */

typedef struct {
  uint8_t *out;
  int64_t first;
  uint64_t key;
  float dsig;
} q2s_ctx;

static void q2s_range(int64_t lo, int64_t hi, void *p) {
  q2s_ctx *c = (q2s_ctx *)p;
  for (int64_t i = lo; i < hi; i++) {
    uint64_t s = stream_for(c->key, (uint64_t)(c->first + i));
    uint8_t *b = c->out + i * 84;
    for (int w = 0; w < 10; w++) { /* 80 random bytes: sm[16] + qs[64] */
      uint64_t r = sm_next(&s);
      memcpy(b + 8 * w, &r, 8);
    }
    double n0, n1;
    normal2(&s, &n0, &n1);
    uint16_t d = to_half((float)fabs(n0 * c->dsig));
    uint16_t m = to_half((float)fabs(n1 * c->dsig));
    memcpy(b + 80, &d, 2);
    memcpy(b + 82, &m, 2);
  }
}

/* Superblocks first .. first+n-1 of the tensor `key`, written to out[0..n). */
void ds4s_q2s(uint8_t *out, int64_t first, int64_t n_superblocks, uint64_t key, float dsig,
              int nthreads) {
  q2s_ctx c = {out, first, key, dsig};
  parallel_for(n_superblocks, nthreads, q2s_range, &c);
}

/* ---------------------------------------------------------------------- */
/* 4-bit superblock (148 bytes): sm[16] | qs[128] | fp16 d | fp16 dmin.     */

static void q4s_range(int64_t lo, int64_t hi, void *p) {
  q2s_ctx *c = (q2s_ctx *)p;
  for (int64_t i = lo; i < hi; i++) {
    uint64_t s = stream_for(c->key, (uint64_t)(c->first + i));
    uint8_t *b = c->out + i * 148;
    for (int w = 0; w < 18; w++) { /* 144 random bytes: sm[16] + qs[128] */
      uint64_t r = sm_next(&s);
      memcpy(b + 8 * w, &r, 8);
    }
    double n0, n1;
    normal2(&s, &n0, &n1);
    uint16_t d = to_half((float)fabs(n0 * c->dsig));
    uint16_t m = to_half((float)fabs(n1 * c->dsig));
    memcpy(b + 144, &d, 2);
    memcpy(b + 146, &m, 2);
  }
}

void ds4s_q4s(uint8_t *out, int64_t first, int64_t n_superblocks, uint64_t key, float dsig,
              int nthreads) {
  q2s_ctx c = {out, first, key, dsig};
  parallel_for(n_superblocks, nthreads, q4s_range, &c);
}

/* ---------------------------------------------------------------------- */
/* Q8_0 block (34 bytes): fp16 d | int8 q[32].                              */

typedef struct {
  uint8_t *out;
  int64_t first;
  uint64_t key;
  float sigma;
} q8_ctx;

static void q8_range(int64_t lo, int64_t hi, void *p) {
  q8_ctx *c = (q8_ctx *)p;
  for (int64_t i = lo; i < hi; i++) {
    uint64_t s = stream_for(c->key, (uint64_t)(c->first + i));
    float w[32];
    for (int j = 0; j < 32; j += 2) {
      double a, b;
      normal2(&s, &a, &b);
      w[j] = (float)(a * c->sigma);
      w[j + 1] = (float)(b * c->sigma);
    }
    float amax = 0.f;
    for (int j = 0; j < 32; j++) {
      float a = fabsf(w[j]);
      if (a > amax) amax = a;
    }
    uint16_t dh = to_half(amax / 127.0f);
    float d = from_half(dh);
    uint8_t *b = c->out + i * 34;
    memcpy(b, &dh, 2);
    for (int j = 0; j < 32; j++) {
      int q = 0;
      if (d > 0.f) {
        float r = roundf(w[j] / d);
        q = r > 127.f ? 127 : (r < -127.f ? -127 : (int)r);
      }
      b[2 + j] = (uint8_t)(int8_t)q;
    }
  }
}

/* Blocks first .. first+n-1 of the tensor `key`, written to out[0..n). */
void ds4s_q8(uint8_t *out, int64_t first, int64_t n_blocks, uint64_t key, float sigma,
             int nthreads) {
  q8_ctx c = {out, first, key, sigma};
  parallel_for(n_blocks, nthreads, q8_range, &c);
}

/* ---------------------------------------------------------------------- */
/* Plain float tensors.                                                    */

typedef struct {
  float *out;
  int64_t n;
  uint64_t key;
  float a, b;
} f32_ctx;

/* Elements 2j and 2j+1 come from stream j. */
static void normal_range(int64_t lo, int64_t hi, void *p) {
  f32_ctx *c = (f32_ctx *)p;
  for (int64_t j = lo; j < hi; j++) {
    uint64_t s = stream_for(c->key, (uint64_t)j);
    double x, y;
    normal2(&s, &x, &y);
    int64_t i = 2 * j;
    c->out[i] = (float)(x * c->a) + c->b;
    if (i + 1 < c->n) c->out[i + 1] = (float)(y * c->a) + c->b;
  }
}

/* out[i] = N(0,1) * sigma + mean. */
void ds4s_normal_f32(float *out, int64_t n, uint64_t key, float sigma, float mean, int nthreads) {
  f32_ctx c = {out, n, key, sigma, mean};
  parallel_for((n + 1) / 2, nthreads, normal_range, &c);
}

static void uniform_range(int64_t lo, int64_t hi, void *p) {
  f32_ctx *c = (f32_ctx *)p;
  for (int64_t i = lo; i < hi; i++) {
    uint64_t s = stream_for(c->key, (uint64_t)i);
    double u = u01(sm_next(&s));
    c->out[i] = (float)(c->a + (c->b - c->a) * u);
  }
}

/* out[i] = U[lo, hi). */
void ds4s_uniform_f32(float *out, int64_t n, uint64_t key, float lo, float hi, int nthreads) {
  f32_ctx c = {out, n, key, lo, hi};
  parallel_for(n, nthreads, uniform_range, &c);
}

/* ---------------------------------------------------------------------- */
/* Integer tensors.                                                        */

/* Uniform integer in [0, n) by Lemire's multiply-shift (bias < 2^-32 n). */
static inline uint32_t below(uint64_t *s, uint32_t n) {
  return (uint32_t)(((sm_next(s) >> 32) * (uint64_t)n) >> 32);
}

/* Token ids uniform over [0, vocab). */
void ds4s_token_ids(int32_t *out, int64_t n, int32_t vocab, uint64_t key) {
  for (int64_t i = 0; i < n; i++) {
    uint64_t s = stream_for(key, (uint64_t)i);
    out[i] = (int32_t)below(&s, (uint32_t)vocab);
  }
}

/* Row v: k distinct values from [0, E) by a partial Fisher-Yates shuffle.
 * The drawn order is the stored order. */
typedef struct {
  int32_t *out;
  int32_t E, k;
  uint64_t key;
} hash_ctx;

static void hash_range(int64_t lo, int64_t hi, void *p) {
  hash_ctx *c = (hash_ctx *)p;
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)c->E);
  for (int64_t v = lo; v < hi; v++) {
    uint64_t s = stream_for(c->key, (uint64_t)v);
    for (int32_t e = 0; e < c->E; e++) perm[e] = e;
    for (int32_t j = 0; j < c->k; j++) {
      int32_t r = j + (int32_t)below(&s, (uint32_t)(c->E - j));
      int32_t t = perm[j];
      perm[j] = perm[r];
      perm[r] = t;
      c->out[v * c->k + j] = perm[j];
    }
  }
  free(perm);
}

void ds4s_hash_table(int32_t *out, int32_t vocab, int32_t E, int32_t k, uint64_t key, int nthreads) {
  hash_ctx c = {out, E, k, key};
  parallel_for(vocab, nthreads, hash_range, &c);
}

/* A uniformly random permutation of [0, n). */
void ds4s_permutation(int32_t *out, int32_t n, uint64_t key) {
  uint64_t s = stream_for(key, 0);
  for (int32_t i = 0; i < n; i++) out[i] = i;
  for (int32_t i = n - 1; i > 0; i--) {
    int32_t r = (int32_t)below(&s, (uint32_t)(i + 1));
    int32_t t = out[i];
    out[i] = out[r];
    out[r] = t;
  }
}
