/*
 * Seeded synthetic inputs for the MoE expert-cache hot path.
 *
 * This file holds no arithmetic of the method itself: it only draws the
 * expert weights, router weights and hidden-state streams that both the
 * CUDA library and the CPU oracle consume.  Every stream is a pure function
 * of (seed, tensor id, a, b, element index), so any single expert of any
 * layer can be regenerated on its own.
 *
 * Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11), key = (seed, tensor id), counter =
 * (block index lo, block index hi, a, b).  One block yields four 32-bit
 * words.  Normals come from the Box-Muller transform on pairs of words,
 * u = (x + 0.5) / 2^32, in double precision.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void ftsynth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static inline void block_words(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b,
                               uint64_t blk, uint32_t w[4]) {
  uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), a, b};
  uint32_t key[2] = {seed, tensor};
  ftsynth_philox4x32_10(ctr, key, w);
}

static inline double unit_open(uint32_t x) { return ((double)x + 0.5) * (1.0 / 4294967296.0); }
/* single-precision variant used by the normal transform: the top 24 bits,
 * (x >> 8) + 0.5 over 2^24, so the value is exact in float and in (0, 1) */
static inline float unit_open_f(uint32_t x) { return ((float)(x >> 8) + 0.5f) * (1.0f / 16777216.0f); }

/* Normal number `idx` of stream (seed, tensor, a, b): element idx lives in
 * block idx/4; words (0,1) give normals 0,1 and words (2,3) give 2,3. */
static inline void block_normals(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b,
                                 uint64_t blk, double z[4]) {
  uint32_t w[4];
  block_words(seed, tensor, a, b, blk, w);
  for (int p = 0; p < 2; ++p) {
    float r = sqrtf(-2.0f * logf(unit_open_f(w[2 * p])));
    float sn, cs;
    sincosf(6.2831853f * unit_open_f(w[2 * p + 1]), &sn, &cs);
    z[2 * p] = (double)(r * cs);
    z[2 * p + 1] = (double)(r * sn);
  }
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void ftsynth_normal_f64(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t offset,
                        uint64_t n, double stddev, double* out) {
  uint64_t i = 0;
  while (i < n) {
    uint64_t e = offset + i;
    uint64_t blk = e >> 2;
    double z[4];
    block_normals(seed, tensor, a, b, blk, z);
    for (uint64_t j = e & 3; j < 4 && i < n; ++j, ++i) out[i] = stddev * z[j];
  }
}

/* bf16(float(stddev * z)) : rounded to fp32 first, then to bf16, both RNE. */
void ftsynth_normal_bf16(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t offset,
                         uint64_t n, double stddev, uint16_t* out) {
  uint64_t i = 0;
  while (i < n) {
    uint64_t e = offset + i;
    uint64_t blk = e >> 2;
    double z[4];
    block_normals(seed, tensor, a, b, blk, z);
    for (uint64_t j = e & 3; j < 4 && i < n; ++j, ++i) out[i] = f32_to_bf16_rne((float)(stddev * z[j]));
  }
}

/* Uniform bytes: byte idx is byte (idx % 16) of block idx/16, little-endian words. */
void ftsynth_bytes(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t offset,
                   uint64_t n, uint8_t* out) {
  uint64_t i = 0;
  while (i < n) {
    uint64_t e = offset + i;
    uint32_t w[4];
    block_words(seed, tensor, a, b, e >> 4, w);
    for (uint64_t j = e & 15; j < 16 && i < n; ++j, ++i) out[i] = (uint8_t)(w[j >> 2] >> (8 * (j & 3)));
  }
}

/* Scale bytes drawn uniformly from {lo, ..., lo+span-1}: one 32-bit word per
 * byte, mapped by the multiply-shift (x * span) >> 32. */
void ftsynth_scale_bytes(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t offset,
                         uint64_t n, uint32_t lo, uint32_t span, uint8_t* out) {
  uint64_t i = 0;
  while (i < n) {
    uint64_t e = offset + i;
    uint32_t w[4];
    block_words(seed, tensor, a, b, e >> 2, w);
    for (uint64_t j = e & 3; j < 4 && i < n; ++j, ++i)
      out[i] = (uint8_t)(lo + (uint32_t)(((uint64_t)w[j] * span) >> 32));
  }
}

/* AR(1) hidden stream h_0 = eps_0, h_t = rho*h_{t-1} + eps_t (fp64), with
 * eps_t[i] = normal (t*dim + i) of stream (seed, tensor, a, b); emitted as
 * bf16(float(h_t)).  out is [steps, dim]. */
void ftsynth_ar1_bf16(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t steps,
                      uint64_t dim, double rho, uint16_t* out) {
  double* h = (double*)calloc(dim, sizeof(double));
  double* eps = (double*)malloc(dim * sizeof(double));
  for (uint64_t t = 0; t < steps; ++t) {
    ftsynth_normal_f64(seed, tensor, a, b, t * dim, dim, 1.0, eps);
    for (uint64_t i = 0; i < dim; ++i) {
      h[i] = (t == 0 ? 0.0 : rho * h[i]) + eps[i];
      out[t * dim + i] = f32_to_bf16_rne((float)h[i]);
    }
  }
  free(h);
  free(eps);
}

/* ---------------- parallel pool writers ---------------- */

typedef struct {
  uint32_t seed;
  int L, E, d, f, dtype;  /* dtype 0 = bf16, 1 = mxfp4 */
  double stddev;
  uint8_t* pool;
  uint64_t expert_bytes;
  int first_layer;
  int next; /* shared work counter */
  pthread_mutex_t mu;
} pool_job;

static void write_expert(pool_job* j, int l, int e) {
  uint64_t df = (uint64_t)j->d * (uint64_t)j->f;
  uint8_t* base = j->pool + ((uint64_t)l * j->E + e) * j->expert_bytes;
  uint32_t la = (uint32_t)(j->first_layer + l);
  if (j->dtype == 0) {
    uint16_t* w = (uint16_t*)base;
    ftsynth_normal_bf16(j->seed, 1, la, (uint32_t)e, 0, df, j->stddev, w);
    ftsynth_normal_bf16(j->seed, 2, la, (uint32_t)e, 0, df, j->stddev, w + df);
    ftsynth_normal_bf16(j->seed, 3, la, (uint32_t)e, 0, df, j->stddev, w + 2 * df);
  } else {
    uint64_t cb = df / 2, sb = df / 32;
    ftsynth_bytes(j->seed, 7, la, (uint32_t)e, 0, cb, base);
    ftsynth_bytes(j->seed, 8, la, (uint32_t)e, 0, cb, base + cb);
    ftsynth_bytes(j->seed, 9, la, (uint32_t)e, 0, cb, base + 2 * cb);
    ftsynth_scale_bytes(j->seed, 10, la, (uint32_t)e, 0, sb, 119, 3, base + 3 * cb);
    ftsynth_scale_bytes(j->seed, 11, la, (uint32_t)e, 0, sb, 119, 3, base + 3 * cb + sb);
    ftsynth_scale_bytes(j->seed, 12, la, (uint32_t)e, 0, sb, 119, 3, base + 3 * cb + 2 * sb);
  }
}

static void* pool_worker(void* arg) {
  pool_job* j = (pool_job*)arg;
  int total = j->L * j->E;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int it = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (it >= total) break;
    write_expert(j, it / j->E, it % j->E);
  }
  return NULL;
}

/* Write L layers x E experts (layers first_layer .. first_layer+L-1 of the
 * stream) into pool, expert (l, e) at byte offset (l*E + e)*expert_bytes.
 * bf16 expert: [W_gate f x d | W_up f x d | W_down d x f], N(0, stddev).
 * mxfp4 expert: [codes gate | codes up | codes down | scales gate | up | down],
 * codes uniform bytes (so every e2m1 code equally likely), scales uniform in
 * {119, 120, 121}.  Returns 0 on success. */
int ftsynth_fill_pool(uint32_t seed, int first_layer, int L, int E, int d, int f, int dtype,
                      double stddev, uint64_t expert_bytes, uint8_t* pool, int nthreads) {
  pool_job j;
  j.seed = seed; j.L = L; j.E = E; j.d = d; j.f = f; j.dtype = dtype; j.stddev = stddev;
  j.pool = pool; j.expert_bytes = expert_bytes; j.first_layer = first_layer; j.next = 0;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < nthreads; ++i)
    if (pthread_create(&th[started], NULL, pool_worker, &j) == 0) ++started;
  pool_worker(&j);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&j.mu);
  return 0;
}

/* Parallel bf16 normals for large activation tensors: rows [rows, cols] with
 * row r drawn from stream (seed, tensor, a, b) elements r*cols .. */
typedef struct {
  uint32_t seed, tensor, a, b;
  uint64_t rows, cols;
  double stddev;
  uint16_t* out;
  uint64_t next;
  pthread_mutex_t mu;
} rows_job;

static void* rows_worker(void* arg) {
  rows_job* j = (rows_job*)arg;
  const uint64_t chunk = 64;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    uint64_t r0 = j->next;
    j->next += chunk;
    pthread_mutex_unlock(&j->mu);
    if (r0 >= j->rows) break;
    uint64_t r1 = r0 + chunk < j->rows ? r0 + chunk : j->rows;
    ftsynth_normal_bf16(j->seed, j->tensor, j->a, j->b, r0 * j->cols, (r1 - r0) * j->cols, j->stddev,
                        j->out + r0 * j->cols);
  }
  return NULL;
}

int ftsynth_normal_bf16_par(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t rows,
                            uint64_t cols, double stddev, uint16_t* out, int nthreads) {
  rows_job j;
  j.seed = seed; j.tensor = tensor; j.a = a; j.b = b; j.rows = rows; j.cols = cols;
  j.stddev = stddev; j.out = out; j.next = 0;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < nthreads; ++i)
    if (pthread_create(&th[started], NULL, rows_worker, &j) == 0) ++started;
  rows_worker(&j);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&j.mu);
  return 0;
}
