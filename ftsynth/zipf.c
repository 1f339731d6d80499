/*
 * Zipf route streams for the cache-control stress workload.
 *
 * Per layer a fixed random rank permutation of the E experts is drawn
 * (experts sorted by a uniform key, ties impossible in practice and broken
 * by index).  Each token then takes k distinct experts by Gumbel-top-k on
 * score_e = -s*ln(rank_e) + G_e, G_e = -ln(-ln u_e): a Plackett-Luce draw
 * without replacement with weights rank^-s, i.e. Zipf(s).  Uniforms come
 * from the same Philox stream family as synth.c (tensor 15 for the rank
 * keys, tensor 16 for the Gumbel noise).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

void ftsynth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]);

static double unit_word(uint32_t seed, uint32_t tensor, uint32_t a, uint32_t b, uint64_t idx) {
  uint32_t ctr[4] = {(uint32_t)(idx >> 2), (uint32_t)(idx >> 34), a, b};
  uint32_t key[2] = {seed, tensor};
  uint32_t w[4];
  ftsynth_philox4x32_10(ctr, key, w);
  return ((double)w[idx & 3] + 0.5) * (1.0 / 4294967296.0);
}

/* rank_out[e] in 1..E for layer `layer`. */
void ftsynth_zipf_ranks(uint32_t seed, uint32_t layer, int E, int32_t* rank_out) {
  double* key = (double*)malloc(sizeof(double) * E);
  for (int e = 0; e < E; ++e) key[e] = unit_word(seed, 15, layer, 0, (uint64_t)e);
  for (int e = 0; e < E; ++e) {
    int r = 1;
    for (int o = 0; o < E; ++o)
      if (key[o] < key[e] || (key[o] == key[e] && o < e)) ++r;
    rank_out[e] = r;
  }
  free(key);
}

typedef struct {
  uint32_t seed;
  int layer, E, T, k;
  uint64_t step0, nsteps;
  double s;
  const int32_t* rank;
  int32_t* out; /* [nsteps, T, k] */
  uint64_t next;
  pthread_mutex_t mu;
} zjob;

static void one_token(const zjob* j, uint64_t step, int t, int32_t* dst) {
  double best[64];
  int bid[64];
  int k = j->k;
  for (int i = 0; i < k; ++i) { best[i] = -INFINITY; bid[i] = -1; }
  uint64_t base = ((step * (uint64_t)j->T) + (uint64_t)t) * (uint64_t)j->E;
  for (int e = 0; e < j->E; ++e) {
    double u = unit_word(j->seed, 16, (uint32_t)j->layer, 0, base + (uint64_t)e);
    double sc = -j->s * log((double)j->rank[e]) - log(-log(u));
    /* insertion into the running top-k, ordered by score desc then index asc */
    if (sc > best[k - 1] || bid[k - 1] < 0) {
      int p = k - 1;
      while (p > 0 && (sc > best[p - 1] || bid[p - 1] < 0)) {
        best[p] = best[p - 1];
        bid[p] = bid[p - 1];
        --p;
      }
      best[p] = sc;
      bid[p] = e;
    }
  }
  for (int i = 0; i < k; ++i) dst[i] = bid[i];
}

static void* zworker(void* arg) {
  zjob* j = (zjob*)arg;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    uint64_t it = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (it >= j->nsteps) break;
    for (int t = 0; t < j->T; ++t)
      one_token(j, j->step0 + it, t, j->out + (it * (uint64_t)j->T + (uint64_t)t) * (uint64_t)j->k);
  }
  return NULL;
}

/* Routes of steps step0 .. step0+nsteps-1 of one layer: out [nsteps, T, k]. */
int ftsynth_zipf_routes(uint32_t seed, int layer, int E, int T, int k, double s, uint64_t step0,
                        uint64_t nsteps, int32_t* out, int nthreads) {
  if (k < 1 || k > 64 || k > E) return -1;
  int32_t* rank = (int32_t*)malloc(sizeof(int32_t) * E);
  ftsynth_zipf_ranks(seed, (uint32_t)layer, E, rank);
  zjob j;
  j.seed = seed; j.layer = layer; j.E = E; j.T = T; j.k = k; j.step0 = step0; j.nsteps = nsteps;
  j.s = s; j.rank = rank; j.out = out; j.next = 0;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < nthreads; ++i)
    if (pthread_create(&th[started], NULL, zworker, &j) == 0) ++started;
  zworker(&j);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&j.mu);
  free(rank);
  return 0;
}
