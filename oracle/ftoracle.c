/*
 * ORACLE -- test infrastructure only.  A plain, slow, fp64 CPU statement of
 * what one MoE-layer step of the FreeToken expert cache computes.  It shares
 * no code, header or constant with the CUDA library; only tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.
 *
 * Source for the method: "FreeToken: Efficient Edge-Native MoE Serving with
 * Bandwidth-Adaptive Execution", as summarised on theainews.cc
 * (2026-08-22-freetoken-edge-moe), cited below by section:
 *   [Why]      为什么个人跑 MoE 这么难 -- top-k of E routed experts per layer
 *   [Design]   设计：三大机制 intro -- full pool in host memory, one cache of
 *              leftover VRAM shared by all MoE layers
 *   [D1-Pre]   设计 1 带宽自适应执行, Prefill bullet -- full-layer double buffer
 *   [D1-Dec]   设计 1, Decode bullet -- q* ~ m*BP/BH split, CPU experts do not
 *              change residency, exact merge of CPU and GPU partial sums
 *   [D2-LRU]   设计 2 语义感知缓存, expert-locality bullet -- shared LRU cache
 *   [Impl-1]   实现要点, first bullet -- one control kernel: dedup, classify
 *              against the residency table, fill count, K-LRU victims in one
 *              scan, logical-to-slot route rewrite
 *   [Related]  与相关工作 -- routing stays exact and unmodified
 * Where the page is silent the reading taken is stated at the function.
 *
 * Parity pins: every function here is checked in tests/ against brute force
 * on tiny inputs, closed forms, invariants or published tables (OCP MX v1.0
 * for MXFP4); none is pinned by a number printed on the page, which reports
 * only end-to-end figures on real models.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EARG -1
#define OR_ENAN -2
#define OR_ERANGE -3
#define OR_EWRAP -4

/* Threads the expert evaluations may use (1 without OpenMP). */
int or_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ routing */

/* order: larger logit first; equal logits -> lower expert index first */
static int before(const float* row, int a, int b) {
  if (row[a] > row[b]) return 1;
  if (row[a] < row[b]) return 0;
  return a < b;
}

/*
 * Top-k routing [Why], [Related]: ids = the k experts with the largest
 * logits, listed in descending logit order, ties to the lower index (a full
 * insertion sort of all E experts).  Weights (the page names none; the
 * Qwen-style reading): softmax over all E in fp64, then renormalised over
 * the k chosen so that they sum to one.
 */
int or_route(const float* logits, int T, int E, int k, int32_t* ids, double* w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return OR_EARG;
  int* order = (int*)malloc(sizeof(int) * (size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  int rc = OR_OK;
  for (int t = 0; t < T; ++t) {
    const float* row = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      if (isnan(row[e])) rc = OR_ENAN;
      order[e] = e;
    }
    if (rc != OR_OK) break;
    for (int i = 1; i < E; ++i) {
      int v = order[i], j = i;
      while (j > 0 && before(row, v, order[j - 1])) {
        order[j] = order[j - 1];
        --j;
      }
      order[j] = v;
    }
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e) mx = fmax(mx, (double)row[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
      p[e] = exp((double)row[e] - mx);
      z += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= z;
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += p[order[j]];
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = order[j];
      w[(size_t)t * k + j] = p[order[j]] / s;
    }
  }
  free(order);
  free(p);
  return rc;
}

/* ------------------------------------------------------------ cache control */

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

typedef struct {
  uint32_t last_use;
  int32_t slot;
} lru_key;

static int cmp_lru(const void* a, const void* b) {
  const lru_key* x = (const lru_key*)a;
  const lru_key* y = (const lru_key*)b;
  if (x->last_use != y->last_use) return x->last_use < y->last_use ? -1 : 1;
  return (x->slot > y->slot) - (x->slot < y->slot);
}

/*
 * One layer step of the shared LRU expert cache ([Design], [D1-Dec],
 * [D2-LRU], [Impl-1]).  State: slot_of[E_tot] (expert -> slot or -1),
 * expert_of[S] (slot -> global expert or -1), last_use[S] (0 = never used),
 * and the step clock *now, advanced once per call (one tick per layer step,
 * since one cache serves every layer).
 *
 * ids are the T*k local expert ids of layer `layer`; global id = layer*E + e.
 *  1. n unique global ids in ascending order.
 *  2. hit if slot_of[u] >= 0; each hit's slot gets last_use = now.
 *  3. m misses; q* = min(m, floor(m*r + 1/2)) with r = r_num/r_den evaluated
 *     exactly: (2*m*r_num + r_den) div (2*r_den).  (The page gives
 *     q* ~ m*BP/BH and says it reaches m as BH approaches BP; the clamp to
 *     [0, m] and the half-up rounding are the reading taken here.)
 *  4. q = min(q*, K_max, #slots with last_use < now); the first q misses in
 *     ascending id are filled, the other m - q run on the CPU and leave the
 *     residency table untouched.
 *  5. victims: slots ordered by (last_use, slot) ascending, restricted to
 *     last_use < now, first q of them; fill i goes to victim i.
 *  6. a victim's old expert loses its slot; the filled expert takes it with
 *     last_use = now.
 *  7. slot_ids[r] = slot_of[global id of route r] (-1 for CPU routes).
 * counts = {n, hits, m, q, m - q}.  evicted[i] = the expert that victim i
 * held before (-1 if empty).
 */
int or_cache_step(int layer, int E, int n_routes, const int32_t* ids, int64_t r_num, int64_t r_den,
                  int K_max, int32_t* slot_of, int E_tot, int32_t* expert_of, uint32_t* last_use, int S,
                  uint32_t* now, int32_t* uniq, int32_t* counts, int32_t* hit_list, int32_t* miss_list,
                  int32_t* fetch, int32_t* victims, int32_t* evicted, int32_t* cpu_list,
                  int32_t* slot_ids, int fill_order) {
  if (E < 1 || layer < 0 || (int64_t)(layer + 1) * E > E_tot || n_routes < 0 || S < 1 || K_max < 0 ||
      r_num < 0 || r_den < 1 || fill_order < 0 || fill_order > 1)
    return OR_EARG;
  for (int r = 0; r < n_routes; ++r)
    if (ids[r] < 0 || ids[r] >= E) return OR_ERANGE;
  if (*now == 0xFFFFFFFFu) return OR_EWRAP;
  uint32_t cur = *now + 1;
  *now = cur;

  /* 1. dedup */
  int32_t* g = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_routes > 0 ? n_routes : 1));
  for (int r = 0; r < n_routes; ++r) g[r] = layer * E + ids[r];
  qsort(g, (size_t)n_routes, sizeof(int32_t), cmp_i32);
  int n = 0;
  for (int r = 0; r < n_routes; ++r)
    if (n == 0 || g[r] != uniq[n - 1]) uniq[n++] = g[r];
  free(g);

  /* 2. classify, touch hits */
  int hits = 0, m = 0;
  for (int i = 0; i < n; ++i) {
    int32_t s = slot_of[uniq[i]];
    if (s >= 0) {
      hit_list[hits++] = uniq[i];
      last_use[s] = cur;
    } else {
      miss_list[m++] = uniq[i];
    }
  }

  /* 3. q* */
  int64_t qstar = (2 * (int64_t)m * r_num + r_den) / (2 * r_den);
  if (qstar > m) qstar = m;

  /* 4. q */
  int avail = 0;
  for (int s = 0; s < S; ++s)
    if (last_use[s] < cur) ++avail;
  int64_t q = qstar;
  if (q > K_max) q = K_max;
  if (q > avail) q = avail;
  if (fill_order == 0 || q == m) {
    /* the first q misses in ascending id */
    for (int i = 0; i < q; ++i) fetch[i] = miss_list[i];
    for (int i = (int)q; i < m; ++i) cpu_list[i - (int)q] = miss_list[i];
  } else {
    /* most-routed first: the q misses chosen by most routes in this step,
       ties to the lower id; both lists stay in ascending id */
    int* nroutes = (int*)calloc((size_t)(m > 0 ? m : 1), sizeof(int));
    char* chosen = (char*)calloc((size_t)(m > 0 ? m : 1), 1);
    for (int i = 0; i < m; ++i)
      for (int r = 0; r < n_routes; ++r)
        if (layer * E + ids[r] == miss_list[i]) ++nroutes[i];
    for (int c = 0; c < q; ++c) {
      int best = -1;
      for (int i = 0; i < m; ++i)
        if (!chosen[i] && (best < 0 || nroutes[i] > nroutes[best])) best = i; /* strict: lower id wins ties */
      chosen[best] = 1;
    }
    int nf = 0, nc = 0;
    for (int i = 0; i < m; ++i) {
      if (chosen[i]) fetch[nf++] = miss_list[i];
      else cpu_list[nc++] = miss_list[i];
    }
    free(nroutes);
    free(chosen);
  }

  /* 5. victims */
  if (q > 0) {
    lru_key* keys = (lru_key*)malloc(sizeof(lru_key) * (size_t)S);
    for (int s = 0; s < S; ++s) {
      keys[s].last_use = last_use[s];
      keys[s].slot = s;
    }
    qsort(keys, (size_t)S, sizeof(lru_key), cmp_lru);
    int c = 0;
    for (int i = 0; i < S && c < q; ++i)
      if (keys[i].last_use < cur) victims[c++] = keys[i].slot;
    free(keys);
  }

  /* 6. table update */
  for (int i = 0; i < q; ++i) {
    int32_t s = victims[i];
    int32_t old = expert_of[s];
    evicted[i] = old;
    if (old >= 0) slot_of[old] = -1;
    slot_of[fetch[i]] = s;
    expert_of[s] = fetch[i];
    last_use[s] = cur;
  }

  /* 7. rewrite */
  for (int r = 0; r < n_routes; ++r) slot_ids[r] = slot_of[layer * E + ids[r]];

  counts[0] = n;
  counts[1] = hits;
  counts[2] = m;
  counts[3] = (int32_t)q;
  counts[4] = m - (int32_t)q;
  return OR_OK;
}

/* ---------------------------------------------------------------- experts */

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* OCP Microscaling Formats (MX) v1.0: e2m1 element = sign bit, 2 exponent
 * bits (bias 1), 1 mantissa bit; e8m0 scale = 2^(E - 127), E = 255 is NaN.
 * Written out from the format definition, not from a table. */
double or_e2m1_value(int code) {
  int sign = (code >> 3) & 1;
  int ex = (code >> 1) & 3;
  int man = code & 1;
  double mag = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
  return sign ? -mag : mag;
}

double or_e8m0_value(int e) { return e == 255 ? NAN : ldexp(1.0, e - 127); }

/* Dequantised element (row, col) of a [rows, cols] MXFP4 matrix: codes are
 * two per byte, element 2i in the low nibble; one scale byte per 32
 * consecutive elements of a row. */
static double mx_elem(const uint8_t* codes, const uint8_t* scales, int cols, int row, int col) {
  size_t idx = (size_t)row * cols + col;
  uint8_t byte = codes[idx / 2];
  int code = (idx & 1) ? (byte >> 4) : (byte & 15);
  return or_e2m1_value(code) * or_e8m0_value(scales[idx / 32]);
}

/* W[row, col] of matrix `which` (0 gate [f,d], 1 up [f,d], 2 down [d,f]) of
 * one expert in the canonical layout:
 *  bf16:  [W_gate | W_up | W_down] row-major,
 *  mxfp4: [codes gate | codes up | codes down | scales gate | up | down]. */
static double weight(const uint8_t* ex, int dtype, int d, int f, int which, int row, int col) {
  size_t df = (size_t)d * f;
  int cols = which == 2 ? f : d;
  if (dtype == 0) {
    const uint16_t* w = (const uint16_t*)ex + (size_t)which * df;
    return bf16_value(w[(size_t)row * cols + col]);
  }
  const uint8_t* codes = ex + (size_t)which * (df / 2);
  const uint8_t* scales = ex + 3 * (df / 2) + (size_t)which * (df / 32);
  return mx_elem(codes, scales, cols, row, col);
}

/*
 * One routed SwiGLU expert, fp64 throughout from the bf16 input x:
 *   y = W_down (silu(W_gate x) * (W_up x)),  silu(z) = z / (1 + e^-z).
 * (The page does not name the activation; SwiGLU is the one of the model
 * families it serves.)
 */
int or_expert_ffn(const uint8_t* ex, int dtype, int d, int f, const uint16_t* x_bf16, double* y) {
  if (d < 1 || f < 1 || (dtype != 0 && dtype != 1)) return OR_EARG;
  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  for (int c = 0; c < d; ++c) x[c] = bf16_value(x_bf16[c]);
  for (int i = 0; i < f; ++i) {
    double gsum = 0.0, usum = 0.0;
    for (int c = 0; c < d; ++c) {
      gsum += weight(ex, dtype, d, f, 0, i, c) * x[c];
      usum += weight(ex, dtype, d, f, 1, i, c) * x[c];
    }
    h[i] = gsum / (1.0 + exp(-gsum)) * usum;
  }
  for (int r = 0; r < d; ++r) {
    double s = 0.0;
    for (int i = 0; i < f; ++i) s += weight(ex, dtype, d, f, 2, r, i) * h[i];
    y[r] = s;
  }
  free(x);
  free(h);
  return OR_OK;
}

/*
 * Routed MoE output of one layer for the selected tokens ([D1-Dec]):
 *   out_full[t] = sum_j w[t,j] * y_{ids[t,j]}(x_t)
 * and, when slot_ids is given, the same sum split by where the route runs:
 * out_gpu over routes with slot_ids >= 0, out_cpu over routes with -1.
 * layer_base points at expert 0 of the layer in the canonical pool.
 * tokens: n_sel token indices (NULL = all T); outputs are [n_sel, d].
 */
int or_moe_forward(const uint8_t* layer_base, uint64_t expert_bytes, int dtype, int d, int f, int T,
                   int k, const int32_t* ids, const double* w, const int32_t* slot_ids,
                   const uint16_t* hidden, const int32_t* tokens, int n_sel, double* out_full,
                   double* out_gpu, double* out_cpu) {
  if (T < 0 || k < 1 || d < 1 || f < 1 || (dtype != 0 && dtype != 1)) return OR_EARG;
  if (tokens == NULL) n_sel = T;
  size_t pairs = (size_t)n_sel * k;
  double* y = (double*)malloc(sizeof(double) * (pairs > 0 ? pairs : 1) * (size_t)d);
#pragma omp parallel for schedule(dynamic, 1)
  for (long p = 0; p < (long)pairs; ++p) {
    int si = (int)(p / k), j = (int)(p % k);
    int t = tokens ? tokens[si] : si;
    int e = ids[(size_t)t * k + j];
    const uint8_t* ex = layer_base + (size_t)e * expert_bytes;
    or_expert_ffn(ex, dtype, d, f, hidden + (size_t)t * d, y + (size_t)p * d);
  }
  for (int si = 0; si < n_sel; ++si) {
    int t = tokens ? tokens[si] : si;
    for (int c = 0; c < d; ++c) {
      double full = 0.0, gpu = 0.0, cpu = 0.0;
      for (int j = 0; j < k; ++j) {
        double v = w[(size_t)t * k + j] * y[((size_t)si * k + j) * d + c];
        full += v;
        if (slot_ids) {
          if (slot_ids[(size_t)t * k + j] >= 0)
            gpu += v;
          else
            cpu += v;
        }
      }
      out_full[(size_t)si * d + c] = full;
      if (out_gpu) out_gpu[(size_t)si * d + c] = gpu;
      if (out_cpu) out_cpu[(size_t)si * d + c] = cpu;
    }
  }
  free(y);
  return OR_OK;
}

/* Dense all-experts MoE: every expert runs on every token and a gate vector
 * g[t, e] (zero off-route) weights it.  Used to pin the routed form. */
int or_dense_moe(const uint8_t* layer_base, uint64_t expert_bytes, int dtype, int d, int f, int T, int E,
                 const double* gates, const uint16_t* hidden, double* out) {
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < d; ++c) out[(size_t)t * d + c] = 0.0;
    for (int e = 0; e < E; ++e) {
      or_expert_ffn(layer_base + (size_t)e * expert_bytes, dtype, d, f, hidden + (size_t)t * d, y);
      for (int c = 0; c < d; ++c) out[(size_t)t * d + c] += gates[(size_t)t * E + e] * y[c];
    }
  }
  free(y);
  return OR_OK;
}

/* ------------------------------------------------- run-time r = BP/BH */

/*
 * [D1-Dec] splits the misses by q* ~ m*BP/BH with BP and BH the bandwidths
 * measured while the system runs.  The page does not say how measurements
 * become r; the reading taken: each measurement window gives at most one
 * sample of each (a value <= 0 = no sample); an estimate starts at its first
 * sample and then moves by est <- est + alpha*(sample - est); once both
 * estimates exist r is BP/BH rounded half up onto the grid 1/r_den, at most
 * r_num_max/r_den, and -1 marks "no r yet".  out[i] is r_num after window i.
 */
int or_adapt_ratio(int n, const double* bp, const double* bh, double alpha, int r_den, int r_num_max, int32_t* out) {
  if (n < 0 || !(alpha > 0.0 && alpha <= 1.0) || r_den < 1 || r_num_max < 0) return OR_EARG;
  double est_p = 0.0, est_h = 0.0;
  int have_p = 0, have_h = 0;
  int32_t r = -1;
  for (int i = 0; i < n; ++i) {
    if (bp[i] > 0.0) {
      est_p = have_p ? alpha * bp[i] + (1.0 - alpha) * est_p : bp[i];
      have_p = 1;
    }
    if (bh[i] > 0.0) {
      est_h = have_h ? alpha * bh[i] + (1.0 - alpha) * est_h : bh[i];
      have_h = 1;
    }
    if (have_p && have_h) {
      double q = floor((double)r_den * est_p / est_h + 0.5);
      r = q >= (double)r_num_max ? r_num_max : (int32_t)q;
    }
    out[i] = r;
  }
  return OR_OK;
}
