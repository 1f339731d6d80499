// The cache-control kernel: one CTA runs the whole per-layer control step.
//
// FreeToken article, section "实现要点" (first bullet): the misses, the number
// of fetches and the evicted slots change every step, and host-driven control
// would cost a synchronisation at every MoE layer; so all routing-dependent
// control runs on the GPU with fixed-shape work buffers and a device-resident
// valid count, and one kernel does dedup, classification against the
// residency table, the fetch count, victim choice and the logical-to-slot
// rewrite.  Victim choice finds the K least-recently-used candidate slots in
// a single pass whatever the miss count.  The fetch count follows the Decode
// bullet of section "设计 1": q* ~ m*BP/BH, CPU-run experts leave residency
// unchanged.
//
// Step (the clock `now` advances once per call; one cache serves all layers):
//  1. count routes per local expert (shared-memory histogram);
//  2. unique experts ascending; hit if slot_of[u] >= 0 (touch: last_use = now);
//  3. q* = min(m, floor(m*r + 1/2)) in exact integer arithmetic,
//     q = min(q*, K_max, #slots with last_use < now);
//  4. the q smallest keys (last_use, slot) among slots with last_use < now:
//     radix select on last_use (8-bit digits, only the bits where the
//     eligible values differ), then the slots below the threshold are ranked
//     and the ones at the threshold taken in slot order;
//  5. fill i -> victim i: evict, install, last_use = now; the rest go to CPU;
//  6. rewrite route ids to slot ids (-1 = CPU);
//  7. group the routes by resident expert for the expert kernel (dispatch).
#include "ft_internal.h"
#include "tma.h"
#include "route_warp.cuh"

namespace ft {
namespace {

constexpr int kMaxWarps = kControlThreads / 32;
constexpr int kControlRoutesSmem = 1024;  // routes kept in shared memory by the fused routing
constexpr int kRankRouteMax = kControlThreads / 2;  // T * E up to which routing ranks every (token, expert) pair
constexpr int kSmallQ = 4;                // up to this many fills, victims by rounds of a block arg-min

struct Smem {
  int ecount[kMaxExperts];   // routes per local expert
  int emap[kMaxExperts];     // slot per local expert after the step (-1 none)
  int gstart[kMaxExperts];   // first group_routes index of the expert's group
  int cursor[kMaxExperts];   // scatter cursor per expert
  int miss_local[kMaxExperts];
  int filled[kMaxExperts];   // 1 if the expert is installed by this step's fill
  int victims[kMaxKmax];
  int eqsel[kMaxKmax];
  unsigned long long cand[kMaxKmax];  // (last_use << 32 | slot) below the threshold
  unsigned hist[256];
  int wsum[kMaxWarps];
  unsigned wmin[kMaxWarps], wmax[kMaxWarps];
  int sc[16];  // scalars
  unsigned long long wkey[kMaxWarps];  // per-warp minimum keys (small-q victim rounds)
  int rids[kControlRoutesSmem];        // the step's routes when routed in this kernel
  float sel[kControlRoutesSmem];       // their logits, in rank order per token
  float lg[kRankRouteMax];             // the step's logits (routing by rank, 2 T E <= threads)
};

// Exclusive block scan (NT threads); total returned through *total.
template <int NT>
__device__ __forceinline__ int block_scan(int v, int* wsum, int* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < NW ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) wsum[lane] = s;
  }
  __syncthreads();
  int base = wid ? wsum[wid - 1] : 0;
  *total = wsum[NW - 1];
  __syncthreads();
  return base + x - v;
}

// RP > 0: route the step's tokens first (one warp per token, RP logits per
// lane); RP = 0: the routes are given.
// NT threads (a multiple of 32, >= E and >= 256).
template <int RP, int NT>
__global__ void __launch_bounds__(NT, 1) control_kernel(ControlArgs a) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(16) unsigned char dyn[];
  Smem& sm = *reinterpret_cast<Smem*>(dyn);
  unsigned* lu = reinterpret_cast<unsigned*>(dyn + sizeof(Smem));  // [S] last_use copy
  const int tid = threadIdx.x;
  const int E = a.E, S = a.S;
  const int base_id = a.layer * E;


  // routes: read from shared memory when this kernel routed them
  const bool rids_smem = RP > 0 && a.n_routes <= kControlRoutesSmem;
  const int32_t* rids = rids_smem ? sm.rids : a.ids;
  if constexpr (RP > 0) {
    const int TE = a.T * E, k = a.k;
    if (rids_smem && 2 * TE <= NT) {
      // 0. routing by rank (few tokens: at least two threads per (token, expert)
      //    pair): expert e of token t is chosen at position
      //    rank(e) = #{e' : l[e'] > l[e], or l[e'] == l[e] and e' < e} if that is < k
      //    (the same order as k rounds of arg-max: larger logit first, ties to
      //    the lower index); P threads share the count of one (t, e) pair.  More
      //    tokens take the warp-per-token path below, which runs them in parallel.
      bool nan_seen = false;
      for (int i = tid; i < TE; i += NT) {
        float x = a.logits[i];
        if (isnan(x)) {
          nan_seen = true;
          x = -INFINITY;
        }
        sm.lg[i] = x;
      }
      if (__syncthreads_or(nan_seen) && tid == 0) atomicOr(a.status, FT_ST_NAN);
      int P = NT / TE;
      P = P >= 8 ? 8 : P >= 4 ? 4 : P >= 2 ? 2 : 1;
      const int part = tid % P;
      for (int pair = tid / P; pair < ((TE + NT / P - 1) / (NT / P)) * (NT / P); pair += NT / P) {
        const bool live = pair < TE;
        const int t = live ? pair / E : 0, e = live ? pair - t * E : 0;
        const float v = live ? sm.lg[pair] : 0.f;
        const float* row = sm.lg + t * E;
        int cnt = 0;
        if (live)
          for (int j = part; j < E; j += P) {
            const float u = row[j];
            cnt += (u > v) || (u == v && j < e);
          }
        for (int o = P >> 1; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        if (live && part == 0 && cnt < k) {
          sm.rids[t * k + cnt] = e;
          sm.sel[t * k + cnt] = v;
        }
      }
      __syncthreads();
      // the routes and weights go to the layer's step buffers, which the
      // previous kernel may still read (a one-layer model's last merge)
      pdl_wait();
      // weights: softmax over the chosen logits (exp(l_j - l_top) / sum), a warp per token
      const int lane = tid & 31;
      for (int t = tid >> 5; t < a.T; t += NW) {
        const float my_val = lane < k ? sm.sel[t * k + lane] : 0.f;
        const float top = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = lane < k ? expf(my_val - top) : 0.f;
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane < k) {
          a.ids_out[(size_t)t * k + lane] = sm.rids[t * k + lane];
          a.w_out[(size_t)t * k + lane] = ex / sum;
        }
      }
    } else {
      // 0. routing, a warp per token, straight into the step buffers (so after
      // the previous kernel); the __syncthreads below makes the routes visible
      pdl_wait();
      for (int t = tid >> 5; t < a.T; t += NW)
        route_token<RP>(a.logits + (size_t)t * E, E, k, a.ids_out + (size_t)t * k, a.w_out + (size_t)t * k, a.status,
                        nullptr, rids_smem ? sm.rids + (size_t)t * k : nullptr);
    }
  }

  // The routing above reads only the logits, so it may run while the previous
  // kernel (the last layer's merge) finishes; its results and the cache table
  // are written only after that kernel has completed.
  pdl_wait();
  const int slot_pre = tid < E ? a.slot_of[base_id + tid] : -1;  // this layer's residency of every expert
  const long long r_num = a.ratio[0], r_den = a.ratio[1];
  const unsigned now0 = *a.now;
  const bool wrap = now0 == 0xFFFFFFFFu;
  const unsigned now = now0 + 1u;

  for (int e = tid; e < E; e += NT) {
    sm.ecount[e] = 0;
    sm.emap[e] = -1;
    sm.cursor[e] = 0;
    sm.filled[e] = 0;
  }
  for (int s = tid; s < S; s += NT) lu[s] = a.last_use[s];
  __syncthreads();

  // 1. count routes
  bool bad = false;
  for (int r = tid; r < a.n_routes; r += NT) {
    int e = rids[r];
    if ((unsigned)e >= (unsigned)E)
      bad = true;
    else if (!wrap)
      atomicAdd(&sm.ecount[e], 1);
  }
  if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, FT_ST_ROUTE_RANGE);
  if (wrap) {
    // The clock cannot advance: leave the table alone and send every route to the CPU.
    if (tid == 0) atomicOr(a.status, FT_ST_CLOCK_WRAP);
    for (int r = tid; r < a.n_routes; r += NT) a.slot_ids[r] = -1;
    if (tid < kCountsLen) a.counts[tid] = 0;
    if (tid == 0) a.group_off[0] = 0;
    return;
  }

  // 2. dedup + classify (E <= NT: one expert per thread)
  const int e = tid;
  const bool present = e < E && sm.ecount[e] > 0;
  int slot = -1;
  if (present) slot = slot_pre;
  const bool hit = present && slot >= 0;
  int tot;
  int ex = block_scan<NT>(present ? (hit ? 1 : 0x10000) : 0, sm.wsum, &tot);
  const int hits = tot & 0xFFFF, m = tot >> 16, n = hits + m;
  const int hpos = ex & 0xFFFF, mpos = ex >> 16;
  if (present) a.uniq[hpos + mpos] = base_id + e;
  if (hit) {
    if ((unsigned)slot >= (unsigned)S) {
      atomicOr(a.status, FT_ST_BAD_SLOT);
    } else {
      a.hit_list[hpos] = base_id + e;
      lu[slot] = now;
      a.last_use[slot] = now;
      sm.emap[e] = slot;
    }
  } else if (present) {
    sm.miss_local[mpos] = e;
  }
  __syncthreads();

  // 3. q*, q.  Each thread owns the contiguous slot range [s0, s1).
  const int per = (S + NT - 1) / NT;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int my_elig = 0;
  unsigned my_min = 0xFFFFFFFFu, my_max = 0;
  for (int s = s0; s < s1; ++s) {
    unsigned v = lu[s];
    if (v < now) {
      ++my_elig;
      my_min = min(my_min, v);
      my_max = max(my_max, v);
    }
  }
  int avail;
  (void)block_scan<NT>(my_elig, sm.wsum, &avail);
  long long qstar = (2LL * m * r_num + r_den) / (2LL * r_den);
  if (qstar > m) qstar = m;
  int q = (int)qstar;
  if (q > a.K_max) q = a.K_max;
  if (q > avail) q = avail;

  // 3b. most-routed first: when only q < m misses are filled, reorder the miss
  //     list so the q with the most routes in the step (ties: lower id) come
  //     first, each part still in ascending id; steps 5+ take the first q.
  if (a.fill_order == FT_FILL_ORDER_MOST_ROUTED && q > 0 && q < m) {
    const bool is_miss = present && !hit;
    int rank = 0;
    if (is_miss) {
      const int c = sm.ecount[e];
      for (int i = 0; i < m; ++i) {
        const int e2 = sm.miss_local[i], c2 = sm.ecount[e2];
        rank += (c2 > c) || (c2 == c && e2 < e);
      }
    }
    const bool chosen = is_miss && rank < q;
    int n_chosen;
    const int cpos = block_scan<NT>(chosen ? 1 : 0, sm.wsum, &n_chosen);  // every rank is read before this returns
    if (is_miss) sm.miss_local[chosen ? cpos : q + (mpos - cpos)] = e;
    __syncthreads();
  }

  // 4. victims: the q smallest (last_use, slot) among eligible slots
  if (q > 0 && q <= kSmallQ) {
    // few fills: q rounds of a block-wide arg-min over the keys; a chosen slot
    // leaves the eligible set by taking the value `now` in the local copy
    const int lane = tid & 31, wid = tid >> 5;
    for (int i = 0; i < q; ++i) {
      unsigned long long best = ~0ull;
      for (int s = s0; s < s1; ++s) {
        const unsigned v = lu[s];
        const unsigned long long key = ((unsigned long long)v << 32) | (unsigned)s;
        if (v < now && key < best) best = key;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other < best ? other : best;
      }
      if (lane == 0) sm.wkey[wid] = best;
      __syncthreads();
      if (wid == 0) {
        unsigned long long b = lane < NW ? sm.wkey[lane] : ~0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, b, o);
          b = other < b ? other : b;
        }
        if (lane == 0) {
          const int vs = (int)(b & 0xFFFFFFFFu);
          sm.victims[i] = vs;
          lu[vs] = now;
        }
      }
      __syncthreads();
    }
  } else if (q > 0) {
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      my_min = min(my_min, __shfl_xor_sync(0xffffffffu, my_min, o));
      my_max = max(my_max, __shfl_xor_sync(0xffffffffu, my_max, o));
    }
    if (lane == 0) {
      sm.wmin[wid] = my_min;
      sm.wmax[wid] = my_max;
    }
    __syncthreads();
    if (wid == 0) {
      // a launch of NW < 32 warps writes only the first NW entries
      unsigned mn = lane < NW ? sm.wmin[lane] : 0xFFFFFFFFu, mx = lane < NW ? sm.wmax[lane] : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        sm.sc[0] = (int)mn;
        sm.sc[1] = (int)mx;
      }
    }
    __syncthreads();
    const unsigned vmin = (unsigned)sm.sc[0], range = (unsigned)sm.sc[1] - vmin;
    const int bits = range ? 32 - __clz(range) : 0;
    const int passes = (bits + 7) / 8;
    unsigned prefix = 0;  // of key' = last_use - vmin, digits fixed so far
    int need = q;         // how many still to take within the current prefix bucket
    for (int p = passes - 1; p >= 0; --p) {
      const int shift = 8 * p;
      if (tid < 256) sm.hist[tid] = 0;
      __syncthreads();
      for (int s = s0; s < s1; ++s) {
        unsigned v = lu[s];
        if (v >= now) continue;
        unsigned kk = v - vmin;
        // higher digits must match the prefix (shift+8 may be 32: test in 64 bits)
        if (((unsigned long long)kk >> (shift + 8)) != ((unsigned long long)prefix >> (shift + 8))) continue;
        atomicAdd(&sm.hist[(kk >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (wid == 0) {
        // lane owns bins [8*lane, 8*lane+8)
        unsigned c[8], loc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = sm.hist[8 * lane + i];
          loc += c[i];
        }
        unsigned incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        unsigned before = incl - loc;
        // the lane whose range crosses `need`
        bool mine = before < (unsigned)need && (unsigned)need <= incl;
        if (mine) {
          unsigned acc = before;
          int d = 0;
          for (; d < 8; ++d) {
            if (acc + c[d] >= (unsigned)need) break;
            acc += c[d];
          }
          sm.sc[2] = 8 * lane + d;
          sm.sc[3] = need - (int)acc;
        }
      }
      __syncthreads();
      prefix |= (unsigned)sm.sc[2] << shift;
      need = sm.sc[3];
      __syncthreads();
    }
    const unsigned thr = vmin + prefix;  // last_use of the q-th smallest key
    const int need_eq = need;             // slots with last_use == thr to take, lowest index first

    int my_lt = 0, my_eq = 0;
    for (int s = s0; s < s1; ++s) {
      unsigned v = lu[s];
      my_lt += v < thr;
      my_eq += v == thr;
    }
    int tot2;
    int ex2 = block_scan<NT>(my_lt | (my_eq << 16), sm.wsum, &tot2);
    int lt_pos = ex2 & 0xFFFF, eq_pos = ex2 >> 16;
    const int c_lt = tot2 & 0xFFFF;
    for (int s = s0; s < s1; ++s) {
      unsigned v = lu[s];
      if (v < thr) {
        sm.cand[lt_pos++] = ((unsigned long long)v << 32) | (unsigned)s;
      } else if (v == thr) {
        if (eq_pos < need_eq) sm.eqsel[eq_pos] = s;
        ++eq_pos;
      }
    }
    __syncthreads();
    for (int i = tid; i < c_lt; i += NT) {
      unsigned long long key = sm.cand[i];
      int rank = 0;
      for (int j = 0; j < c_lt; ++j) rank += sm.cand[j] < key;
      sm.victims[rank] = (int)(key & 0xFFFFFFFFu);
    }
    for (int i = tid; i < need_eq; i += NT) sm.victims[c_lt + i] = sm.eqsel[i];
    __syncthreads();
  }

  // 5. table update (fill i -> victim i) and CPU list
  int my_evict = 0;
  for (int i = tid; i < q; i += NT) {
    int s = sm.victims[i];
    int le = sm.miss_local[i];
    int u = base_id + le;
    int old = a.expert_of[s];
    a.evicted[i] = old;
    if (old >= 0) {
      a.slot_of[old] = -1;
      my_evict = 1;
    }
    a.slot_of[u] = s;
    a.expert_of[s] = u;
    a.last_use[s] = now;
    a.fetch[i] = u;
    a.victims[i] = s;
    sm.emap[le] = s;
    sm.filled[le] = 1;
  }
  for (int i = q + tid; i < m; i += NT) a.cpu_list[i - q] = base_id + sm.miss_local[i];
  const int evictions = __syncthreads_count(my_evict);

  // 6. rewrite
  for (int r = tid; r < a.n_routes; r += NT) {
    int le = rids[r];
    a.slot_ids[r] = ((unsigned)le < (unsigned)E) ? sm.emap[le] : -1;
  }

  // 7. groups of routes per resident expert, experts ascending
  const bool resident = present && sm.emap[e] >= 0;
  int tot3;
  int ex3 = block_scan<NT>(resident ? (sm.ecount[e] | 0x10000) : 0, sm.wsum, &tot3);
  const int n_groups = tot3 >> 16, n_grouped = tot3 & 0xFFFF;
  if (resident) {
    int gi = ex3 >> 16, off = ex3 & 0xFFFF;
    a.group_slot[gi] = sm.emap[e];
    a.group_new[gi] = sm.filled[e];
    a.group_off[gi] = off;
    sm.gstart[e] = off;
  }
  if (tid == 0) a.group_off[n_groups] = n_grouped;
  __syncthreads();
  for (int r = tid; r < a.n_routes; r += NT) {
    int le = rids[r];
    if ((unsigned)le < (unsigned)E && sm.emap[le] >= 0) {
      int pos = sm.gstart[le] + atomicAdd(&sm.cursor[le], 1);
      a.group_routes[pos] = r;
    }
  }

  if (tid == 0) {
    a.counts[0] = n;
    a.counts[1] = hits;
    a.counts[2] = m;
    a.counts[3] = q;
    a.counts[4] = m - q;
    a.counts[5] = n_groups;
    a.counts[6] = (int)now;
    a.counts[7] = 0;
    *a.now = now;
    a.counters[0] += (unsigned long long)hits;
    a.counters[1] += (unsigned long long)m;
    a.counters[2] += (unsigned long long)q;
    a.counters[3] += (unsigned long long)(m - q);
    a.counters[4] += (unsigned long long)evictions;
    a.counters[5] += 1ull;
  }
}

}  // namespace

size_t control_smem_bytes(int S) { return sizeof(Smem) + sizeof(unsigned) * (size_t)S; }

namespace {
template <int RP, int NT>
cudaError_t launch_rp(const ControlArgs& a, cudaStream_t st) {
  const size_t smem = control_smem_bytes(a.S);
  static thread_local int configured_for = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_for != dev) {
    cudaError_t e = cudaFuncSetAttribute(control_kernel<RP, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)control_smem_bytes(kMaxSlots));
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(cfg, attr, dim3(1), dim3(NT), smem, st);
  return cudaLaunchKernelEx(&cfg, control_kernel<RP, NT>, a);
}

__global__ void set_ratio_kernel(long long* ratio, long long r_num, long long r_den) {
  ratio[0] = r_num;
  ratio[1] = r_den;
}
}  // namespace

cudaError_t launch_set_ratio(long long* ratio, long long r_num, long long r_den, cudaStream_t st) {
  set_ratio_kernel<<<1, 1, 0, st>>>(ratio, r_num, r_den);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_nt(const ControlArgs& a, cudaStream_t st) {
  if (!a.logits) return launch_rp<0, NT>(a, st);
  if (a.ids != a.ids_out || a.T * a.k != a.n_routes) return cudaErrorInvalidValue;
  const int per = (a.E + 31) / 32;
  if (per <= 1) return launch_rp<1, NT>(a, st);
  if (per <= 4) return launch_rp<4, NT>(a, st);
  if (per <= 8) return launch_rp<8, NT>(a, st);
  return launch_rp<kMaxExperts / 32, NT>(a, st);
}

cudaError_t launch_control(const ControlArgs& a, cudaStream_t st) {
  // Half the threads for a step of few routes, when every expert still has
  // its own: each of the many block-wide barriers then costs less (route +
  // control of an A3B decode step: 7.0 instead of 8.2 us; 256 threads were
  // slower again).  Steps of many routes, with many misses to place, keep the
  // full block (64 tokens x top-8 with ~120 fills: 8.2 us, 9.5 with half).
  if (a.E <= kControlThreads / 2 && a.n_routes <= 128) return launch_nt<kControlThreads / 2>(a, st);
  return launch_nt<kControlThreads>(a, st);
}

}  // namespace ft
