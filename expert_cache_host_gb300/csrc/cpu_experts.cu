// CPU expert executor: the host side of the decode split.
//
// FreeToken article, section "设计 1" (bandwidth-adaptive execution), Decode
// bullet.  Of a step's m missed experts the control kernel fills q into slots;
// the routes of the remaining misses are computed here on the host cores from
// the pool bytes, and the merge kernel adds the GPU's routes to this sum, so
// the layer output is unchanged by the split.  For the routes of a step that
// got no slot (slot id < 0) this file computes
//     partial[t] = sum_j w[t,j] * SwiGLU expert ids[t,j] applied to hidden[t]
// on the host cores, in fp32, reading the expert bytes from the pool in the
// canonical layout (bf16, or MXFP4 codes with e8m0 scales).
//
// Work split (deterministic for any thread count): the intermediate rows
// h[route][i] = silu(W_gate[i] . x) * (W_up[i] . x) are divided among the
// threads, then the output rows; each output element sums its routes in route
// order, so the result does not depend on how the rows were divided.
//
// In a context the executor runs inside the stream order: copies of the step's
// route arrays and hidden rows to pinned host memory and a host function
// (capturable in a CUDA graph) that writes the partial sum into mapped pinned
// memory, on a stream of its own that runs beside the fill and the GPU experts;
// the merge waits for it and reads the sum there.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "ft_internal.h"

namespace ft {
namespace {

// ------------------------------------------------------------ element values

inline float bf16_value(uint16_t v) {
  const uint32_t u = (uint32_t)v << 16;
  float f;
  memcpy(&f, &u, sizeof(f));
  return f;
}

// e2m1 (OCP Microscaling v1.0): sign, 2 exponent bits, 1 mantissa bit.
const float kE2m1[16] = {0.0f,  0.5f,  1.0f,  1.5f,  2.0f,  3.0f,  4.0f,  6.0f,
                         -0.0f, -0.5f, -1.0f, -1.5f, -2.0f, -3.0f, -4.0f, -6.0f};

// e8m0 scale: 2^(E - 127); E = 255 is NaN.
inline float e8m0_value(uint8_t e) { return e == 255 ? NAN : ldexpf(1.0f, (int)e - 127); }

// Dot products of one weight row with an fp32 vector; eight partial sums in a
// fixed order (n is a multiple of 32 for every shape the library accepts).
float dot_bf16(const uint16_t* w, const float* x, int n) {
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < n; j += 8)
    for (int u = 0; u < 8; ++u) a[u] += bf16_value(w[j + u]) * x[j + u];
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// One MXFP4 row: n/2 code bytes (element 2i in the low nibble) and n/32 scales.
float dot_mxfp4(const uint8_t* codes, const uint8_t* scales, const float* x, int n) {
  float acc = 0.f;
  for (int g = 0; g < n / 32; ++g) {
    const uint8_t* c = codes + 16 * g;
    const float* xg = x + 32 * g;
    float s0 = 0.f, s1 = 0.f;
    for (int b = 0; b < 16; ++b) {
      s0 += kE2m1[c[b] & 15] * xg[2 * b];
      s1 += kE2m1[c[b] >> 4] * xg[2 * b + 1];
    }
    acc += e8m0_value(scales[g]) * (s0 + s1);
  }
  return acc;
}

inline float silu(float g) { return g / (1.f + expf(-g)); }

// ------------------------------------------------------------ worker pool

// A fixed set of threads that run one function over [0, n) in contiguous
// ranges; the calling thread takes the first range.  Between tasks a worker
// polls for the next one for a short while (decode layers follow each other
// within a fraction of a millisecond) and then sleeps on a condition variable.
class WorkerPool {
 public:
  explicit WorkerPool(int threads) : n_(threads < 1 ? 1 : threads) {
    for (int i = 1; i < n_; ++i) th_.emplace_back([this, i] { loop(i); });
  }
  ~WorkerPool() {
    {
      std::lock_guard<std::mutex> l(mu_);
      stop_.store(true);
    }
    cv_.notify_all();
    for (auto& t : th_) t.join();
  }
  int size() const { return n_; }

  // fn(begin, end) over the items [0, n), one range per thread.
  void parallel(int n, const std::function<void(int, int)>& fn) {
    if (n <= 0) return;
    const int parts = n < n_ ? n : n_;
    auto range = [n, parts](int i, int* b, int* e) {
      *b = (int)((long long)n * i / parts);
      *e = (int)((long long)n * (i + 1) / parts);
    };
    if (parts == 1) {
      fn(0, n);
      return;
    }
    task_ = [&fn, &range, parts](int i) {
      if (i >= parts) return;
      int b, e;
      range(i, &b, &e);
      fn(b, e);
    };
    pending_.store(n_ - 1);
    {
      std::lock_guard<std::mutex> l(mu_);  // a worker about to sleep sees the new generation
      gen_.fetch_add(1, std::memory_order_release);
    }
    cv_.notify_all();
    int b, e;
    range(0, &b, &e);
    fn(b, e);
    while (pending_.load(std::memory_order_acquire) != 0) {
    }
  }

 private:
  void loop(int i) {
    long long seen = 0;
    for (;;) {
      const auto t0 = std::chrono::steady_clock::now();
      for (int spin = 0; gen_.load(std::memory_order_acquire) == seen && !stop_.load(); ++spin) {
        if ((spin & 255) == 255 && std::chrono::steady_clock::now() - t0 > std::chrono::microseconds(kSpinUs)) {
          std::unique_lock<std::mutex> l(mu_);
          cv_.wait(l, [&] { return stop_.load() || gen_.load() != seen; });
          break;
        }
      }
      if (stop_.load()) return;
      seen = gen_.load(std::memory_order_acquire);
      task_(i);
      pending_.fetch_sub(1, std::memory_order_release);
    }
  }

  static constexpr int kSpinUs = 300;
  int n_;
  std::vector<std::thread> th_;
  std::mutex mu_;
  std::condition_variable cv_;
  std::function<void(int)> task_;
  std::atomic<long long> gen_{0};
  std::atomic<int> pending_{0};
  std::atomic<bool> stop_{false};
};

}  // namespace

// ------------------------------------------------------------ the partial sum

struct CpuModel {
  const uint8_t* pool;  // host pool, canonical layout
  int E, k, d, f, dtype;
  size_t Bx;
};

struct CpuScratch {
  std::vector<float> x, h;  // [T][d] activations, [routes][f] intermediate
  std::vector<int> rt, re;  // token and expert of each CPU route
  std::vector<float> rw;    // its routing weight
};

namespace {

// partial [T, d] (written) for the routes with slot_ids < 0 and an expert id
// in [0, E); the other routes are the GPU's.  Returns the number of routes
// computed (each reads its expert's B_x bytes once).
int cpu_partial(const CpuModel& m, int layer, int T, const int32_t* ids, const float* w, const int32_t* slot_ids,
                const uint16_t* hidden, float* partial, WorkerPool& pool, CpuScratch& s) {
  const int d = m.d, f = m.f, k = m.k;
  const size_t df = (size_t)d * f;
  s.rt.clear();
  s.re.clear();
  s.rw.clear();
  for (int r = 0; r < T * k; ++r) {
    if (slot_ids[r] >= 0) continue;
    const int e = ids[r];
    if (e < 0 || e >= m.E) continue;
    s.rt.push_back(r / k);
    s.re.push_back(e);
    s.rw.push_back(w[r]);
  }
  const int nc = (int)s.rt.size();
  if (nc == 0) {
    memset(partial, 0, sizeof(float) * (size_t)T * d);
    return 0;
  }
  s.x.resize((size_t)T * d);
  for (size_t i = 0; i < (size_t)T * d; ++i) s.x[i] = bf16_value(hidden[i]);
  s.h.resize((size_t)nc * f);
  auto expert = [&](int e) { return m.pool + ((size_t)layer * m.E + e) * m.Bx; };
  const bool bf16 = m.dtype == FT_DTYPE_BF16;

  // h[route][i] = silu(W_gate[i] . x) * (W_up[i] . x), over blocks of routes
  // small enough that the item count stays an int
  const int rb = (int)std::max<long long>(1, (1LL << 30) / f);
  for (int r0 = 0; r0 < nc; r0 += rb) {
    const int nr = std::min(rb, nc - r0);
    pool.parallel(nr * f, [&](int b, int end) {
      for (int it = b; it < end; ++it) {
        const int ri = r0 + it / f, i = it % f;
        const uint8_t* ex = expert(s.re[ri]);
        const float* x = s.x.data() + (size_t)s.rt[ri] * d;
        float g, u;
        if (bf16) {
          const uint16_t* wg = reinterpret_cast<const uint16_t*>(ex);
          g = dot_bf16(wg + (size_t)i * d, x, d);
          u = dot_bf16(wg + df + (size_t)i * d, x, d);
        } else {
          const uint8_t* sc = ex + 3 * df / 2;  // scales gate [f][d/32], then up
          g = dot_mxfp4(ex + (size_t)i * (d / 2), sc + (size_t)i * (d / 32), x, d);
          u = dot_mxfp4(ex + df / 2 + (size_t)i * (d / 2), sc + df / 32 + (size_t)i * (d / 32), x, d);
        }
        s.h[(size_t)ri * f + i] = silu(g) * u;
      }
    });
  }

  // partial[t][row] = sum over the CPU routes of token t, in route order,
  // of w * (W_down[row] . h[route])
  pool.parallel(d, [&](int b, int end) {
    for (int row = b; row < end; ++row) {
      for (int t = 0; t < T; ++t) partial[(size_t)t * d + row] = 0.f;
      for (int ri = 0; ri < nc; ++ri) {
        const uint8_t* ex = expert(s.re[ri]);
        const float* h = s.h.data() + (size_t)ri * f;
        float y;
        if (bf16) {
          const uint16_t* wd = reinterpret_cast<const uint16_t*>(ex) + 2 * df;  // [d][f]
          y = dot_bf16(wd + (size_t)row * f, h, f);
        } else {
          const uint8_t* sc = ex + 3 * df / 2 + 2 * (df / 32);  // scales down [d][f/32]
          y = dot_mxfp4(ex + df + (size_t)row * (f / 2), sc + (size_t)row * (f / 32), h, f);
        }
        partial[(size_t)s.rt[ri] * d + row] += s.rw[ri] * y;
      }
    }
  });
  return nc;
}

}  // namespace

// ------------------------------------------------------------ in a context

struct CpuJob {
  CpuExec* ex;
  int layer, T;
};

struct CpuExec {
  explicit CpuExec(int threads) : pool(threads) {}
  CpuModel m{};
  int L = 0, t_max = 0;
  WorkerPool pool;
  CpuScratch s;
  cudaStream_t st = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // pinned staging of one step: route ids | weights | slot ids (each t_max*k
  // entries, the layout of a layer's step buffers, so one copy can bring all
  // three), the hidden rows, and the result (mapped: the merge reads it there)
  int32_t* h_routes = nullptr;
  int32_t* h_ids = nullptr;
  float* h_w = nullptr;
  int32_t* h_slot = nullptr;
  uint16_t* h_hidden = nullptr;
  float* h_partial = nullptr;
  float* d_partial = nullptr;  // device view of h_partial
  std::vector<CpuJob> jobs;    // [L][t_max]: the host function's argument per (layer, T)
  // host-side rate (the BH of the split): expert bytes read and compute time
  // of the host functions that had routes to compute
  std::atomic<unsigned long long> meter_bytes{0}, meter_ns{0}, meter_calls{0};
};

namespace {

void CUDART_CB cpu_job_fn(void* p) {
  const CpuJob* j = static_cast<const CpuJob*>(p);
  CpuExec* ex = j->ex;
  const auto t0 = std::chrono::steady_clock::now();
  const int nc =
      cpu_partial(ex->m, j->layer, j->T, ex->h_ids, ex->h_w, ex->h_slot, ex->h_hidden, ex->h_partial, ex->pool, ex->s);
  if (nc > 0) {
    const auto ns = std::chrono::duration_cast<std::chrono::nanoseconds>(std::chrono::steady_clock::now() - t0);
    ex->meter_bytes += (unsigned long long)nc * ex->m.Bx;
    ex->meter_ns += (unsigned long long)ns.count();
    ex->meter_calls += 1;
  }
}

}  // namespace

void cpu_exec_destroy(CpuExec* ex) {
  if (!ex) return;
  if (ex->st) cudaStreamSynchronize(ex->st);
  if (ex->h_routes) cudaFreeHost(ex->h_routes);
  if (ex->h_hidden) cudaFreeHost(ex->h_hidden);
  if (ex->h_partial) cudaFreeHost(ex->h_partial);
  if (ex->ev_fork) cudaEventDestroy(ex->ev_fork);
  if (ex->ev_join) cudaEventDestroy(ex->ev_join);
  if (ex->st) cudaStreamDestroy(ex->st);
  delete ex;
}

int cpu_exec_create(CpuExec** out, int threads, const uint8_t* pool_host, int L, int E, int k, int d, int f,
                    int dtype, size_t Bx, int t_max) {
  *out = nullptr;
  CpuExec* ex = new CpuExec(threads);
  ex->m = CpuModel{pool_host, E, k, d, f, dtype, Bx};
  ex->L = L;
  ex->t_max = t_max;
  const size_t R = (size_t)t_max * k, TD = (size_t)t_max * d;
  bool ok = cudaStreamCreateWithFlags(&ex->st, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&ex->ev_fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ex->ev_join, cudaEventDisableTiming) == cudaSuccess &&
            cudaHostAlloc(reinterpret_cast<void**>(&ex->h_routes), sizeof(int32_t) * 3 * R, 0) == cudaSuccess &&
            cudaHostAlloc(reinterpret_cast<void**>(&ex->h_hidden), sizeof(uint16_t) * TD, 0) == cudaSuccess &&
            cudaHostAlloc(reinterpret_cast<void**>(&ex->h_partial), sizeof(float) * TD, cudaHostAllocMapped) ==
                cudaSuccess &&
            cudaHostGetDevicePointer(reinterpret_cast<void**>(&ex->d_partial), ex->h_partial, 0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    cpu_exec_destroy(ex);
    return record_error(FT_E_NOMEM, "CPU executor: stream, events or staging buffers could not be allocated");
  }
  ex->h_ids = ex->h_routes;
  ex->h_w = reinterpret_cast<float*>(ex->h_routes + R);
  ex->h_slot = ex->h_routes + 2 * R;
  ex->jobs.resize((size_t)L * t_max);
  for (int l = 0; l < L; ++l)
    for (int t = 1; t <= t_max; ++t) ex->jobs[(size_t)l * t_max + (t - 1)] = CpuJob{ex, l, t};
  *out = ex;
  return FT_OK;
}

cudaError_t cpu_exec_fork(CpuExec* ex, int layer, int T, const int32_t* slot_ids, const int32_t* ids, const float* w,
                          const uint16_t* hidden, cudaStream_t st, Profiler& prof) {
  const size_t R = (size_t)T * ex->m.k, TD = (size_t)T * ex->m.d, RC = (size_t)ex->t_max * ex->m.k;
  cudaError_t e;
  if ((e = cudaEventRecord(ex->ev_fork, st)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(ex->st, ex->ev_fork, 0)) != cudaSuccess) return e;
  cudaEvent_t pb = prof.begin(ex->st);
  const bool one_block = reinterpret_cast<const void*>(w) == ids + RC && slot_ids == ids + 2 * RC;
  if (one_block) {
    // ids | w | slot_ids adjacent on the device, as in the staging block
    e = cudaMemcpyAsync(ex->h_routes, ids, sizeof(int32_t) * (2 * RC + R), cudaMemcpyDeviceToHost, ex->st);
  } else if ((e = cudaMemcpyAsync(ex->h_ids, ids, sizeof(int32_t) * R, cudaMemcpyDeviceToHost, ex->st)) == cudaSuccess &&
             (e = cudaMemcpyAsync(ex->h_w, w, sizeof(float) * R, cudaMemcpyDeviceToHost, ex->st)) == cudaSuccess) {
    e = cudaMemcpyAsync(ex->h_slot, slot_ids, sizeof(int32_t) * R, cudaMemcpyDeviceToHost, ex->st);
  }
  if (e != cudaSuccess) return e;
  if ((e = cudaMemcpyAsync(ex->h_hidden, hidden, sizeof(uint16_t) * TD, cudaMemcpyDeviceToHost, ex->st)) != cudaSuccess)
    return e;
  // the result lands in mapped host memory, which the merge reads directly
  if ((e = cudaLaunchHostFunc(ex->st, cpu_job_fn, &ex->jobs[(size_t)layer * ex->t_max + (T - 1)])) != cudaSuccess)
    return e;
  prof.end(ex->st, FT_K_CPU, pb);
  return cudaEventRecord(ex->ev_join, ex->st);
}

cudaError_t cpu_exec_join(CpuExec* ex, cudaStream_t st) { return cudaStreamWaitEvent(st, ex->ev_join, 0); }

const float* cpu_exec_partial(const CpuExec* ex) { return ex->d_partial; }

void cpu_exec_meter(CpuExec* ex, unsigned long long* bytes, unsigned long long* ns, unsigned long long* calls,
                    int reset) {
  if (reset) {
    *bytes = ex->meter_bytes.exchange(0);
    *ns = ex->meter_ns.exchange(0);
    *calls = ex->meter_calls.exchange(0);
  } else {
    *bytes = ex->meter_bytes.load();
    *ns = ex->meter_ns.load();
    *calls = ex->meter_calls.load();
  }
}

}  // namespace ft

// ------------------------------------------------------------ standalone entry

extern "C" int ft_cpu_experts(const void* pool_host, int num_experts, int top_k, int hidden, int inter, int dtype,
                              int layer, int T, const int32_t* ids, const float* weights, const int32_t* slot_ids,
                              const uint16_t* hidden_rows, float* partial, int threads) {
  using namespace ft;
  if (!pool_host || !ids || !weights || !slot_ids || !hidden_rows || !partial)
    return record_error(FT_E_ARG, "null pointer argument");
  if (num_experts < 1 || top_k < 1 || top_k > num_experts || layer < 0 || T < 1 || (long long)T * top_k > (1 << 24))
    return record_error(FT_E_ARG, "bad num_experts, top_k, layer or T (T * top_k <= 2^24)");
  if (hidden < 32 || hidden % 32 || inter < 32 || inter % 32 || hidden > (1 << 20) || inter > (1 << 20))
    return record_error(FT_E_ARG, "hidden and inter must be multiples of 32 in [32, 2^20]");
  if (dtype != FT_DTYPE_BF16 && dtype != FT_DTYPE_MXFP4) return record_error(FT_E_ARG, "dtype must be BF16 or MXFP4");
  if (threads < 1 || threads > 1024) return record_error(FT_E_ARG, "threads must be in [1, 1024]");
  const size_t df = (size_t)hidden * inter;
  const size_t Bx = dtype == FT_DTYPE_BF16 ? 6 * df : 3 * df / 2 + 3 * df / 32;
  const CpuModel m{static_cast<const uint8_t*>(pool_host), num_experts, top_k, hidden, inter, dtype, Bx};
  WorkerPool pool(threads);
  CpuScratch s;
  cpu_partial(m, layer, T, ids, weights, slot_ids, hidden_rows, partial, pool, s);
  return FT_OK;
}
