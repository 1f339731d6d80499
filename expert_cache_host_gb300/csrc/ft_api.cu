// C ABI: context, host-pool pinning, per-layer step buffers, streams, and the
// order in which one MoE layer step's kernels are enqueued.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "ft_internal.h"
#include "prefill.h"
#include "tma.h"

using namespace ft;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

#define CU(call)                                                                              \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess) return fail(FT_E_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

size_t expert_bytes(const ft_config& c) {
  size_t df = (size_t)c.hidden * (size_t)c.inter;
  return c.dtype == FT_DTYPE_BF16 ? 6 * df : 3 * df / 2 + 3 * df / 32;
}

}  // namespace

int ft::record_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

struct ft_ctx {
  ft_config cfg{};
  int device = 0;
  int sm_count = 0;
  int S = 0;
  int E_tot = 0;
  size_t Bx = 0;
  int epoch = 0;

  void* host_pool = nullptr;
  size_t pool_bytes = 0;
  bool registered = false;
  const uint8_t* pool_dev = nullptr;

  uint8_t* arena = nullptr;
  CUtensorMap tmap_wd{};  // (f, d, slot) view of every slot's W_down, for the decode expert kernel
  CUtensorMap tmap_gu{};  // (d, f, {gate, up}, slot) view of every slot's W_gate / W_up
  int32_t* slot_of = nullptr;
  int32_t* expert_of = nullptr;
  uint32_t* last_use = nullptr;
  uint32_t* now = nullptr;
  long long* ratio = nullptr;  // [2] r_num, r_den
  uint32_t* status = nullptr;
  unsigned long long* counters = nullptr;

  void* layer_mem = nullptr;
  std::vector<LayerBufs> layers;
  float* ypart = nullptr;
  int n_chunks = 0;

  cudaStream_t xfer = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;

  // copy-engine fill mode: host copies of the step's fetch list
  int32_t* h_counts = nullptr;
  int32_t* h_fetch = nullptr;
  int32_t* h_victims = nullptr;

  PrefillState* prefill = nullptr;
  CpuExec* cpu = nullptr;  // host expert executor, or none
  Profiler prof;

  FillMeter* meter = nullptr;  // device: [0] the decode fill's link rate, [1] the fused path's resident-expert phase

  // fused decode path (FT_DECODE_FUSED): one CTA per SM, fill_ctas of them fill
  bool fused = false;
  int fused_ns = 0, fused_fill = 0, fused_groups = 0, fused_grid = 0;
  uint32_t* ready = nullptr;         // [K_max] clock stamp of each fetch entry's completed fill
  unsigned int* fill_done = nullptr;  // [K_max] fill CTAs done with each entry
  unsigned int* sched = nullptr;      // [2] work-item counter and CTAs done of the fused kernel
  // host expert rate reported by the caller (ft_report_host_rate) since the last reset
  double host_bytes = 0.0, host_s = 0.0;
};

namespace {

int check_config(const ft_config& c) {
  if (c.num_layers < 1) return fail(FT_E_ARG, "num_layers must be >= 1");
  if (c.num_experts < 1 || c.num_experts > kMaxExperts) return fail(FT_E_ARG, "num_experts must be in [1, %d]", kMaxExperts);
  if (c.top_k < 1 || c.top_k > kMaxTopK || c.top_k > c.num_experts) return fail(FT_E_ARG, "top_k must be in [1, min(32, E)]");
  if (c.hidden < 256 || c.hidden % 256) return fail(FT_E_ARG, "hidden must be a positive multiple of 256");
  if (c.inter < 128 || c.inter % 128) return fail(FT_E_ARG, "inter must be a positive multiple of 128");
  if (c.dtype != FT_DTYPE_BF16 && c.dtype != FT_DTYPE_MXFP4) return fail(FT_E_ARG, "dtype must be BF16 or MXFP4");
  if (c.num_slots < 1 || c.num_slots > kMaxSlots) return fail(FT_E_ARG, "num_slots must be in [1, %d]", kMaxSlots);
  if (c.k_max < 1 || c.k_max > kMaxKmax) return fail(FT_E_ARG, "k_max must be in [1, %d]", kMaxKmax);
  if (c.t_max < 1 || c.t_max > 1024 || c.t_max * c.top_k > 32768) return fail(FT_E_ARG, "t_max must be in [1, 1024] with t_max*k <= 32768");
  if (c.r_num < 0 || c.r_den < 1) return fail(FT_E_ARG, "r = r_num/r_den needs r_num >= 0, r_den >= 1");
  if (c.prefill_buffers < 0 || c.prefill_buffers > 2) return fail(FT_E_ARG, "prefill_buffers must be 0, 1 or 2");
  if (c.prefill_buffers > 0 && (c.prefill_t_max < 1 || c.prefill_t_max > 65536))
    return fail(FT_E_ARG, "prefill_t_max must be in [1, 65536] when prefill_buffers > 0");
  if (c.prefill_buffers > 0 && c.dtype == FT_DTYPE_MXFP4 && (c.hidden % 512 || c.inter % 512))
    return fail(FT_E_UNSUPPORTED, "MXFP4 prefill needs hidden and inter multiples of 512");
  if (c.fill_mode != FT_FILL_KERNEL && c.fill_mode != FT_FILL_COPY_ENGINE) return fail(FT_E_ARG, "bad fill_mode");
  if (c.fill_order != FT_FILL_ORDER_ID && c.fill_order != FT_FILL_ORDER_MOST_ROUTED) return fail(FT_E_ARG, "bad fill_order");
  if (c.decode_path != FT_DECODE_FUSED && c.decode_path != FT_DECODE_SPLIT) return fail(FT_E_ARG, "bad decode_path");
  if (c.fill_ctas < 0 || c.fill_ctas > 1024) return fail(FT_E_ARG, "fill_ctas must be in [0, 1024]");
  if (c.reserved[0]) return fail(FT_E_ARG, "reserved fields must be zero");
  if ((long long)c.num_layers * c.num_experts > 0x7fffffffLL) return fail(FT_E_ARG, "too many experts");
  return FT_OK;
}

int alloc_arena(ft_ctx* c, int S) {
  c->S = 0;
  size_t bytes = (size_t)S * c->Bx;
  if (cudaMalloc(&c->arena, bytes) != cudaSuccess) {
    cudaGetLastError();
    c->arena = nullptr;
    return fail(FT_E_NOMEM, "slot arena of %d slots (%zu bytes) does not fit", S, bytes);
  }
  if (cudaMalloc(&c->expert_of, sizeof(int32_t) * S) != cudaSuccess ||
      cudaMalloc(&c->last_use, sizeof(uint32_t) * S) != cudaSuccess) {
    cudaGetLastError();
    return fail(FT_E_NOMEM, "residency table allocation failed");
  }
  if (c->cfg.dtype == FT_DTYPE_BF16) {
    const uint64_t d = c->cfg.hidden, f = c->cfg.inter;
    const uint64_t dims[3] = {f, d, (uint64_t)S};
    const uint64_t strides[2] = {f * 2, c->Bx};
    const uint32_t box[3] = {(uint32_t)kDecodeChunk, 256, 1};
    char msg[160] = "";
    if (!encode_tensor_map(&c->tmap_wd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c->arena + 4 * d * f, dims, strides, box,
                           msg, sizeof(msg)))
      return fail(FT_E_CUDA, "tensor map of the slot arena: %s", msg);
    const uint64_t dims4[4] = {d, f, 2, (uint64_t)S};
    const uint64_t strides4[3] = {d * 2, d * f * 2, c->Bx};
    const uint32_t box4[4] = {256, (uint32_t)kDecodeChunk, 1, 1};
    if (!encode_tensor_map(&c->tmap_gu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, c->arena, dims4, strides4, box4, msg,
                           sizeof(msg)))
      return fail(FT_E_CUDA, "tensor map of the slot arena: %s", msg);
  } else {
    // MXFP4: byte views of the codes -- gate/up (d/2, f, {g, u}, slot), down (f/2, d, slot)
    const uint64_t d = c->cfg.hidden, f = c->cfg.inter;
    const uint64_t dims[3] = {f / 2, d, (uint64_t)S};
    const uint64_t strides[2] = {f / 2, c->Bx};
    const uint32_t box[3] = {(uint32_t)kDecodeChunkFp4 / 2, 256, 1};
    char msg[160] = "";
    if (!encode_tensor_map(&c->tmap_wd, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c->arena + d * f, dims, strides, box, msg,
                           sizeof(msg)))
      return fail(FT_E_CUDA, "tensor map of the slot arena: %s", msg);
    const uint64_t dims4[4] = {d / 2, f, 2, (uint64_t)S};
    const uint64_t strides4[3] = {d / 2, d * f / 2, c->Bx};
    const uint32_t box4[4] = {256, (uint32_t)kDecodeChunkFp4, 1, 1};
    if (!encode_tensor_map(&c->tmap_gu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, c->arena, dims4, strides4, box4, msg,
                           sizeof(msg)))
      return fail(FT_E_CUDA, "tensor map of the slot arena: %s", msg);
  }
  c->S = S;
  return FT_OK;
}

int reset_table(ft_ctx* c) {
  CU(cudaMemset(c->slot_of, 0xFF, sizeof(int32_t) * c->E_tot));
  CU(cudaMemset(c->expert_of, 0xFF, sizeof(int32_t) * c->S));
  CU(cudaMemset(c->last_use, 0, sizeof(uint32_t) * c->S));
  CU(cudaMemset(c->now, 0, sizeof(uint32_t)));
  // the fused path's fill stamps hold clock values: the clock restarts, so must they
  if (c->ready) CU(cudaMemset(c->ready, 0, sizeof(uint32_t) * c->cfg.k_max));
  CU(cudaMemset(c->counters, 0, sizeof(unsigned long long) * kCountersPerLayer * c->cfg.num_layers));
  for (auto& lb : c->layers) lb.last_T = -1;
  return FT_OK;
}

void free_all(ft_ctx* c) {
  if (c->prefill) prefill_destroy(c->prefill);
  c->prof.destroy();
  cudaFree(c->arena);
  cudaFree(c->slot_of);
  cudaFree(c->expert_of);
  cudaFree(c->last_use);
  cudaFree(c->now);
  cudaFree(c->ratio);
  cudaFree(c->status);
  cudaFree(c->counters);
  cudaFree(c->layer_mem);
  cudaFree(c->ypart);
  cudaFree(c->meter);
  cudaFree(c->ready);
  cudaFree(c->fill_done);
  cudaFree(c->sched);
  if (c->h_counts) cudaFreeHost(c->h_counts);
  if (c->h_fetch) cudaFreeHost(c->h_fetch);
  if (c->h_victims) cudaFreeHost(c->h_victims);
  cpu_exec_destroy(c->cpu);
  c->cpu = nullptr;
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  if (c->xfer) cudaStreamDestroy(c->xfer);
  if (c->registered) cudaHostUnregister(c->host_pool);
}

int check_layer(ft_ctx* c, int layer) {
  if (!c) return fail(FT_E_ARG, "null context");
  if (layer < 0 || layer >= c->cfg.num_layers) return fail(FT_E_ARG, "layer %d outside [0, %d)", layer, c->cfg.num_layers);
  if (c->S < 1) return fail(FT_E_STATE, "the cache has no slots (a rebuild failed)");
  return FT_OK;
}

// logits == nullptr: control on the given routes; else route into the layer's
// ids / weights first, in the same kernel.
int enqueue_control(ft_ctx* c, int layer, const float* logits, const int32_t* ids, int T, cudaStream_t st) {
  LayerBufs& lb = c->layers[layer];
  ControlArgs a{};
  a.layer = layer;
  if (logits) {
    a.logits = logits;
    a.T = T;
    a.k = c->cfg.top_k;
    a.ids_out = lb.ids;
    a.w_out = lb.w;
    ids = lb.ids;
  }
  a.E = c->cfg.num_experts;
  a.n_routes = T * c->cfg.top_k;
  a.S = c->S;
  a.K_max = c->cfg.k_max;
  a.ratio = c->ratio;
  a.fill_order = c->cfg.fill_order;
  a.ids = ids;
  lb.ids_src = ids;
  a.slot_of = c->slot_of;
  a.expert_of = c->expert_of;
  a.last_use = c->last_use;
  a.now = c->now;
  a.status = c->status;
  a.counters = c->counters + (size_t)kCountersPerLayer * layer;
  a.slot_ids = lb.slot_ids;
  a.uniq = lb.uniq;
  a.hit_list = lb.hit_list;
  a.fetch = lb.fetch;
  a.victims = lb.victims;
  a.evicted = lb.evicted;
  a.cpu_list = lb.cpu_list;
  a.counts = lb.counts;
  a.group_slot = lb.group_slot;
  a.group_new = lb.group_new;
  a.group_off = lb.group_off;
  a.group_routes = lb.group_routes;
  cudaEvent_t pb = c->prof.begin(st);
  CU(launch_control(a, st));
  c->prof.end(st, FT_K_CONTROL, pb);
  lb.last_T = T;
  return FT_OK;
}

void fill_out(ft_ctx* c, int layer, ft_step_out* out) {
  if (!out) return;
  LayerBufs& lb = c->layers[layer];
  out->ids = lb.ids;
  out->weights = lb.w;
  out->slot_ids = lb.slot_ids;
  out->uniq = lb.uniq;
  out->hit_list = lb.hit_list;
  out->fetch = lb.fetch;
  out->victims = lb.victims;
  out->evicted = lb.evicted;
  out->cpu_list = lb.cpu_list;
  out->counts = lb.counts;
}

int enqueue_fill(ft_ctx* c, int layer, int T, cudaStream_t st) {
  LayerBufs& lb = c->layers[layer];
  CU(cudaEventRecord(c->ev_fork, st));
  CU(cudaStreamWaitEvent(c->xfer, c->ev_fork, 0));
  cudaEvent_t pb = nullptr;
  if (c->cfg.fill_mode == FT_FILL_KERNEL) {
    pb = c->prof.begin(c->xfer);
    // Default grid, measured on the V4-style MXFP4 decode: at one token per
    // step 3/8 of the SMs carry the link as fast as all of them (~200 GB/s)
    // and the resident experts beside the fill stream ~1.5x faster (0.21
    // instead of 0.14 of HBM) on the SMs left free; at batch 16 the long
    // fills stream best from every SM.
    const int grid = c->cfg.fill_ctas ? std::min(c->cfg.fill_ctas, c->sm_count)
                                      : (T == 1 ? std::max(4, c->sm_count * 3 / 8) : c->sm_count);
    CU(launch_fill(c->pool_dev, c->arena, lb.counts, lb.fetch, lb.victims, c->Bx, c->S, c->E_tot, c->status,
                   &c->meter[0], grid, c->xfer));
  } else {
    // Copy-engine fills need the fetch list on the host: this reads it back.
    CU(cudaMemcpyAsync(c->h_counts, lb.counts, sizeof(int32_t) * kCountsLen, cudaMemcpyDeviceToHost, c->xfer));
    CU(cudaMemcpyAsync(c->h_fetch, lb.fetch, sizeof(int32_t) * c->cfg.k_max, cudaMemcpyDeviceToHost, c->xfer));
    CU(cudaMemcpyAsync(c->h_victims, lb.victims, sizeof(int32_t) * c->cfg.k_max, cudaMemcpyDeviceToHost, c->xfer));
    CU(cudaStreamSynchronize(c->xfer));
    pb = c->prof.begin(c->xfer);
    const int q = c->h_counts[3];
    for (int i = 0; i < q; ++i) {
      const int u = c->h_fetch[i], s = c->h_victims[i];
      if (u < 0 || u >= c->E_tot || s < 0 || s >= c->S) return fail(FT_E_STATE, "corrupt fetch list entry %d", i);
      CU(cudaMemcpyAsync(c->arena + (size_t)s * c->Bx, (const uint8_t*)c->host_pool + (size_t)u * c->Bx, c->Bx,
                         cudaMemcpyHostToDevice, c->xfer));
    }
  }
  c->prof.end(c->xfer, FT_K_FILL, pb);
  CU(cudaEventRecord(c->ev_join, c->xfer));  // the caller's stream waits on it before the installed experts run
  return FT_OK;
}

}  // namespace

extern "C" {

const char* ft_last_error(void) { return g_err; }

int ft_moe_init(const ft_config* cfg, void* host_pool, size_t pool_bytes, ft_ctx** out) {
  g_err[0] = 0;
  if (!cfg || !out) return fail(FT_E_ARG, "null config or output pointer");
  *out = nullptr;
  int rc = check_config(*cfg);
  if (rc) return rc;
  if (!host_pool) return fail(FT_E_ARG, "null host pool");
  ft_ctx* c = new (std::nothrow) ft_ctx();
  if (!c) return fail(FT_E_NOMEM, "host allocation failed");
  c->cfg = *cfg;
  c->E_tot = cfg->num_layers * cfg->num_experts;
  c->Bx = expert_bytes(*cfg);
  c->host_pool = host_pool;
  c->pool_bytes = pool_bytes;
  if (pool_bytes < (size_t)c->E_tot * c->Bx) {
    delete c;
    return fail(FT_E_ARG, "pool_bytes %zu < L*E*B_x = %zu", pool_bytes, (size_t)c->E_tot * c->Bx);
  }
  auto bail = [&](int code) {
    free_all(c);
    delete c;
    return code;
  };
  if (cudaGetDevice(&c->device) != cudaSuccess) return bail(fail(FT_E_CUDA, "no CUDA device"));
  cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);

  // Pin after write: the caller has already written the final layout.
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, host_pool) == cudaSuccess && pa.type == cudaMemoryTypeHost) {
    c->registered = false;
  } else {
    cudaGetLastError();
    cudaError_t e = cudaHostRegister(host_pool, pool_bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return bail(fail(FT_E_PIN, "cudaHostRegister of %zu bytes failed: %s", pool_bytes, cudaGetErrorString(e)));
    }
    c->registered = true;
  }
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, host_pool, 0) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(FT_E_PIN, "the host pool is pinned but not mapped into the device address space"));
  }
  c->pool_dev = static_cast<const uint8_t*>(dp);

  if (cudaMalloc(&c->slot_of, sizeof(int32_t) * c->E_tot) != cudaSuccess ||
      cudaMalloc(&c->now, sizeof(uint32_t)) != cudaSuccess || cudaMalloc(&c->status, sizeof(uint32_t)) != cudaSuccess ||
      cudaMalloc(&c->ratio, 2 * sizeof(long long)) != cudaSuccess ||
      cudaMalloc(&c->counters, sizeof(unsigned long long) * kCountersPerLayer * cfg->num_layers) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(FT_E_NOMEM, "table allocation failed"));
  }
  {
    const long long r[2] = {cfg->r_num, cfg->r_den};
    if (cudaMemcpy(c->ratio, r, sizeof(r), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return bail(fail(FT_E_CUDA, "ratio upload failed"));
    }
  }
  if ((rc = alloc_arena(c, cfg->num_slots))) return bail(rc);

  // per-layer step buffers, one allocation
  const int E = cfg->num_experts, TK = cfg->t_max * cfg->top_k, K = cfg->k_max;
  const size_t per_layer_words = (size_t)TK * 4 /*ids w slot_ids group_routes*/ +
                                 (size_t)E * 5 /*uniq hit cpu gslot gnew*/ + (E + 1) /*goff*/ + (size_t)K * 3 +
                                 kCountsLen;
  const size_t per_layer = (per_layer_words * 4 + 255) / 256 * 256;
  if (cudaMalloc(&c->layer_mem, per_layer * cfg->num_layers) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(FT_E_NOMEM, "step buffer allocation failed"));
  }
  c->layers.resize(cfg->num_layers);
  for (int l = 0; l < cfg->num_layers; ++l) {
    int32_t* p = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(c->layer_mem) + per_layer * l);
    LayerBufs& lb = c->layers[l];
    lb.ids = p; p += TK;
    lb.ids_src = lb.ids;
    lb.w = reinterpret_cast<float*>(p); p += TK;
    lb.slot_ids = p; p += TK;
    lb.group_routes = p; p += TK;
    lb.uniq = p; p += E;
    lb.hit_list = p; p += E;
    lb.cpu_list = p; p += E;
    lb.group_slot = p; p += E;
    lb.group_new = p; p += E;
    lb.group_off = p; p += E + 1;
    lb.fetch = p; p += K;
    lb.victims = p; p += K;
    lb.evicted = p; p += K;
    lb.counts = p; p += kCountsLen;
    lb.last_T = -1;
  }
  c->n_chunks = cfg->inter / (cfg->dtype == FT_DTYPE_BF16 ? kDecodeChunk : kDecodeChunkFp4);
  if (cudaMalloc(&c->ypart, sizeof(float) * (size_t)TK * c->n_chunks * cfg->hidden) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(FT_E_NOMEM, "decode work buffer allocation failed"));
  }
  if (cudaMemset(c->layer_mem, 0, per_layer * cfg->num_layers) != cudaSuccess ||
      cudaMemset(c->status, 0, sizeof(uint32_t)) != cudaSuccess)
    return bail(fail(FT_E_CUDA, "memset failed"));
  {
    const FillMeter m0[2] = {{~0ull, 0ull, 0ull, 0ull, 0ull, 0u, 0u}, {~0ull, 0ull, 0ull, 0ull, 0ull, 0u, 0u}};
    if (cudaMalloc(&c->meter, sizeof(m0)) != cudaSuccess ||
        cudaMemcpy(c->meter, m0, sizeof(m0), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&c->ready, sizeof(uint32_t) * K) != cudaSuccess ||
        cudaMalloc(&c->fill_done, sizeof(unsigned int) * K) != cudaSuccess ||
        cudaMemset(c->ready, 0, sizeof(uint32_t) * K) != cudaSuccess ||
        cudaMemset(c->fill_done, 0, sizeof(unsigned int) * K) != cudaSuccess ||
        cudaMalloc(&c->sched, 2 * sizeof(unsigned int)) != cudaSuccess ||
        cudaMemset(c->sched, 0, 2 * sizeof(unsigned int)) != cudaSuccess) {
      cudaGetLastError();
      return bail(fail(FT_E_NOMEM, "meter / fill stamp allocation failed"));
    }
  }
  // The fused decode path needs one CTA per SM with a ring of at least four
  // stages; where that does not fit, the split path serves the context.
  if ((cfg->dtype == FT_DTYPE_BF16 || (cfg->dtype == FT_DTYPE_MXFP4 && cfg->hidden % 512 == 0)) &&
      cfg->fill_mode == FT_FILL_KERNEL && cfg->decode_path == FT_DECODE_FUSED && cfg->hidden <= 8192) {
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    const int mg = std::min(TK, E);
    // as many CTAs per SM as the kernel is built for, if each still gets a ring of four stages; else one
    int want_per_sm = decode_layer_ctas_per_sm();
    int ns = decode_layer_ring_stages(cfg->hidden, mg, optin, want_per_sm, cfg->dtype);
    if (ns < 4) {
      want_per_sm = 1;
      ns = decode_layer_ring_stages(cfg->hidden, mg, optin, 1, cfg->dtype);
    }
    int per_sm = 0;
    if (ns >= 4 && decode_layer_max_blocks_per_sm(cfg->hidden, ns, mg, &per_sm, cfg->dtype) == cudaSuccess &&
        per_sm >= want_per_sm) {
      c->fused = true;
      c->fused_ns = ns;
      c->fused_groups = mg;
      c->fused_grid = want_per_sm * c->sm_count;
      // default: bf16 experts, 3/8 of the SMs fill (A3B decode, measured: 57 of 152 fill at 0.90-0.92
      // of the link, and the other 95 still finish the resident experts well before the fill; 38
      // lost 1 % tok/s); MXFP4 experts, 1/4 (V4 decode: 38 fill at the same ~200 GB/s and tok/s as
      // 57, and the issue-bound MXFP4 items stream 1.13x faster on the other 114)
      const int share = cfg->dtype == FT_DTYPE_MXFP4 ? c->fused_grid / 4 : c->fused_grid * 3 / 8;
      const int want = cfg->fill_ctas ? cfg->fill_ctas : std::max(4, share);
      c->fused_fill = std::min(want, c->fused_grid - 1);
    }
    cudaGetLastError();
  }
  if ((rc = reset_table(c))) return bail(rc);

  int lo = 0, hi = 0;
  cudaDeviceGetStreamPriorityRange(&lo, &hi);
  if (cudaStreamCreateWithPriority(&c->xfer, cudaStreamNonBlocking, hi) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming) != cudaSuccess)
    return bail(fail(FT_E_CUDA, "stream/event creation failed"));
  if (cfg->fill_mode == FT_FILL_COPY_ENGINE) {
    if (cudaMallocHost(&c->h_counts, sizeof(int32_t) * kCountsLen) != cudaSuccess ||
        cudaMallocHost(&c->h_fetch, sizeof(int32_t) * K) != cudaSuccess ||
        cudaMallocHost(&c->h_victims, sizeof(int32_t) * K) != cudaSuccess)
      return bail(fail(FT_E_NOMEM, "pinned host allocation failed"));
  }
  if (cfg->prefill_buffers > 0) {
    PrefillConfig pc{cfg->num_layers, cfg->num_experts, cfg->top_k, cfg->hidden, cfg->inter, cfg->dtype,
                     cfg->prefill_buffers, cfg->prefill_t_max, c->Bx, c->pool_dev, c->host_pool, c->status,
                     c->sm_count};
    char msg[256] = "";
    c->prefill = prefill_create(pc, msg, sizeof(msg));
    if (!c->prefill) return bail(fail(FT_E_NOMEM, "prefill buffers: %s", msg));
  }
  // Touch every 4 KB of the pool from the GPU once: the first GPU access to a
  // host page can be far slower than the next ones, and fills and uploads
  // should not pay it.  The meter's unused pad word is the loads' sink.
  if (launch_touch(c->pool_dev, (size_t)c->E_tot * c->Bx, reinterpret_cast<int*>(&c->meter[0].pad), 2 * c->sm_count,
                   0) != cudaSuccess)
    return bail(fail(FT_E_CUDA, "pool touch launch failed"));
  if (cudaDeviceSynchronize() != cudaSuccess) return bail(fail(FT_E_CUDA, "initialisation failed"));
  *out = c;
  return FT_OK;
}

int ft_moe_destroy(ft_ctx* c) {
  if (!c) return FT_OK;
  if (c->xfer) cudaStreamSynchronize(c->xfer);
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
  return FT_OK;
}

int ft_cpu_executor(ft_ctx* c, int threads) {
  if (!c) return fail(FT_E_ARG, "null context");
  if (threads < 0 || threads > 1024) return fail(FT_E_ARG, "threads must be in [0, 1024]");
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(c->xfer, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return fail(FT_E_STATE, "the CPU executor cannot change during a stream capture");
  CU(cudaDeviceSynchronize());
  cpu_exec_destroy(c->cpu);
  c->cpu = nullptr;
  if (threads == 0) return FT_OK;
  return cpu_exec_create(&c->cpu, threads, static_cast<const uint8_t*>(c->host_pool), c->cfg.num_layers,
                         c->cfg.num_experts, c->cfg.top_k, c->cfg.hidden, c->cfg.inter, c->cfg.dtype, c->Bx,
                         c->cfg.t_max);
}

int ft_set_ratio(ft_ctx* c, int32_t r_num, int32_t r_den, void* stream) {
  if (!c) return fail(FT_E_ARG, "null context");
  if (r_num < 0 || r_den < 1) return fail(FT_E_ARG, "r = r_num/r_den needs r_num >= 0, r_den >= 1");
  CU(launch_set_ratio(c->ratio, r_num, r_den, static_cast<cudaStream_t>(stream)));
  return FT_OK;
}

int ft_cache_rebuild_retain(ft_ctx* c, int new_slots) {
  if (!c) return fail(FT_E_ARG, "null context");
  if (new_slots < 1 || new_slots > kMaxSlots) return fail(FT_E_ARG, "new_slots must be in [1, %d]", kMaxSlots);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(c->xfer, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return fail(FT_E_STATE, "rebuild during stream capture");
  CU(cudaDeviceSynchronize());
  const int S_old = c->S;
  std::vector<int32_t> eo(S_old);
  std::vector<uint32_t> lu(S_old);
  CU(cudaMemcpy(eo.data(), c->expert_of, sizeof(int32_t) * S_old, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(lu.data(), c->last_use, sizeof(uint32_t) * S_old, cudaMemcpyDeviceToHost));
  // residents, most recent first (ties: lower slot); the first new_slots stay
  std::vector<int> kept;
  for (int s = 0; s < S_old; ++s)
    if (eo[s] >= 0) kept.push_back(s);
  std::stable_sort(kept.begin(), kept.end(), [&](int x, int y) { return lu[x] > lu[y]; });
  if ((int)kept.size() > new_slots) kept.resize(new_slots);

  // The new arena and tables are built next to the old ones; the context
  // switches to them only once every copy has succeeded, so on any failure
  // the old cache is left as it was.  slot_of is shared: its old contents are
  // kept on the host to put back.
  std::vector<int32_t> so_old(c->E_tot);
  CU(cudaMemcpy(so_old.data(), c->slot_of, sizeof(int32_t) * c->E_tot, cudaMemcpyDeviceToHost));
  uint8_t* old_arena = c->arena;
  int32_t* old_eo = c->expert_of;
  uint32_t* old_lu = c->last_use;
  const CUtensorMap old_wd = c->tmap_wd, old_gu = c->tmap_gu;
  c->arena = nullptr;
  c->expert_of = nullptr;
  c->last_use = nullptr;
  auto restore = [&](int code) {
    cudaStreamSynchronize(c->xfer);
    cudaGetLastError();
    cudaFree(c->arena);
    cudaFree(c->expert_of);
    cudaFree(c->last_use);
    c->arena = old_arena;
    c->expert_of = old_eo;
    c->last_use = old_lu;
    c->tmap_wd = old_wd;
    c->tmap_gu = old_gu;
    c->S = S_old;
    cudaMemcpy(c->slot_of, so_old.data(), sizeof(int32_t) * c->E_tot, cudaMemcpyHostToDevice);
    return code;
  };
  int rc = alloc_arena(c, new_slots);
  if (rc) return restore(rc);
#define CU_OR_RESTORE(call)                                                                               \
  do {                                                                                                    \
    cudaError_t e_ = (call);                                                                              \
    if (e_ != cudaSuccess) return restore(fail(FT_E_CUDA, "%s: %s", #call, cudaGetErrorString(e_))); \
  } while (0)
  std::vector<int32_t> so_new(c->E_tot, -1), eo_new(new_slots, -1);
  std::vector<uint32_t> lu_new(new_slots, 0);
  for (size_t i = 0; i < kept.size(); ++i) {
    const int s = kept[i], u = eo[s];
    eo_new[i] = u;
    so_new[u] = (int32_t)i;
    lu_new[i] = lu[s];
    CU_OR_RESTORE(cudaMemcpyAsync(c->arena + i * c->Bx, old_arena + (size_t)s * c->Bx, c->Bx,
                                  cudaMemcpyDeviceToDevice, c->xfer));
  }
  CU_OR_RESTORE(cudaMemcpy(c->expert_of, eo_new.data(), sizeof(int32_t) * new_slots, cudaMemcpyHostToDevice));
  CU_OR_RESTORE(cudaMemcpy(c->last_use, lu_new.data(), sizeof(uint32_t) * new_slots, cudaMemcpyHostToDevice));
  CU_OR_RESTORE(cudaStreamSynchronize(c->xfer));
  CU_OR_RESTORE(cudaMemcpy(c->slot_of, so_new.data(), sizeof(int32_t) * c->E_tot, cudaMemcpyHostToDevice));
#undef CU_OR_RESTORE
  cudaFree(old_arena);
  cudaFree(old_eo);
  cudaFree(old_lu);
  for (auto& lb : c->layers) lb.last_T = -1;
  ++c->epoch;
  return FT_OK;
}

int ft_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return fail(FT_E_ARG, "ft_host_alloc needs bytes > 0 and an output pointer");
  *out = nullptr;
  cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *out = nullptr;
    return fail(FT_E_PIN, "cudaHostAlloc of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
  }
  return FT_OK;
}

int ft_host_free(void* p) {
  if (!p) return FT_OK;
  CU(cudaFreeHost(p));
  return FT_OK;
}

int ft_cache_step(ft_ctx* c, int layer, const float* logits, int T, ft_step_out* out, void* stream) {
  int rc = check_layer(c, layer);
  if (rc) return rc;
  if (T < 1 || T > c->cfg.t_max) return fail(FT_E_ARG, "T=%d outside [1, t_max=%d]", T, c->cfg.t_max);
  if (!logits) return fail(FT_E_ARG, "null logits");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = enqueue_control(c, layer, logits, nullptr, T, st))) return rc;
  fill_out(c, layer, out);
  return FT_OK;
}

int ft_cache_control(ft_ctx* c, int layer, const int32_t* ids, int T, ft_step_out* out, void* stream) {
  int rc = check_layer(c, layer);
  if (rc) return rc;
  if (T < 1 || T > c->cfg.t_max) return fail(FT_E_ARG, "T=%d outside [1, t_max=%d]", T, c->cfg.t_max);
  if (!ids) return fail(FT_E_ARG, "null ids");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = enqueue_control(c, layer, nullptr, ids, T, st))) return rc;
  fill_out(c, layer, out);
  if (out) out->ids = const_cast<int32_t*>(ids);  // the control kernel read the caller's routes in place
  return FT_OK;
}

int ft_moe_forward(ft_ctx* c, int layer, int mode, const float* logits, const uint16_t* hidden, int T,
                   const float* partial, float* out, void* stream) {
  int rc = check_layer(c, layer);
  if (rc) return rc;
  if (!hidden || !out) return fail(FT_E_ARG, "null hidden or out");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mode == FT_PREFILL_LAYER) {
    if (!c->prefill) return fail(FT_E_STATE, "the context was created with prefill_buffers = 0");
    if (!logits) return fail(FT_E_ARG, "prefill needs router logits");
    if (T < 1 || T > c->cfg.prefill_t_max) return fail(FT_E_ARG, "T=%d outside [1, prefill_t_max]", T);
    char msg[256] = "";
    int r = prefill_forward(c->prefill, layer, logits, hidden, T, partial, out, st, &c->prof, msg, sizeof(msg));
    if (r) return fail(r, "prefill: %s", msg);
    return FT_OK;
  }
  if (mode != FT_DECODE_CACHED) return fail(FT_E_ARG, "unknown mode %d", mode);
  LayerBufs& lb = c->layers[layer];
  if (lb.last_T != T) return fail(FT_E_STATE, "decode forward of layer %d with T=%d needs a cache step with the same T", layer, T);
  // The CPU routes (if the executor is on) run on its stream and the fill on
  // the transfer stream; experts already resident run meanwhile on the
  // caller's stream, those the step installs after the fill.
  if (c->cpu) {
    if (partial) return fail(FT_E_ARG, "partial_dev must be NULL while the CPU executor is enabled");
    CU(cpu_exec_fork(c->cpu, layer, T, lb.slot_ids, lb.ids_src, lb.w, hidden, st, c->prof));
  }
  if (c->fused) {
    LayerArgs la{};
    DecodeArgs& a = la.d;
    a.arena = c->arena;
    a.Bx = c->Bx;
    a.S = c->S;
    a.d = c->cfg.hidden;
    a.f = c->cfg.inter;
    a.k = c->cfg.top_k;
    a.dtype = c->cfg.dtype;
    a.max_groups = c->fused_groups;
    a.T = T;
    a.counts = lb.counts;
    a.group_slot = lb.group_slot;
    a.group_off = lb.group_off;
    a.group_routes = lb.group_routes;
    a.group_new = lb.group_new;
    a.hidden = hidden;
    a.ypart = c->ypart;
    a.status = c->status;
    a.tmap_wd = &c->tmap_wd;
    a.tmap_gu = &c->tmap_gu;
    la.pool = reinterpret_cast<const int4*>(c->pool_dev);
    la.fetch = lb.fetch;
    la.victims = lb.victims;
    la.E_tot = c->E_tot;
    la.n_fill = c->fused_fill;
    la.ns = c->fused_ns;
    la.ready = c->ready;
    la.fill_done = c->fill_done;
    la.meter = &c->meter[0];
    la.xmeter = &c->meter[1];
    la.sched = c->sched;
    cudaEvent_t pb = c->prof.begin(st);
    cudaError_t e = launch_decode_layer(la, c->fused_grid, st);
    if (e != cudaSuccess) return fail(FT_E_CUDA, "fused decode layer launch failed: %s", cudaGetErrorString(e));
    c->prof.end(st, FT_K_EXPERTS, pb);
    if (c->cpu) {
      CU(cpu_exec_join(c->cpu, st));
      partial = cpu_exec_partial(c->cpu);
    }
    pb = c->prof.begin(st);
    CU(launch_merge(c->ypart, c->n_chunks, lb.slot_ids, lb.w, partial, out, T, c->cfg.top_k, c->cfg.hidden, st));
    c->prof.end(st, FT_K_MERGE, pb);
    return FT_OK;
  }
  if ((rc = enqueue_fill(c, layer, T, st))) return rc;
  DecodeArgs a{};
  a.arena = c->arena;
  a.Bx = c->Bx;
  a.S = c->S;
  a.d = c->cfg.hidden;
  a.f = c->cfg.inter;
  a.k = c->cfg.top_k;
  a.dtype = c->cfg.dtype;
  a.max_groups = T * c->cfg.top_k < c->cfg.num_experts ? T * c->cfg.top_k : c->cfg.num_experts;
  a.T = T;
  a.counts = lb.counts;
  a.group_slot = lb.group_slot;
  a.group_off = lb.group_off;
  a.group_routes = lb.group_routes;
  a.group_new = lb.group_new;
  a.hidden = hidden;
  a.ypart = c->ypart;
  a.status = c->status;
  a.tmap_wd = &c->tmap_wd;
  a.tmap_gu = &c->tmap_gu;
  cudaEvent_t pb = nullptr;
  for (int sel = 1; sel <= 2; ++sel) {
    if (sel == 2) CU(cudaStreamWaitEvent(st, c->ev_join, 0));
    a.select = sel;
    pb = c->prof.begin(st);
    cudaError_t e = c->cfg.dtype == FT_DTYPE_BF16 ? launch_decode_experts(a, st) : launch_decode_experts_mxfp4(a, T, st);
    if (e == cudaErrorNotSupported) return fail(FT_E_UNSUPPORTED, "decode experts for this dtype are not built");
    if (e == cudaErrorInvalidValue)
      return fail(FT_E_UNSUPPORTED, "decode experts need d <= 8192 (bf16) or d a multiple of 512 (MXFP4)");
    CU(e);
    c->prof.end(st, FT_K_EXPERTS, pb);
  }
  if (c->cpu) {
    CU(cpu_exec_join(c->cpu, st));
    partial = cpu_exec_partial(c->cpu);
  }
  pb = c->prof.begin(st);
  CU(launch_merge(c->ypart, c->n_chunks, lb.slot_ids, lb.w, partial, out, T, c->cfg.top_k, c->cfg.hidden, st));
  c->prof.end(st, FT_K_MERGE, pb);
  return FT_OK;
}

int ft_cache_rebuild(ft_ctx* c, int new_slots) {
  if (!c) return fail(FT_E_ARG, "null context");
  if (new_slots < 1 || new_slots > kMaxSlots) return fail(FT_E_ARG, "new_slots must be in [1, %d]", kMaxSlots);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(c->xfer, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return fail(FT_E_STATE, "rebuild during stream capture");
  CU(cudaDeviceSynchronize());
  cudaFree(c->arena);
  cudaFree(c->expert_of);
  cudaFree(c->last_use);
  c->arena = nullptr;
  c->expert_of = nullptr;
  c->last_use = nullptr;
  c->S = 0;
  ++c->epoch;
  int rc = alloc_arena(c, new_slots);
  if (rc) return rc;
  if ((rc = reset_table(c))) return rc;
  CU(cudaDeviceSynchronize());
  return FT_OK;
}

int ft_get_status(ft_ctx* c, uint32_t* status, int clear) {
  if (!c || !status) return fail(FT_E_ARG, "null argument");
  CU(cudaDeviceSynchronize());
  CU(cudaMemcpy(status, c->status, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  if (clear) CU(cudaMemset(c->status, 0, sizeof(uint32_t)));
  return FT_OK;
}

int ft_get_counters(ft_ctx* c, uint64_t* counters) {
  if (!c || !counters) return fail(FT_E_ARG, "null argument");
  CU(cudaDeviceSynchronize());
  CU(cudaMemcpy(counters, c->counters, sizeof(unsigned long long) * kCountersPerLayer * c->cfg.num_layers,
                cudaMemcpyDeviceToHost));
  return FT_OK;
}

int ft_get_table(ft_ctx* c, int32_t* slot_of, int32_t* expert_of, uint32_t* last_use, uint32_t* now) {
  if (!c) return fail(FT_E_ARG, "null context");
  CU(cudaDeviceSynchronize());
  if (slot_of) CU(cudaMemcpy(slot_of, c->slot_of, sizeof(int32_t) * c->E_tot, cudaMemcpyDeviceToHost));
  if (expert_of && c->S) CU(cudaMemcpy(expert_of, c->expert_of, sizeof(int32_t) * c->S, cudaMemcpyDeviceToHost));
  if (last_use && c->S) CU(cudaMemcpy(last_use, c->last_use, sizeof(uint32_t) * c->S, cudaMemcpyDeviceToHost));
  if (now) CU(cudaMemcpy(now, c->now, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  return FT_OK;
}

void* ft_slot_ptr(ft_ctx* c, int slot) {
  if (!c || slot < 0 || slot >= c->S) return nullptr;
  return c->arena + (size_t)slot * c->Bx;
}

int ft_ratio_adapter_init(ft_ratio_adapter* a, double alpha, int32_t r_den, int32_t r_num_max) {
  if (!a) return fail(FT_E_ARG, "null adapter");
  if (!(alpha > 0.0 && alpha <= 1.0)) return fail(FT_E_ARG, "alpha must be in (0, 1]");
  if (r_den < 1 || r_num_max < 0) return fail(FT_E_ARG, "r_den must be >= 1 and r_num_max >= 0");
  *a = ft_ratio_adapter{};
  a->alpha = alpha;
  a->r_den = r_den;
  a->r_num_max = r_num_max;
  a->r_num = -1;
  return FT_OK;
}

int ft_ratio_adapter_update(ft_ratio_adapter* a, double bp, double bh) {
  if (!a || !(a->alpha > 0.0 && a->alpha <= 1.0) || a->r_den < 1 || a->r_num_max < 0)
    return fail(FT_E_ARG, "adapter not initialised");
  auto blend = [&](double est, double x) { return est > 0.0 ? a->alpha * x + (1.0 - a->alpha) * est : x; };
  if (bp > 0.0) a->bp_gbs = blend(a->bp_gbs, bp);
  if (bh > 0.0) a->bh_gbs = blend(a->bh_gbs, bh);
  if (!(a->bp_gbs > 0.0 && a->bh_gbs > 0.0)) return 0;
  // r = BP/BH on the grid 1/r_den, rounded half up, capped
  const double x = (double)a->r_den * (a->bp_gbs / a->bh_gbs);
  const double cap = (double)a->r_num_max;
  const int32_t r = x + 0.5 >= cap ? a->r_num_max : (int32_t)floor(x + 0.5);
  ++a->updates;
  if (r == a->r_num) return 0;
  a->r_num = r;
  return 1;
}

int ft_report_host_rate(ft_ctx* c, double bytes, double seconds) {
  if (!c) return fail(FT_E_ARG, "null context");
  if (!(bytes >= 0.0) || !(seconds > 0.0)) return fail(FT_E_ARG, "bytes must be >= 0 and seconds > 0");
  c->host_bytes += bytes;
  c->host_s += seconds;
  return FT_OK;
}

int ft_measured_bandwidths(ft_ctx* c, double* bp_gbs, double* bh_gbs, int reset) {
  if (!c) return fail(FT_E_ARG, "null context");
  CU(cudaDeviceSynchronize());
  FillMeter m{};
  CU(cudaMemcpy(&m, &c->meter[0], sizeof(m), cudaMemcpyDeviceToHost));
  unsigned long long cb = 0, cns = 0, calls = 0;
  if (c->cpu) cpu_exec_meter(c->cpu, &cb, &cns, &calls, reset);
  const double hb = c->host_bytes + (double)cb, hs = c->host_s + (double)cns * 1e-9;
  if (bp_gbs) *bp_gbs = m.ns ? (double)m.bytes / (double)m.ns : 0.0;  // bytes per ns = GB/s
  if (bh_gbs) *bh_gbs = hs > 0.0 ? hb / hs / 1e9 : 0.0;
  if (reset) {
    // the three sums only: t0 / t1 / done hold their between-launch values here
    const unsigned long long z[3] = {0ull, 0ull, 0ull};
    CU(cudaMemcpy(&c->meter[0].bytes, z, sizeof(z), cudaMemcpyHostToDevice));
    c->host_bytes = c->host_s = 0.0;
  }
  return FT_OK;
}

int ft_decode_meters(ft_ctx* c, double* out, int reset) {
  if (!c || !out) return fail(FT_E_ARG, "null argument");
  CU(cudaDeviceSynchronize());
  FillMeter m[2];
  CU(cudaMemcpy(m, c->meter, sizeof(m), cudaMemcpyDeviceToHost));
  for (int i = 0; i < 2; ++i) {
    out[3 * i + 0] = (double)m[i].bytes;
    out[3 * i + 1] = (double)m[i].ns * 1e-9;
    out[3 * i + 2] = (double)m[i].launches;
  }
  if (reset) {
    const unsigned long long z[3] = {0ull, 0ull, 0ull};
    for (int i = 0; i < 2; ++i) CU(cudaMemcpy(&c->meter[i].bytes, z, sizeof(z), cudaMemcpyHostToDevice));
  }
  return FT_OK;
}

int ft_decode_path(ft_ctx* c) { return c ? (c->fused ? FT_DECODE_FUSED : FT_DECODE_SPLIT) : fail(FT_E_ARG, "null context"); }

int ft_adapt_ratio(ft_ctx* c, ft_ratio_adapter* a, void* stream, int* changed) {
  if (!c || !a) return fail(FT_E_ARG, "null context or adapter");
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess ||
      cs != cudaStreamCaptureStatusNone)
    return fail(FT_E_STATE, "ft_adapt_ratio reads measurements back and cannot be captured");
  double bp = 0.0, bh = 0.0;
  int rc = ft_measured_bandwidths(c, &bp, &bh, 1);
  if (rc) return rc;
  rc = ft_ratio_adapter_update(a, bp, bh);
  if (rc < 0) return rc;
  if (changed) *changed = rc;
  if (rc == 1) return ft_set_ratio(c, a->r_num, a->r_den, stream);
  return FT_OK;
}

int ft_get_epoch(ft_ctx* c) { return c ? c->epoch : fail(FT_E_ARG, "null context"); }

int ft_num_slots(ft_ctx* c) { return c ? c->S : fail(FT_E_ARG, "null context"); }

int ft_profile_enable(ft_ctx* c, int on) {
  if (!c) return fail(FT_E_ARG, "null context");
  c->prof.on = on != 0;
  return FT_OK;
}

int ft_profile_read(ft_ctx* c, double* total_ms, uint64_t* launches, int reset) {
  if (!c) return fail(FT_E_ARG, "null context");
  CU(cudaDeviceSynchronize());
  for (int k = 0; k < FT_K_COUNT; ++k) {
    double ms = 0.0;
    for (auto& p : c->prof.rec[k]) {
      float x = 0.f;
      CU(cudaEventElapsedTime(&x, p.first, p.second));
      ms += x;
    }
    if (total_ms) total_ms[k] = ms;
    if (launches) launches[k] = c->prof.rec[k].size();
  }
  if (reset) c->prof.reset();
  return FT_OK;
}

int ft_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, uint32_t* status, void* stream) {
  if (!logits || !ids || !w) return fail(FT_E_ARG, "null pointer");
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopK || k > E)
    return fail(FT_E_ARG, "bad routing shape T=%d E=%d k=%d", T, E, k);
  CU(launch_route(logits, T, E, k, ids, w, status, nullptr, static_cast<cudaStream_t>(stream)));
  return FT_OK;
}

}  // extern "C"
