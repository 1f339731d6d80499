// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "../../include/ft_moe.h"

struct CUtensorMap_st;

namespace ft {

constexpr int kCountsLen = 8;     // n, hits, m, q, cpu, n_groups, now, 0
constexpr int kCountersPerLayer = 6;  // hits, misses, fills, cpu, evictions, steps
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxSlots = 32768;
constexpr int kMaxKmax = 1024;
constexpr int kControlThreads = 1024;

// Rows of the intermediate dimension f handled by one decode work unit
// (bf16 experts / MXFP4 experts).
constexpr int kDecodeChunk = 32;
constexpr int kDecodeChunkFp4 = 32;

// Per-layer fixed-shape step buffers (device).
struct LayerBufs {
  int32_t* ids;
  float* w;
  int32_t* slot_ids;
  int32_t* uniq;
  int32_t* hit_list;
  int32_t* fetch;
  int32_t* victims;
  int32_t* evicted;
  int32_t* cpu_list;
  int32_t* counts;
  int32_t* group_slot;
  int32_t* group_new;  // 1 if the group's expert is installed by this step's fill
  int32_t* group_off;
  int32_t* group_routes;
  const int32_t* ids_src;  // routes of the last step: ids, or the caller's array (ft_cache_control)
  int last_T;  // T of the last step (host-side record, -1 = none)
};

struct ControlArgs {
  int layer, E, n_routes, S, K_max;
  int fill_order;  // FT_FILL_ORDER_*
  const long long* ratio;  // device [2]: r_num, r_den of r = BP/BH (set at init or by ft_set_ratio)
  // Fused routing: when logits ([T, E] fp32) is given, the kernel first routes
  // the T tokens into ids_out / w_out ([T, k]) and then reads ids = ids_out.
  const float* logits;
  int T, k;
  int32_t* ids_out;
  float* w_out;
  const int32_t* ids;
  int32_t* slot_of;
  int32_t* expert_of;
  uint32_t* last_use;
  uint32_t* now;
  uint32_t* status;
  unsigned long long* counters;  // this layer's row
  int32_t* slot_ids;
  int32_t* uniq;
  int32_t* hit_list;
  int32_t* fetch;
  int32_t* victims;
  int32_t* evicted;
  int32_t* cpu_list;
  int32_t* counts;
  int32_t* group_slot;
  int32_t* group_new;
  int32_t* group_off;
  int32_t* group_routes;
};

// Shared memory the control kernel needs for S slots.
size_t control_smem_bytes(int S);
cudaError_t launch_control(const ControlArgs& a, cudaStream_t st);

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, uint32_t* status,
                         int32_t* hist, cudaStream_t st);

// Link rate of the decode fill, accumulated on the device: bytes copied and
// the summed spans (first CTA start to last CTA end, ns) of the launches that
// copied something.  t0 / t1 / done are one launch's working values (t0 =
// ~0, t1 = 0, done = 0 between launches).
struct FillMeter {
  unsigned long long t0, t1, bytes, ns, launches;
  unsigned int done, pad;
};

// Fill: copy counts[3] experts fetch[i] (global ids, pool offset id*Bx) into
// arena slot victims[i]; adds the launch to *meter.
cudaError_t launch_fill(const uint8_t* pool_dev, uint8_t* arena, const int32_t* counts, const int32_t* fetch,
                        const int32_t* victims, size_t Bx, int S, int E_tot, uint32_t* status, FillMeter* meter,
                        int grid, cudaStream_t st);

// Read one 16-byte word of every 4 KB of the mapped host pool from the GPU
// (pays the first-access cost of every page at start-up).
cudaError_t launch_touch(const uint8_t* pool_dev, size_t bytes, int* sink, int grid, cudaStream_t st);

struct DecodeArgs {
  const uint8_t* arena;  // slot s at arena + s*Bx
  size_t Bx;
  int S, d, f, k, dtype;
  int max_groups;
  const int32_t* counts;
  const int32_t* group_slot;
  const int32_t* group_off;
  const int32_t* group_routes;
  const uint16_t* hidden;  // [T, d] bf16
  float* ypart;            // [T*k][f/kDecodeChunk][d]
  uint32_t* status;
  const CUtensorMap_st* tmap_wd;  // 3-D map (f, d, slot) over the arena's down projections
  const CUtensorMap_st* tmap_gu;  // 4-D map (d, f, {gate, up}, slot) over the arena's gate/up projections
  // Group selection, so that experts resident before the step can run while
  // the step's fill is still in flight: 0 = every group; 1 = groups with
  // group_new[g] == 0; 2 = groups with group_new[g] != 0.
  const int32_t* group_new;
  int select;
  int T;    // tokens of the step
  int pdl;  // launch as a programmatic dependent of the previous kernel
};
cudaError_t launch_decode_experts(const DecodeArgs& a, cudaStream_t st);
// MXFP4 experts; ypart is [T*k][f/kDecodeChunkFp4][d]; tokens = T of the step.
cudaError_t launch_decode_experts_mxfp4(const DecodeArgs& a, int tokens, cudaStream_t st);

// Fused decode layer (bf16 or MXFP4): the step's fill and all of its experts in one
// cooperative launch (decode_layer.cu).  CTAs [0, n_fill) fill first, then
// every CTA takes (expert, 32-row chunk) work items from a device-wide
// counter; ready[i] receives the step's clock once fetch entry i is in its
// slot; fill_done[i] counts the fill CTAs done with entry i (0 between
// launches).
struct LayerArgs {
  DecodeArgs d;
  const int4* pool;  // device view of the mapped host pool
  const int32_t* fetch;
  const int32_t* victims;
  int E_tot;
  int n_fill;  // fill CTAs
  int ns;      // ring stages of a compute CTA
  uint32_t* ready;
  unsigned int* fill_done;
  FillMeter* meter;   // the fill CTAs' link rate
  FillMeter* xmeter;  // the resident-expert phase: bytes, span from the first CTA start to the last resident item end
  unsigned int* sched;  // [2]: next work item, CTAs done (both 0 between launches; the last CTA out resets them)
};
// Ring stages that fit one CTA per SM at hidden size d (0: none).
// Ring stages of a fused-kernel CTA when ctas_per_sm of them share an SM (0: none fit).
int decode_layer_ring_stages(int d, int max_groups, int smem_optin, int ctas_per_sm, int dtype);
int decode_layer_ctas_per_sm();  // CTAs per SM the kernel is built for (its register bound)
cudaError_t decode_layer_max_blocks_per_sm(int d, int ns, int max_groups, int* out, int dtype);
cudaError_t launch_decode_layer(const LayerArgs& la, int grid, cudaStream_t st);

// out[t] = partial[t] + sum_j [slot_ids >= 0] w[t,j] * sum_c ypart[t*k+j][c]
// Launch attributes for programmatic dependent launch: the kernel may start
// while the previous kernel of the stream runs and calls pdl_wait() before it
// touches anything that kernel (or an earlier one) writes or reads.
inline void pdl_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// ratio[0] = r_num, ratio[1] = r_den, stream-ordered (capturable).
cudaError_t launch_set_ratio(long long* ratio, long long r_num, long long r_den, cudaStream_t st);

cudaError_t launch_merge(const float* ypart, int n_chunks, const int32_t* slot_ids, const float* w,
                         const float* partial, float* out, int T, int k, int d, cudaStream_t st);

// Record the calling thread's error message (read back by ft_last_error) and
// return `code`.
int record_error(int code, const char* fmt, ...);

// Event pairs around launches, for ft_profile_read.  Records nothing while
// the stream is being captured.
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> rec[FT_K_COUNT];

  cudaEvent_t get() {
    cudaEvent_t e = nullptr;
    if (!pool.empty()) {
      e = pool.back();
      pool.pop_back();
    } else if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
    }
    return e;
  }
  // Returns the start event, or nullptr when not recording.
  cudaEvent_t begin(cudaStream_t st) {
    if (!on) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
    cudaEvent_t b = get();
    if (b) cudaEventRecord(b, st);
    return b;
  }
  void end(cudaStream_t st, int kind, cudaEvent_t b) {
    if (!b) return;
    cudaEvent_t e = get();
    if (!e) return;
    cudaEventRecord(e, st);
    rec[kind].push_back({b, e});
  }
  void reset() {
    for (auto& v : rec) {
      for (auto& p : v) {
        pool.push_back(p.first);
        pool.push_back(p.second);
      }
      v.clear();
    }
  }
  void destroy() {
    reset();
    for (auto e : pool) cudaEventDestroy(e);
    pool.clear();
  }
};

// CPU expert executor (cpu_experts.cu): the routes of a decode step that got
// no slot run on the host from the pool; their partial sum reaches the device
// in stream order (fork after the control kernel, join before the merge).
struct CpuExec;
int cpu_exec_create(CpuExec** out, int threads, const uint8_t* pool_host, int L, int E, int k, int d, int f,
                    int dtype, size_t Bx, int t_max);
void cpu_exec_destroy(CpuExec* ex);
cudaError_t cpu_exec_fork(CpuExec* ex, int layer, int T, const int32_t* slot_ids, const int32_t* ids, const float* w,
                          const uint16_t* hidden, cudaStream_t st, Profiler& prof);
cudaError_t cpu_exec_join(CpuExec* ex, cudaStream_t st);
const float* cpu_exec_partial(const CpuExec* ex);
// Expert bytes the executor's host functions read and the nanoseconds they
// spent computing, since the last call with reset != 0.
void cpu_exec_meter(CpuExec* ex, unsigned long long* bytes, unsigned long long* ns, unsigned long long* calls,
                    int reset);

}  // namespace ft
