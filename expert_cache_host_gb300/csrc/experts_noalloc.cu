// Allocation-free variant of the decode expert step (experts + merge).
//
// Some callers cannot allocate device memory at the moment they run the
// step: a serving runtime that fixes its memory budget once at start-up and
// forbids allocation afterwards, a host framework that owns every device
// buffer through its own pool, or code running while a stream capture in
// global mode is open, where cudaMalloc is not permitted.  This entry point
// takes every input and output from the caller and keeps its scratch (route
// groups and per-chunk partial sums) in one file-scope device array of fixed
// size, so it calls no cudaMalloc, cudaFree or allocating library routine.
// The paper has no counterpart: it is an interface for such callers.
//
// The array is resolved with cudaGetSymbolAddress once per device, the first
// time the entry point runs on that device (so that first call should come
// before any stream capture).  Every call on a device shares the array and
// the array keeps the last call's contents; calls whose work overlaps on the
// GPU (for example on two concurrent streams) race on it.
#include <cstdio>
#include <mutex>

#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// One group per route that has a slot: group g = the g-th such route.
// merge_sid receives the slot ids the merge acts on: a route whose slot id is
// outside [0, S) is reported and becomes -1 there, so it adds nothing (its
// partial-sum rows are not written by this call and may hold an earlier
// call's values).
__global__ void route_groups_kernel(const int32_t* __restrict__ slot_ids, int n_routes, int S,
                                    int32_t* __restrict__ counts, int32_t* __restrict__ group_slot,
                                    int32_t* __restrict__ group_off, int32_t* __restrict__ group_routes,
                                    int32_t* __restrict__ merge_sid, uint32_t* __restrict__ status) {
  __shared__ int n;
  if (threadIdx.x == 0) n = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int r = 0; r < n_routes; ++r) {
      const int s = slot_ids[r];
      merge_sid[r] = s < S ? s : -1;
      if (s < 0) continue;
      if (s >= S) {
        atomicOr(status, FT_ST_BAD_SLOT);
        continue;
      }
      group_slot[n] = s;
      group_off[n] = n;
      group_routes[n] = r;
      ++n;
    }
    group_off[n] = n;
    for (int i = 0; i < kCountsLen; ++i) counts[i] = 0;
    counts[5] = n;
  }
}

}  // namespace

size_t noalloc_scratch_needed(int T, int k, int d, int f) {
  const size_t R = (size_t)T * k;
  const size_t small = 256 + 4 * (4 * R + 1) + 4 /*status*/;
  const size_t small_pad = (small + 255) / 256 * 256;
  return small_pad + R * (size_t)(f / kDecodeChunk) * d * sizeof(float);
}

}  // namespace ft

extern "C" int ft_decode_experts_noalloc(const void* arena_dev, int num_slots, int hidden, int inter, int top_k, int T,
                                         const int32_t* slot_ids_dev, const float* weights_dev,
                                         const uint16_t* hidden_dev, const float* partial_dev, float* out_dev,
                                         uint32_t* status_dev, void* stream) {
  using namespace ft;
  char msg[256] = "";
  auto fail = [](int code, const char* m) { return record_error(code, "%s", m); };
  if (!arena_dev || !slot_ids_dev || !weights_dev || !hidden_dev || !out_dev) return fail(FT_E_ARG, "null pointer");
  if (num_slots < 1 || T < 1 || top_k < 1 || top_k > kMaxTopK) return fail(FT_E_ARG, "bad slot count, T or top_k");
  if (hidden < 256 || hidden % 256 || hidden > 8192) return fail(FT_E_ARG, "hidden must be a multiple of 256, <= 8192");
  if (inter < kDecodeChunk || inter % kDecodeChunk) return record_error(FT_E_ARG, "inter must be a multiple of %d", kDecodeChunk);
  if (reinterpret_cast<uintptr_t>(arena_dev) % 16) return fail(FT_E_ARG, "the arena must be 16-byte aligned");
  const size_t need = noalloc_scratch_needed(T, top_k, hidden, inter);
  if (need > kStaticScratchBytes) {
    return record_error(FT_E_ARG,
                        "T*k*(inter/32)*hidden*4 bytes of partial sums (%zu bytes with route groups) exceed the "
                        "static scratch of %zu bytes",
                        need, kStaticScratchBytes);
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(FT_E_CUDA, "no usable device");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
      cudaError_t e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_scratch_addr[dev] = nullptr;
        return record_error(FT_E_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                            cudaGetErrorString(e));
      }
    }
    base = g_scratch_addr[dev];
  }
  const int R = T * top_k;
  unsigned char* p = static_cast<unsigned char*>(base);
  int32_t* counts = reinterpret_cast<int32_t*>(p);
  int32_t* group_slot = counts + 64;
  int32_t* group_off = group_slot + R;
  int32_t* group_routes = group_off + R + 1;
  int32_t* merge_sid = group_routes + R;
  uint32_t* status = status_dev ? status_dev : reinterpret_cast<uint32_t*>(merge_sid + R);
  size_t small = 256 + 4 * (4 * (size_t)R + 1) + 4;
  float* ypart = reinterpret_cast<float*>(p + (small + 255) / 256 * 256);

  const uint64_t d = hidden, f = inter;
  const size_t Bx = 6 * d * f;
  CUtensorMap tmap_wd, tmap_gu;
  {
    const uint64_t dims[3] = {f, d, (uint64_t)num_slots};
    const uint64_t strides[2] = {f * 2, Bx};
    const uint32_t box[3] = {(uint32_t)kDecodeChunk, 256, 1};
    if (!encode_tensor_map(&tmap_wd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<unsigned char*>(static_cast<const unsigned char*>(arena_dev)) + 4 * d * f, dims,
                           strides, box, msg, sizeof(msg)))
      return record_error(FT_E_CUDA, "%s", msg);
    const uint64_t dims4[4] = {d, f, 2, (uint64_t)num_slots};
    const uint64_t strides4[3] = {d * 2, d * f * 2, Bx};
    const uint32_t box4[4] = {256, (uint32_t)kDecodeChunk, 1, 1};
    if (!encode_tensor_map(&tmap_gu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(arena_dev), dims4,
                           strides4, box4, msg, sizeof(msg)))
      return record_error(FT_E_CUDA, "%s", msg);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  route_groups_kernel<<<1, 32, 0, st>>>(slot_ids_dev, R, num_slots, counts, group_slot, group_off, group_routes,
                                        merge_sid, status);
  if (cudaGetLastError() != cudaSuccess) return fail(FT_E_CUDA, "route group launch failed");
  DecodeArgs a{};
  a.arena = static_cast<const uint8_t*>(arena_dev);
  a.Bx = Bx;
  a.S = num_slots;
  a.d = hidden;
  a.f = inter;
  a.k = top_k;
  a.dtype = FT_DTYPE_BF16;
  a.max_groups = R;
  a.T = T;
  a.pdl = 1;  // no fill runs beside this launch
  a.counts = counts;
  a.group_slot = group_slot;
  a.group_off = group_off;
  a.group_routes = group_routes;
  a.hidden = hidden_dev;
  a.ypart = ypart;
  a.status = status;
  a.tmap_wd = &tmap_wd;
  a.tmap_gu = &tmap_gu;
  cudaError_t e = launch_decode_experts(a, st);
  if (e != cudaSuccess) return record_error(FT_E_CUDA, "expert launch failed: %s", cudaGetErrorString(e));
  e = launch_merge(ypart, inter / kDecodeChunk, merge_sid, weights_dev, partial_dev, out_dev, T, top_k, hidden, st);
  if (e != cudaSuccess) return record_error(FT_E_CUDA, "merge launch failed: %s", cudaGetErrorString(e));
  return FT_OK;
}
