// Decode fill: copy the fetched experts from the host pool into their slots.
//
// FreeToken article, section "设计 1" Decode bullet: the q* filled experts
// enter the GPU cache, run on the GPU and stay resident for reuse.  The
// fetch list and its length are device-resident (written by the control
// kernel), so a copy-engine memcpy would need their values on the host.  This
// kernel reads them on the device instead and streams the bytes with 16-byte
// loads from the pool, which is registered as mapped pinned memory and read
// over the host link (NVLink-C2C on GB300); the launch has a fixed shape and
// can be captured in a CUDA graph.
#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kFillThreads = 512;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kFillThreads)
    fill_kernel(const int4* __restrict__ pool, int4* __restrict__ arena, const int32_t* __restrict__ counts,
                const int32_t* __restrict__ fetch, const int32_t* __restrict__ victims, size_t bx16, int S,
                int E_tot, uint32_t* __restrict__ status) {
  const int q = counts[3];
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  for (int i = 0; i < q; ++i) {
    const int u = fetch[i], s = victims[i];
    if ((unsigned)u >= (unsigned)E_tot || (unsigned)s >= (unsigned)S) {
      if (tid == 0) atomicOr(status, FT_ST_BAD_SLOT);
      continue;
    }
    const int4* src = pool + (size_t)u * bx16;
    int4* dst = arena + (size_t)s * bx16;
    size_t v = tid;
    for (; v + (kUnroll - 1) * nthreads < bx16; v += kUnroll * nthreads) {
      int4 r[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) r[j] = src[v + j * nthreads];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) dst[v + j * nthreads] = r[j];
    }
    for (; v < bx16; v += nthreads) dst[v] = src[v];
  }
}

}  // namespace

cudaError_t launch_fill(const uint8_t* pool_dev, uint8_t* arena, const int32_t* counts, const int32_t* fetch,
                        const int32_t* victims, size_t Bx, int S, int E_tot, uint32_t* status, int grid,
                        cudaStream_t st) {
  // The fill needs no shared memory, but the expert kernel that runs beside it
  // needs ~100 KB per CTA: keep the SMs in the largest shared-memory split, or
  // an SM running a fill CTA cannot take an expert CTA until it drains.
  static thread_local int configured_for = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_for != dev) {
    cudaError_t e = cudaFuncSetAttribute(fill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  fill_kernel<<<grid, kFillThreads, 0, st>>>(reinterpret_cast<const int4*>(pool_dev), reinterpret_cast<int4*>(arena),
                                             counts, fetch, victims, Bx / 16, S, E_tot, status);
  return cudaGetLastError();
}

}  // namespace ft
