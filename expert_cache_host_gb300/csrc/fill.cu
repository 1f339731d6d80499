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
//
// The kernel also measures the link rate it achieves (the BP of the q* ~
// m*BP/BH split): the first CTA start and the last CTA end of every launch
// that copies something are taken from %globaltimer, and the CTA that
// finishes last adds the launch's bytes and span to the context's FillMeter
// (no CTA waits for another).
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int kFillThreads = 512;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kFillThreads)
    fill_kernel(const int4* __restrict__ pool, int4* __restrict__ arena, const int32_t* __restrict__ counts,
                const int32_t* __restrict__ fetch, const int32_t* __restrict__ victims, size_t bx16, int S,
                int E_tot, uint32_t* __restrict__ status, FillMeter* __restrict__ meter) {
  const int q = counts[3];
  if (q <= 0) return;  // every CTA sees the same q: nothing to copy or measure
  if (threadIdx.x == 0) atomicMin(&meter->t0, (unsigned long long)global_ns());
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
    // batches of kUnroll loads in flight, the last one predicated: a
    // copy-one-then-the-next tail would cost a host round trip per piece
    for (size_t v = tid; v < bx16; v += kUnroll * nthreads) {
      int4 r[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j)
        if (v + j * nthreads < bx16) r[j] = src[v + j * nthreads];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j)
        if (v + j * nthreads < bx16) dst[v + j * nthreads] = r[j];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's copies are visible before its end time is taken
    atomicMax(&meter->t1, (unsigned long long)global_ns());
    __threadfence();
    if (atomicAdd(&meter->done, 1u) == gridDim.x - 1) {
      // last CTA of the launch: every other CTA's start and end are in t0 / t1
      __threadfence();
      const unsigned long long t0 = atomicAdd(&meter->t0, 0ull), t1 = atomicAdd(&meter->t1, 0ull);
      atomicAdd(&meter->bytes, (unsigned long long)q * bx16 * 16ull);
      atomicAdd(&meter->ns, t1 > t0 ? t1 - t0 : 0ull);
      atomicAdd(&meter->launches, 1ull);
      atomicExch(&meter->t0, ~0ull);
      atomicExch(&meter->t1, 0ull);
      atomicExch(&meter->done, 0u);
    }
  }
}

// One 16-byte read of every 4 KB of the mapped pool.  The first GPU access to
// a page of host memory can be far slower than later ones (measured on the
// GB300 hosts: 1 GiB regions at 7-120 GB/s on first touch, 211 GB/s after),
// so the context pays it once at start-up instead of in the first fills and
// uploads that reach each page.
__global__ void touch_kernel(const int4* __restrict__ pool, size_t n16, int* __restrict__ sink) {
  constexpr size_t kStride = 4096 / 16;
  const size_t nt = (size_t)gridDim.x * blockDim.x;
  int acc = 0;
  for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * kStride; i < n16; i += nt * kStride)
    acc ^= __ldcs(pool + i).x;
  if (acc == 0x5EED5EED) atomicAdd(sink, 1);  // keeps the loads; the value itself is never used
}

}  // namespace

cudaError_t launch_touch(const uint8_t* pool_dev, size_t bytes, int* sink, int grid, cudaStream_t st) {
  touch_kernel<<<grid, 512, 0, st>>>(reinterpret_cast<const int4*>(pool_dev), bytes / 16, sink);
  return cudaGetLastError();
}

cudaError_t launch_fill(const uint8_t* pool_dev, uint8_t* arena, const int32_t* counts, const int32_t* fetch,
                        const int32_t* victims, size_t Bx, int S, int E_tot, uint32_t* status, FillMeter* meter,
                        int grid, cudaStream_t st) {
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
                                             counts, fetch, victims, Bx / 16, S, E_tot, status, meter);
  return cudaGetLastError();
}

}  // namespace ft
