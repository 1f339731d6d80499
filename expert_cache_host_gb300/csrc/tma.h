// Tensor Memory Accelerator helpers: bulk copies global -> shared completed
// on an mbarrier, bounded mbarrier waits, and host-side tensor-map encoding
// through the driver entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ft {

// Wall-clock bound of one mbarrier wait: a wait that has not completed after
// this long is declared failed (the caller records FT_ST_TIMEOUT and winds
// down).  Once a thread has seen a failed wait it passes give_up = true so
// later waits try once and return, keeping the kernel's exit prompt.
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// A ring stage read with ordinary shared-memory loads is refilled by TMA, which
// writes through the async proxy: order this thread's reads before any later
// async-proxy write of the stage (write-after-read across proxies).  Without
// it a slow load can still be pending when the refill lands.
__device__ __forceinline__ void proxy_fence_reads() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Ordinary shared-memory writes that a TMA store will read: make them visible
// to the async proxy first (read-after-write across proxies).
__device__ __forceinline__ void proxy_fence_writes() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch.  pdl_wait: block until the grid this one
// depends on (the previous kernel in the stream, when launched with
// programmatic stream serialization) has completed and its writes are
// visible; a no-op otherwise.  pdl_trigger: let the dependent grid launch now
// (it still waits with pdl_wait before using this grid's results).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Plain arrival (count 1) on a barrier of this CTA.
__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(a), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with parity `parity` to complete.  The clock is
// read once every 64 tries only, so a wait that ends soon costs no timer reads.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, bool give_up = false) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try(a, parity)) return true;
  if (give_up) return false;
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(a, parity)) return true;
    if ((it & 63u) == 0) {
      const uint64_t t = global_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kWaitNs) {
        return false;
      }
    }
  }
}

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// 2-D tiled tensor copy of one box at coordinates (x, y).
__device__ __forceinline__ void tensor_g2s_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled store of one box from shared memory at coordinates (x, y) (x and
// y >= 0); bulk-group completion (commit, then wait before reusing the source).
__device__ __forceinline__ void tensor_s2g_2d(const CUtensorMap* map, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N committed bulk groups of this thread still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until every committed bulk group of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 3-D tiled tensor copy of one box at coordinates (x, y, z).
__device__ __forceinline__ void tensor_g2s_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 4-D tiled tensor copy of one box at coordinates (x, y, z, w).
__device__ __forceinline__ void tensor_g2s_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// Host: encode a tiled tensor map (returns false if the driver refuses it).
// swizzle128 selects the 128-byte swizzle layout (inner box extent must then be 128 bytes).
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, char* msg, size_t msg_len,
                       bool swizzle128 = false);

}  // namespace ft
