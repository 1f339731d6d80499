// bf16 dot-product helpers of the decode expert kernels (HBM-bound GEMV on
// CUDA cores): bf16 pairs widened exactly to fp32 with shifts and masks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ft {

__device__ __forceinline__ float bf_lo(unsigned v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(unsigned v) { return __uint_as_float(v & 0xFFFF0000u); }

// s + sum of 8 products of bf16 weights and bf16 activations
__device__ __forceinline__ float dot8(const uint4 w, const uint4 x, float s) {
  s = fmaf(bf_lo(w.x), bf_lo(x.x), s);
  s = fmaf(bf_hi(w.x), bf_hi(x.x), s);
  s = fmaf(bf_lo(w.y), bf_lo(x.y), s);
  s = fmaf(bf_hi(w.y), bf_hi(x.y), s);
  s = fmaf(bf_lo(w.z), bf_lo(x.z), s);
  s = fmaf(bf_hi(w.z), bf_hi(x.z), s);
  s = fmaf(bf_lo(w.w), bf_lo(x.w), s);
  s = fmaf(bf_hi(w.w), bf_hi(x.w), s);
  return s;
}

// s + sum of 8 products of bf16 weights and fp32 values h0, h1
__device__ __forceinline__ float dot8h(const uint4 w, const float4 h0, const float4 h1, float s) {
  s = fmaf(bf_lo(w.x), h0.x, s);
  s = fmaf(bf_hi(w.x), h0.y, s);
  s = fmaf(bf_lo(w.y), h0.z, s);
  s = fmaf(bf_hi(w.y), h0.w, s);
  s = fmaf(bf_lo(w.z), h1.x, s);
  s = fmaf(bf_hi(w.z), h1.y, s);
  s = fmaf(bf_lo(w.w), h1.z, s);
  s = fmaf(bf_hi(w.w), h1.w, s);
  return s;
}

// 16-byte read-only load kept where it is written (not sunk past the branches
// that follow), so that it overlaps the loads issued after it.
__device__ __forceinline__ uint4 ld_nc_early(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace ft
