// MXFP4 arithmetic helpers of the decode expert kernels (split and fused):
// e2m1 codes (two per byte, element 2i in the low nibble) times an e8m0 scale
// per 32 consecutive elements of a row (OCP Microscaling v1.0).  A group's
// products with f16 activations accumulate in HFMA2 chains (exact e2m1
// values, products <= 6|x|), the group sum is widened to fp32 and multiplied
// by the exact power of two.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ft {

// Exact 2^(E-127) for an e8m0 byte (E = 255 is NaN, E = 0 the subnormal 2^-127).
__device__ __forceinline__ float e8m0(unsigned e) {
  return e == 255u ? __int_as_float(0x7FC00000) : (e ? __int_as_float((int)(e << 23)) : __int_as_float(0x00400000));
}

// Four code bytes -> four f16x2 pairs (low nibble -> low half).
__device__ __forceinline__ void e2m1x8(unsigned w, unsigned& p0, unsigned& p1, unsigned& p2, unsigned& p3) {
  asm("{ .reg .b8 a0, a1, a2, a3; mov.b32 {a0, a1, a2, a3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a0; cvt.rn.f16x2.e2m1x2 %1, a1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, a2; cvt.rn.f16x2.e2m1x2 %3, a3; }"
      : "=r"(p0), "=r"(p1), "=r"(p2), "=r"(p3)
      : "r"(w));
}

__device__ __forceinline__ __half2 h2(unsigned v) { return *reinterpret_cast<__half2*>(&v); }

// Shared-memory position of activation word i (an f16 pair) of a token row:
// the four 16-byte chunks of each 16-word piece are rotated by (piece / 2),
// so the 16 pieces of a column block read chunk c from all 32 banks (two
// wavefronts) instead of two bank groups.
__device__ __forceinline__ int xs_swz(int i) {
  const int piece = i >> 4, c = (i >> 2) & 3;
  return (piece << 4) | (((c + (piece >> 1)) & 3) << 2) | (i & 3);
}

// Sum over one 32-element group: 16 code bytes (w) against 16 f16x2 activation
// pairs (x[0..3] as four uint4), returned in fp32 (unscaled).
__device__ __forceinline__ float group_dot(const uint4 w, const uint4* x) {
  __half2 a0 = __float2half2_rn(0.f), a1 = __float2half2_rn(0.f);
  const unsigned ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    unsigned p0, p1, p2, p3;
    e2m1x8(ww[i], p0, p1, p2, p3);
    const uint4 xv = x[i];
    if (i < 2) {
      a0 = __hfma2(h2(p0), h2(xv.x), a0);
      a0 = __hfma2(h2(p1), h2(xv.y), a0);
      a0 = __hfma2(h2(p2), h2(xv.z), a0);
      a0 = __hfma2(h2(p3), h2(xv.w), a0);
    } else {
      a1 = __hfma2(h2(p0), h2(xv.x), a1);
      a1 = __hfma2(h2(p1), h2(xv.y), a1);
      a1 = __hfma2(h2(p2), h2(xv.z), a1);
      a1 = __hfma2(h2(p3), h2(xv.w), a1);
    }
  }
  const float2 f0 = __half22float2(a0), f1 = __half22float2(a1);
  return (f0.x + f0.y) + (f1.x + f1.y);
}

// Power-of-two range scale for the f16 copy of h: for the largest |h| of a
// chunk (one token, 32 rows of f), `up` = 2^(8-e) brings it into [2^8, 2^9)
// (e its binary exponent), so that h*up keeps f16's full precision and the
// down projection's products with e2m1 values (|v| <= 6), summed 16 at a time
// in f16, stay far below the f16 range whatever the weight scales; `down` =
// 2^(e-8) undoes it exactly on the fp32 partial sums.  Zero, subnormal or
// non-finite maxima take 1.
__device__ __forceinline__ void h_range_scale(float mx, float& up, float& down) {
  const unsigned eb = (__float_as_uint(mx) >> 23) & 255u;  // biased exponent
  if (!(mx > 0.f) || eb == 0u || eb == 255u) {
    up = down = 1.f;
    return;
  }
  const int e = (int)eb - 127;  // -126 .. 127
  if (e >= -118) {
    up = __int_as_float((127 + 8 - e) << 23);    // 2^(8-e), biased exponent 8 .. 253
    down = __int_as_float((127 - 8 + e) << 23);  // 2^(e-8), biased exponent 1 .. 246
  } else {  // 2^(8-e) would leave the fp32 range: scale by 2^126 only
    up = __int_as_float(253 << 23);
    down = __int_as_float(1 << 23);
  }
}

// bf16 pair -> f16 pair (the activations' f16 copy)
__device__ __forceinline__ unsigned bf2_to_h2(unsigned v) {
  const __half2 hv = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  return *reinterpret_cast<const unsigned*>(&hv);
}

}  // namespace ft
