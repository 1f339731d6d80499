// Top-k routing of one token by one warp (device function shared by the
// routing kernel and the fused route + control kernel).
//
// Each token picks k of its E routed experts (FreeToken article, section
// "为什么个人跑 MoE 这么难": e.g. 6 of 256 per layer); routing itself is kept
// exact and unmodified (section "与相关工作").  Order: larger logit first,
// equal logits to the lower expert index.  Weights: softmax over the E logits
// renormalised over the k chosen, which is exp(l_j - l_top) / sum over the
// chosen -- the full softmax denominator cancels.
//
// Each lane holds PER_LANE = ceil(E/32) logits in registers (coalesced
// loads); k rounds of a warp arg-max pick the experts.  NaN logits count as
// -inf and set FT_ST_NAN.
#pragma once
#include <math.h>

#include "ft_internal.h"

namespace ft {

__device__ __forceinline__ bool route_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Route token row `row` (E logits); lanes j < k write ids[j], w[j] (and
// ids2[j] if given, e.g. a shared-memory copy); if hist is given, every chosen
// expert is counted in it.
template <int PER_LANE>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int32_t* __restrict__ ids,
                                            float* __restrict__ w, uint32_t* __restrict__ status,
                                            int32_t* __restrict__ hist, int32_t* ids2 = nullptr) {
  const int lane = threadIdx.x & 31;
  float v[PER_LANE];
  bool nan_seen = false;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = row[e];
      if (isnan(x)) {
        nan_seen = true;
        x = -INFINITY;
      }
    }
    v[i] = x;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0 && status) atomicOr(status, FT_ST_NAN);
  unsigned taken = 0;
  float my_val = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && route_better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (route_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_val = bv;
      my_id = bi;
    }
  }
  float top = __shfl_sync(0xffffffffu, my_val, 0);
  float ex = lane < k ? expf(my_val - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    ids[lane] = my_id;
    if (ids2) ids2[lane] = my_id;
    w[lane] = ex / sum;
    if (hist) atomicAdd(&hist[my_id], 1);
  }
}

}  // namespace ft
