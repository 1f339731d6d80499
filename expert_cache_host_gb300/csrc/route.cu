// Top-k routing kernel.
//
// Each token picks k of its E routed experts (FreeToken article, section
// "为什么个人跑 MoE 这么难": e.g. 6 of 256 per layer); routing itself is kept
// exact and unmodified (section "与相关工作").  Order: larger logit first,
// equal logits to the lower expert index.  Weights: softmax over the E logits
// renormalised over the k chosen, which is exp(l_j - l_top) / sum over the
// chosen -- the full softmax denominator cancels.
//
// One warp per token; each lane holds E/32 logits in registers (coalesced
// loads), and k rounds of a warp arg-max pick the experts.
#include <math.h>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxPerLane = kMaxExperts / 32;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int PER_LANE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                 float* __restrict__ w, uint32_t* __restrict__ status, int32_t* __restrict__ hist) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
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
      if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
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
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = ex / sum;
    if (hist) atomicAdd(&hist[my_id], 1);
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, uint32_t* status,
                         int32_t* hist, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  dim3 grid((T + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
  int per = (E + 31) / 32;
  if (per <= 1)
    route_kernel<1><<<grid, block, 0, st>>>(logits, T, E, k, ids, w, status, hist);
  else if (per <= 4)
    route_kernel<4><<<grid, block, 0, st>>>(logits, T, E, k, ids, w, status, hist);
  else if (per <= 8)
    route_kernel<8><<<grid, block, 0, st>>>(logits, T, E, k, ids, w, status, hist);
  else
    route_kernel<kMaxPerLane><<<grid, block, 0, st>>>(logits, T, E, k, ids, w, status, hist);
  return cudaGetLastError();
}

}  // namespace ft
