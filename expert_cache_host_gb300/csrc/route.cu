// Top-k routing kernel: one warp per token (see route_warp.cuh for the
// order, the weights and the FreeToken sections they follow).
#include "route_warp.cuh"

namespace ft {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxPerLane = kMaxExperts / 32;

template <int PER_LANE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                 float* __restrict__ w, uint32_t* __restrict__ status, int32_t* __restrict__ hist) {
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token<PER_LANE>(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k, status, hist);
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
