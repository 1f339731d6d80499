// Partial-sum merge.
//
// FreeToken article, section "设计 1" Decode bullet: the CPU and the GPU each
// compute a partial sum over their experts and the two are merged exactly,
// with no algorithmic approximation.  Here the CPU-side sum arrives as a
// float32 buffer `partial` (NULL = 0), and the GPU side is the weighted sum of
// the expert outputs of the routes that have a slot:
//     out[t] = partial[t] + sum_j [slot_ids[t,j] >= 0] w[t,j] * sum_c ypart[t*k+j, c]
// in a fixed order (j ascending, c ascending), 16-byte loads and stores.
#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    merge_kernel(const float4* __restrict__ ypart, int n_chunks, const int32_t* __restrict__ slot_ids,
                 const float* __restrict__ w, const float4* __restrict__ partial, float4* __restrict__ out, int k,
                 int d4) {
  const int t = blockIdx.y;
  const int i = blockIdx.x * kThreads + threadIdx.x;
  if (i >= d4) return;
  float4 acc = partial ? partial[(size_t)t * d4 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int r = t * k + j;
    if (slot_ids[r] < 0) continue;
    const float wr = w[r];
    const float4* y = ypart + (size_t)r * n_chunks * d4 + i;
    float4 s = y[0];
    for (int c = 1; c < n_chunks; ++c) {
      float4 v = y[(size_t)c * d4];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    acc.x = fmaf(wr, s.x, acc.x);
    acc.y = fmaf(wr, s.y, acc.y);
    acc.z = fmaf(wr, s.z, acc.z);
    acc.w = fmaf(wr, s.w, acc.w);
  }
  out[(size_t)t * d4 + i] = acc;
}

}  // namespace

cudaError_t launch_merge(const float* ypart, int n_chunks, const int32_t* slot_ids, const float* w,
                         const float* partial, float* out, int T, int k, int d, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int d4 = d / 4;
  dim3 grid((d4 + kThreads - 1) / kThreads, T), block(kThreads);
  merge_kernel<<<grid, block, 0, st>>>(reinterpret_cast<const float4*>(ypart), n_chunks, slot_ids, w,
                                       reinterpret_cast<const float4*>(partial), reinterpret_cast<float4*>(out), k,
                                       d4);
  return cudaGetLastError();
}

}  // namespace ft
