// Partial-sum merge.
//
// FreeToken article, section "设计 1" Decode bullet: the CPU and the GPU each
// compute a partial sum over their experts and the two are merged exactly,
// with no algorithmic approximation.  Here the CPU-side sum arrives as a
// float32 buffer `partial` (NULL = 0), and the GPU side is the weighted sum of
// the expert outputs of the routes that have a slot:
//     out[t] = partial[t] + sum_j [slot_ids[t,j] >= 0] w[t,j] * sum_c ypart[t*k+j, c]
// A block owns 32 float4 columns of one token; its 8 warps-rows split the k
// routes, each summing the chunk partials of its routes, and the final sum
// over routes runs in a fixed order, so the result is deterministic.
#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kCols = 32;  // float4 columns per block
constexpr int kRows = 8;   // route lanes per block

__global__ void __launch_bounds__(kCols* kRows)
    merge_kernel(const float4* __restrict__ ypart, int n_chunks, const int32_t* __restrict__ slot_ids,
                 const float* __restrict__ w, const float4* __restrict__ partial, float4* __restrict__ out, int k,
                 int d4) {
  __shared__ float4 red[kRows][kCols];
  const int t = blockIdx.y;
  const int col = threadIdx.x & (kCols - 1), jl = threadIdx.x / kCols;
  const int i = blockIdx.x * kCols + col;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i < d4) {
    for (int j = jl; j < k; j += kRows) {
      const int r = t * k + j;
      if (slot_ids[r] < 0) continue;
      const float wr = w[r];
      const float4* y = ypart + (size_t)r * n_chunks * d4 + i;
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      int c = 0;
      for (; c + 4 <= n_chunks; c += 4) {
        float4 v0 = y[(size_t)c * d4], v1 = y[(size_t)(c + 1) * d4], v2 = y[(size_t)(c + 2) * d4],
               v3 = y[(size_t)(c + 3) * d4];
        s.x += v0.x; s.y += v0.y; s.z += v0.z; s.w += v0.w;
        s.x += v1.x; s.y += v1.y; s.z += v1.z; s.w += v1.w;
        s.x += v2.x; s.y += v2.y; s.z += v2.z; s.w += v2.w;
        s.x += v3.x; s.y += v3.y; s.z += v3.z; s.w += v3.w;
      }
      for (; c < n_chunks; ++c) {
        float4 v = y[(size_t)c * d4];
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
      }
      acc.x = fmaf(wr, s.x, acc.x);
      acc.y = fmaf(wr, s.y, acc.y);
      acc.z = fmaf(wr, s.z, acc.z);
      acc.w = fmaf(wr, s.w, acc.w);
    }
  }
  red[jl][col] = acc;
  __syncthreads();
  if (jl == 0 && i < d4) {
    float4 o = partial ? partial[(size_t)t * d4 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
      o.x += red[q][col].x;
      o.y += red[q][col].y;
      o.z += red[q][col].z;
      o.w += red[q][col].w;
    }
    out[(size_t)t * d4 + i] = o;
  }
}

}  // namespace

cudaError_t launch_merge(const float* ypart, int n_chunks, const int32_t* slot_ids, const float* w,
                         const float* partial, float* out, int T, int k, int d, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int d4 = d / 4;
  dim3 grid((d4 + kCols - 1) / kCols, T), block(kCols * kRows);
  merge_kernel<<<grid, block, 0, st>>>(reinterpret_cast<const float4*>(ypart), n_chunks, slot_ids, w,
                                       reinterpret_cast<const float4*>(partial), reinterpret_cast<float4*>(out), k,
                                       d4);
  return cudaGetLastError();
}

}  // namespace ft
