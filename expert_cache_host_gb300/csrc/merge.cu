// Partial-sum merge.
//
// FreeToken article, section "设计 1" Decode bullet: the CPU and the GPU each
// compute a partial sum over their experts and the two are merged exactly,
// with no algorithmic approximation.  Here the CPU-side sum arrives as a
// float32 buffer `partial` (NULL = 0), and the GPU side is the weighted sum of
// the expert outputs of the routes that have a slot:
//     out[t] = partial[t] + sum_j [slot_ids[t,j] >= 0] w[t,j] * sum_c ypart[t*k+j, c]
// A block owns 8 float4 columns of one token; its 32 thread rows split the
// k * n_chunks (route, chunk) partials of those columns (each row issues its
// loads together, so the merge costs about one L2 round trip), and the rows
// are then summed in a fixed order, so the result is deterministic.
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int kCols = 8;   // float4 columns per block
constexpr int kRows = 32;  // (route, chunk) lanes per block

__global__ void __launch_bounds__(kCols* kRows)
    merge_kernel(const float4* __restrict__ ypart, int n_chunks, const int32_t* __restrict__ slot_ids,
                 const float* __restrict__ w, const float4* __restrict__ partial, float4* __restrict__ out, int k,
                 int d4) {
  __shared__ float4 red[kRows][kCols];
  // the next kernel (the next layer's routing) may start now; this one waits
  // for the experts' partial sums
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int col = threadIdx.x % kCols, row = threadIdx.x / kCols;
  const int i = blockIdx.x * kCols + col;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i < d4) {
    const int npairs = k * n_chunks;
    for (int p0 = row; p0 < npairs; p0 += 4 * kRows) {
      float4 v[4];
      float wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int p = p0 + u * kRows;
        wv[u] = 0.f;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p < npairs) {
          const int j = p / n_chunks, c = p - j * n_chunks, r = t * k + j;
          if (slot_ids[r] >= 0) {
            wv[u] = w[r];
            v[u] = ypart[((size_t)r * n_chunks + c) * d4 + i];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x = fmaf(wv[u], v[u].x, acc.x);
        acc.y = fmaf(wv[u], v[u].y, acc.y);
        acc.z = fmaf(wv[u], v[u].z, acc.z);
        acc.w = fmaf(wv[u], v[u].w, acc.w);
      }
    }
  }
  red[row][col] = acc;
  __syncthreads();
  if (row == 0 && i < d4) {
    float4 o = partial ? partial[(size_t)t * d4 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
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
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(cfg, attr, grid, block, 0, st);
  return cudaLaunchKernelEx(&cfg, merge_kernel, reinterpret_cast<const float4*>(ypart), n_chunks, slot_ids, w,
                            reinterpret_cast<const float4*>(partial), reinterpret_cast<float4*>(out), k, d4);
}

}  // namespace ft
