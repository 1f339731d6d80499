// Partial-sum merge (FreeToken article, section "设计 1", Decode bullet).
//
// Contract: the routes a decode step leaves to the host side contribute one
// float32 buffer `partial` [T, d] (NULL means zero); this kernel adds the
// weighted outputs of the routes that run on the GPU, so that the layer's
// output is the same sum the unsplit MoE would give:
//     out[t] = partial[t] + sum_j [slot_ids[t,j] >= 0] w[t,j] * sum_c ypart[t*k+j, c]
// A block owns 4 float4 columns of one token; its 64 thread rows split the
// k * n_chunks (route, chunk) partials of those columns (each row issues up
// to 8 loads together, so the merge costs about one L2 round trip), and the
// rows are then summed in a fixed order (eight runs of eight rows, then the
// eight run sums), so the result is deterministic.
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int kCols = 4;   // float4 columns per block
constexpr int kRows = 64;  // (route, chunk) lanes per block
constexpr int kUn = 8;     // loads in flight per lane
constexpr int kRun = 8;    // rows per run of the final sum

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
    for (int p0 = row; p0 < npairs; p0 += kUn * kRows) {
      float4 v[kUn];
      float wv[kUn];
#pragma unroll
      for (int u = 0; u < kUn; ++u) {
        const int p = p0 + u * kRows;
        wv[u] = 0.f;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p < npairs) {
          // the three loads are independent (ypart is allocated for every
          // route); a route without a slot then contributes exactly nothing
          const int j = p / n_chunks, c = p - j * n_chunks, r = t * k + j;
          const int sid = __ldg(slot_ids + r);
          const float wr = __ldg(w + r);
          const float4 y = ypart[((size_t)r * n_chunks + c) * d4 + i];
          if (sid >= 0) {
            wv[u] = wr;
            v[u] = y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUn; ++u) {
        acc.x = fmaf(wv[u], v[u].x, acc.x);
        acc.y = fmaf(wv[u], v[u].y, acc.y);
        acc.z = fmaf(wv[u], v[u].z, acc.z);
        acc.w = fmaf(wv[u], v[u].w, acc.w);
      }
    }
  }
  red[row][col] = acc;
  __syncthreads();
  // each run of kRun rows into its first row, in row order
  if (row < kRows / kRun) {
    float4 s = red[row * kRun][col];
#pragma unroll
    for (int q = 1; q < kRun; ++q) {
      const float4 x = red[row * kRun + q][col];
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    red[row * kRun][col] = s;
  }
  __syncthreads();
  if (row == 0 && i < d4) {
    float4 o = partial ? partial[(size_t)t * d4 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kRows / kRun; ++q) {
      const float4 x = red[q * kRun][col];
      o.x += x.x;
      o.y += x.y;
      o.z += x.z;
      o.w += x.w;
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
