// Decode expert kernel: routed SwiGLU experts for a few tokens, HBM-bound.
//
// For every resident expert of the step (a "group": the routes that chose it,
// built by the control kernel) and every chunk c of kDecodeChunk rows of the
// intermediate dimension f, one CTA computes
//     h[t, i] = silu(W_gate[i] . x_t) * (W_up[i] . x_t)        i in chunk c
//     ypart[route(t), c, :] = W_down[:, chunk c] . h[t, chunk c]
// with fp32 accumulation.  Splitting f this way needs no grid-wide barrier
// between the gate/up and down projections; the per-chunk partial sums are
// reduced in a fixed order by the merge kernel, so results are deterministic.
// Weights are read once per step with 16-byte coalesced loads (gate/up rows
// are d-contiguous; a down chunk is 2*kDecodeChunk contiguous bytes per row).
// The page's activation is not named; SwiGLU is the one of the served models
// (FreeToken article, section "核心亮点": Qwen3.6-35B-A3B, DeepSeek-V4-Flash).
#include <math.h>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int FC = kDecodeChunk;        // 32 rows of f per CTA
constexpr int kThreads = 256;           // 8 warps
constexpr int kRowsPerWarp = FC / 8;    // 4
constexpr int kTokBatch = 4;            // tokens per pass over the weights

__device__ __forceinline__ int4 ldg_stream(const void* p) {
  int4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf_lo(unsigned v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(unsigned v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float dot8(const int4 w, const int4 x) {
  float s = bf_lo(w.x) * bf_lo(x.x);
  s = fmaf(bf_hi(w.x), bf_hi(x.x), s);
  s = fmaf(bf_lo(w.y), bf_lo(x.y), s);
  s = fmaf(bf_hi(w.y), bf_hi(x.y), s);
  s = fmaf(bf_lo(w.z), bf_lo(x.z), s);
  s = fmaf(bf_hi(w.z), bf_hi(x.z), s);
  s = fmaf(bf_lo(w.w), bf_lo(x.w), s);
  s = fmaf(bf_hi(w.w), bf_hi(x.w), s);
  return s;
}

__device__ __forceinline__ float dot8h(const int4 w, const float* h) {
  float s = bf_lo(w.x) * h[0];
  s = fmaf(bf_hi(w.x), h[1], s);
  s = fmaf(bf_lo(w.y), h[2], s);
  s = fmaf(bf_hi(w.y), h[3], s);
  s = fmaf(bf_lo(w.z), h[4], s);
  s = fmaf(bf_hi(w.z), h[5], s);
  s = fmaf(bf_lo(w.w), h[6], s);
  s = fmaf(bf_hi(w.w), h[7], s);
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kThreads) decode_bf16_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  const int d = a.d, f = a.f;
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn);                        // [kTokBatch][d]
  float* hs = reinterpret_cast<float*>(dyn + (size_t)kTokBatch * d * 2);  // [kTokBatch][FC]
  int* rs = reinterpret_cast<int*>(hs + kTokBatch * FC);                  // [kTokBatch] routes

  const int c = blockIdx.x, g = blockIdx.y;
  if (g >= a.counts[5]) return;
  const int slot = a.group_slot[g];
  if ((unsigned)slot >= (unsigned)a.S) {
    if (threadIdx.x == 0) atomicOr(a.status, FT_ST_BAD_SLOT);
    return;
  }
  const int r0 = a.group_off[g], r1 = a.group_off[g + 1];
  const size_t df = (size_t)d * f;
  const uint16_t* Wg = reinterpret_cast<const uint16_t*>(a.arena + (size_t)slot * a.Bx);
  const uint16_t* Wu = Wg + df;
  const uint16_t* Wd = Wg + 2 * df;
  const int n_chunks = f / FC;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nit = d / 256;

  for (int tb = r0; tb < r1; tb += kTokBatch) {
    const int nt = min(kTokBatch, r1 - tb);
    __syncthreads();  // xs/hs reuse
    if (threadIdx.x < nt) rs[threadIdx.x] = a.group_routes[tb + threadIdx.x];
    for (int t = 0; t < nt; ++t) {
      const int tok = a.group_routes[tb + t] / a.k;
      const int4* src = reinterpret_cast<const int4*>(a.hidden + (size_t)tok * d);
      int4* dst = reinterpret_cast<int4*>(xs + (size_t)t * d);
      for (int i = threadIdx.x; i < d / 8; i += kThreads) dst[i] = src[i];
    }
    __syncthreads();

    // gate/up rows of this chunk: warp wid owns rows wid + 8*rr
    float ag[kRowsPerWarp][kTokBatch], au[kRowsPerWarp][kTokBatch];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) ag[rr][t] = au[rr][t] = 0.f;
    const size_t row0 = (size_t)c * FC + wid;
    for (int it = 0; it < nit; ++it) {
      const int col = it * 256 + lane * 8;
      int4 wg[kRowsPerWarp], wu[kRowsPerWarp];
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        wg[rr] = ldg_stream(Wg + (row0 + 8 * rr) * d + col);
        wu[rr] = ldg_stream(Wu + (row0 + 8 * rr) * d + col);
      }
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) {
        if (t < nt) {
          const int4 x = *reinterpret_cast<const int4*>(xs + (size_t)t * d + col);
#pragma unroll
          for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            ag[rr][t] += dot8(wg[rr], x);
            au[rr][t] += dot8(wu[rr], x);
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) {
        if (t < nt) {
          float gs = warp_sum(ag[rr][t]);
          float us = warp_sum(au[rr][t]);
          if (lane == 0) hs[t * FC + wid + 8 * rr] = gs / (1.f + expf(-gs)) * us;
        }
      }
    __syncthreads();

    // down projection of this chunk: 4 threads per row of W_down, 64 rows per pass
    const int quad = threadIdx.x & 3, rowq = threadIdx.x >> 2;
    float hq[kTokBatch][8];
#pragma unroll
    for (int t = 0; t < kTokBatch; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) hq[t][i] = t < nt ? hs[t * FC + quad * 8 + i] : 0.f;
    const uint16_t* wdc = Wd + (size_t)c * FC + quad * 8;
    constexpr int kUnroll = 8;
    for (int rb = 0; rb < d; rb += 64 * kUnroll) {
      int4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = rb + u * 64 + rowq;
        w[u] = r < d ? ldg_stream(wdc + (size_t)r * f) : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = rb + u * 64 + rowq;
#pragma unroll
        for (int t = 0; t < kTokBatch; ++t) {
          if (t < nt) {
            float p = dot8h(w[u], hq[t]);
            p += __shfl_xor_sync(0xffffffffu, p, 1);
            p += __shfl_xor_sync(0xffffffffu, p, 2);
            if (quad == 0 && r < d) a.ypart[((size_t)rs[t] * n_chunks + c) * d + r] = p;
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_decode_experts(const DecodeArgs& a, cudaStream_t st) {
  if (a.dtype != FT_DTYPE_BF16) return cudaErrorNotSupported;
  dim3 grid(a.f / FC, a.max_groups), block(kThreads);
  size_t smem = (size_t)kTokBatch * a.d * 2 + kTokBatch * FC * 4 + kTokBatch * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  decode_bf16_kernel<<<grid, block, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace ft
