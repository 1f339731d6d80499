// Decode expert kernel: routed SwiGLU experts for a few tokens, HBM-bound.
//
// For every resident expert of the step (a "group": the routes that chose it,
// built by the control kernel) and every chunk c of FC = 32 rows of the
// intermediate dimension f, one CTA computes
//     h[t, i] = silu(W_gate[i] . x_t) * (W_up[i] . x_t)        i in chunk c
//     ypart[route(t), c, :] = W_down[:, chunk c] . h[t, chunk c]
// with fp32 accumulation.  Splitting f this way needs no grid-wide barrier
// between the gate/up and the down projection; the per-chunk partial sums are
// reduced in a fixed order by the merge kernel, so results are deterministic.
//
// Data movement (warp-specialised): a producer warp streams the CTA's weights
// through a ring of NS 16 KB shared-memory stages with the Tensor Memory
// Accelerator, each stage guarded by a "full" mbarrier (TMA transaction
// bytes) and an "empty" mbarrier (one arrival per consumer warp).
//  - gate/up tiles: 32 rows x 256 columns boxes of a 4-D tensor map over the
//    arena (d, f, {gate, up}, slot); a consumer thread owns one row and 16
//    columns of every column block, so it accumulates its row over all blocks
//    in registers and one 16-lane reduction per row finishes the dot product;
//  - down tiles: 256 rows x 32 columns boxes of a 3-D map (f, d, slot).
// The ring runs from the gate/up tiles straight into the down tiles.  Every
// mbarrier wait is bounded; a wait that runs out records FT_ST_TIMEOUT and
// the kernel carries on to a bounded drain, so it always terminates.
// The kernel waits for the previous kernel of the stream before its first load
// (so it may be launched as a programmatic dependent where no other kernel
// needs the SMs meanwhile); with one token the hidden row is fetched beside
// the group values, and the route ids only after the gate/up pass.
// The page's activation is not named; SwiGLU is the one of the served model
// families (FreeToken article, section "核心亮点").
#include <math.h>

#include "decode_bf16.cuh"
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int FC = kDecodeChunk;           // 32 rows of f per CTA
constexpr int kConsumers = 512;            // 16 consumer warps
constexpr int kThreads = kConsumers + 32;  // + 1 producer warp
constexpr int kTokBatch = 4;               // tokens per pass over the weights
constexpr int NS = 5;                      // ring stages
constexpr int kTile = 16384;               // bytes per stage
constexpr int kXPre = 2;                   // uint4 of a hidden row per consumer (d <= 8192)

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}

struct Layout {
  size_t ring, full, empty, xs, gu, hs, rs, total;
};

__host__ __device__ inline Layout smem_layout(int d) {
  Layout L{};
  L.ring = 0;
  L.full = L.ring + (size_t)NS * kTile;
  L.empty = L.full + 8 * NS;
  L.xs = (L.empty + 8 * NS + 15) / 16 * 16;
  L.gu = L.xs + (size_t)kTokBatch * d * 2;           // [2][FC][kTokBatch] row sums
  L.hs = L.gu + sizeof(float) * 2 * FC * kTokBatch;  // [kTokBatch][FC]
  L.rs = L.hs + sizeof(float) * kTokBatch * FC;      // [kTokBatch]
  L.total = L.rs + sizeof(int) * kTokBatch;
  return L;
}

__global__ void __launch_bounds__(kThreads, 2)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmap_gu, const __grid_constant__ CUtensorMap tmap_wd,
                       DecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char dyn[];
  const int d = a.d, f = a.f;
  const Layout Ly = smem_layout(d);
  unsigned char* ring = dyn + Ly.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + Ly.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(dyn + Ly.empty);
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn + Ly.xs);  // [kTokBatch][d]
  float* gu = reinterpret_cast<float*>(dyn + Ly.gu);        // [2][FC][kTokBatch]
  float* hs = reinterpret_cast<float*>(dyn + Ly.hs);        // [kTokBatch][FC]
  int* rs = reinterpret_cast<int*>(dyn + Ly.rs);            // [kTokBatch]

  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  // Everything below reads what earlier kernels of the stream wrote.
  pdl_wait();
  // One token (decode): every route reads hidden row 0, so its copy can start
  // now, beside the loads of the group values.
  const bool one_tok = a.T == 1;
  uint4 xpre[kXPre];
  if (one_tok && tid < kConsumers) {
    const uint4* src = reinterpret_cast<const uint4*>(a.hidden);
#pragma unroll
    for (int j = 0; j < kXPre; ++j) {
      const int i = tid + j * kConsumers;
      if (i < d / 8) xpre[j] = ld_nc_early(src + i);
    }
  }
  // Fetch every per-group value at once (one memory round trip before the
  // first TMA issue); the group arrays hold at least max_groups (+1) entries,
  // so these loads are in bounds for every g of the grid.
  const int n_groups = a.counts[5];
  const int is_new = a.select != 0 ? a.group_new[g] : 0;
  const int slot = a.group_slot[g];
  const int r0 = a.group_off[g], r1 = a.group_off[g + 1];
  if (g >= n_groups) return;
  // select 1: only experts resident before the step; 2: only those it installed
  if (a.select != 0 && (is_new != 0) != (a.select == 2)) return;
  if ((unsigned)slot >= (unsigned)a.S) {
    if (tid == 0) atomicOr(a.status, FT_ST_BAD_SLOT);
    return;
  }
  const int n_batches = (r1 - r0 + kTokBatch - 1) / kTokBatch;
  const int cb_n = d / 256;           // column blocks per gate (or up) matrix
  const int P1 = 2 * cb_n;            // gate/up tiles per batch
  const int NTL = P1 + d / 256;       // + down tiles (256 rows each)
  const int total = n_batches * NTL;  // tiles over all token batches

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (tid >= kConsumers) {
    // ---------------- producer warp ----------------
    if (tid == kConsumers) {
      bool late = false;
      int s = 0;
      uint32_t ph = 0;
      for (int n = 0, i = 0; n < total; ++n) {
        if (n >= NS && !mbar_wait(&empty[s], ph ^ 1u, late)) late = true;
        unsigned char* dst = ring + s * kTile;
        mbar_expect_tx(&full[s], kTile);
        if (i < P1) {
          const int m = i < cb_n ? 0 : 1, cb = i - m * cb_n;
          tensor_g2s_4d(dst, &tmap_gu, cb * 256, c * FC, m, slot, &full[s]);
        } else {
          tensor_g2s_3d(dst, &tmap_wd, c * FC, (i - P1) * 256, slot, &full[s]);
        }
        if (++i == NTL) i = 0;
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
      // drain: the last use of every stage must have landed before the CTA exits
      for (int k = 0; k < NS && k < total; ++k) {
        const int n = total - 1 - k;
        if (!mbar_wait(&full[n % NS], (uint32_t)((n / NS) & 1), late)) late = true;
      }
      if (late) atomicOr(a.status, FT_ST_TIMEOUT);
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int lane = tid & 31;
  // gate/up tile (32 rows x 512 B): thread = row rl, columns 8cq..8cq+7 and 128+8cq..
  // down tile (256 rows x 64 B): thread = quarter q of rows tid/4 and 128 + tid/4
  // (lanes of a quarter-warp read 128 contiguous bytes: no bank conflicts)
  const int rl = tid >> 4, cq = tid & 15;
  const int rowq = tid >> 2, q = tid & 3;
  const int n_chunks = f / FC;
  bool late = false;
  int s = 0;
  uint32_t ph = 0;
  auto release = [&]() {
    proxy_fence_reads();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
  };

  if (one_tok) {
    // the one token's row in every batch row, for every batch (the first
    // barrier of the batch loop publishes it)
    for (int t = 0; t < kTokBatch; ++t) {
      uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * d);
#pragma unroll
      for (int j = 0; j < kXPre; ++j) {
        const int i = tid + j * kConsumers;
        if (i < d / 8) dst[i] = xpre[j];
      }
    }
  }
  for (int b = 0; b < n_batches; ++b) {
    const int tb = r0 + b * kTokBatch;
    const int nt = min(kTokBatch, r1 - tb);
    // route ids of the batch: needed only for the partial-sum rows, so they
    // reach shared memory after the gate/up pass
    const int my_route = tid < nt ? a.group_routes[tb + tid] : 0;
    consumer_sync();  // previous batch done with xs / rs / hs
    if (!one_tok) {
      for (int t = 0; t < nt; ++t) {
        const int tok = a.group_routes[tb + t] / a.k;
        const uint4* src = reinterpret_cast<const uint4*>(a.hidden + (size_t)tok * d);
        uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * d);
        for (int i = tid; i < d / 8; i += kConsumers) dst[i] = src[i];
      }
    }
    consumer_sync();

    float acc[2][kTokBatch];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) acc[m][t] = 0.f;

    // gate (m = 0) then up (m = 1) column blocks
#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll 1
      for (int cb = 0; cb < cb_n; ++cb) {
        if (!mbar_wait(&full[s], ph, late)) late = true;
        const unsigned char* buf = ring + s * kTile + rl * 512 + cq * 16;
        const uint4 w0 = *reinterpret_cast<const uint4*>(buf);
        const uint4 w1 = *reinterpret_cast<const uint4*>(buf + 256);
        release();
        const uint16_t* xp = xs + cb * 256 + cq * 8;
#pragma unroll
        for (int t = 0; t < kTokBatch; ++t) {
          if (t < nt) {
            const uint4 x0 = *reinterpret_cast<const uint4*>(xp + (size_t)t * d);
            const uint4 x1 = *reinterpret_cast<const uint4*>(xp + (size_t)t * d + 128);
            acc[m][t] = dot8(w1, x1, dot8(w0, x0, acc[m][t]));
          }
        }
      }
    }
    // row sums: 16 lanes per row
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) {
        float v = acc[m][t];
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        if (cq == 0 && t < nt) gu[(m * FC + rl) * kTokBatch + t] = v;
      }
    if (tid < nt) rs[tid] = my_route;
    consumer_sync();
    if (tid < FC * kTokBatch) {
      const int row = tid % FC, t = tid / FC;
      if (t < nt) {
        const float gs = gu[(0 * FC + row) * kTokBatch + t], us = gu[(1 * FC + row) * kTokBatch + t];
        hs[t * FC + row] = gs / (1.f + expf(-gs)) * us;
      }
    }
    consumer_sync();

    // down projection: 256 rows per tile, 4 threads per row, 2 rows per thread
#pragma unroll 1
    for (int j = 0; j < d / 256; ++j) {
      if (!mbar_wait(&full[s], ph, late)) late = true;
      const unsigned char* buf = ring + s * kTile + tid * 16;
      const uint4 w0 = *reinterpret_cast<const uint4*>(buf);
      const uint4 w1 = *reinterpret_cast<const uint4*>(buf + 8192);
      release();
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) {
        if (t < nt) {
          const float4* hp = reinterpret_cast<const float4*>(hs + t * FC + q * 8);
          const float4 h0 = hp[0], h1 = hp[1];
          float v0 = dot8h(w0, h0, h1, 0.f), v1 = dot8h(w1, h0, h1, 0.f);
          v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
          v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
          v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
          v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
          if (q == 0) {
            float* yp = a.ypart + ((size_t)rs[t] * n_chunks + c) * d + j * 256 + rowq;
            yp[0] = v0;
            yp[128] = v1;
          }
        }
      }
    }
  }
  if (late) atomicOr(a.status, FT_ST_TIMEOUT);
}

}  // namespace

size_t decode_bf16_smem_bytes(int d) { return smem_layout(d).total; }

cudaError_t launch_decode_experts(const DecodeArgs& a, cudaStream_t st) {
  if (a.dtype != FT_DTYPE_BF16) return cudaErrorNotSupported;
  if (a.d > 8192 || a.d % 256 || a.f % FC || !a.tmap_wd || !a.tmap_gu) return cudaErrorInvalidValue;
  dim3 grid(a.f / FC, a.max_groups), block(kThreads);
  const size_t smem = decode_bf16_smem_bytes(a.d);
  static thread_local int configured_dev = -1;
  static thread_local size_t configured_smem = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev || configured_smem < smem) {
    cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
    configured_smem = smem;
  }
  if (!a.pdl) {
    decode_bf16_kernel<<<grid, block, smem, st>>>(*a.tmap_gu, *a.tmap_wd, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(cfg, attr, grid, block, smem, st);
  return cudaLaunchKernelEx(&cfg, decode_bf16_kernel, *a.tmap_gu, *a.tmap_wd, a);
}

}  // namespace ft
