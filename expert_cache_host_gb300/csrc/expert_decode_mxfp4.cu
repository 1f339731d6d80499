// Decode expert kernel for MXFP4 experts (e2m1 codes, one e8m0 scale per 32
// consecutive elements of a row; OCP Microscaling v1.0), HBM-bound.
//
// Same work split and data movement as the bf16 decode kernel: one CTA per
// (resident expert, chunk of FC = 32 rows of f), a producer warp streaming
// 16 KB stages through a TMA ring with full/empty mbarriers, 16 consumer warps.
//  - gate/up codes: 32 rows x 256 bytes boxes of a 4-D map (d/2, f, {g,u}, slot),
//    two column blocks per stage; the chunk's gate/up scales (32 rows x d/32
//    bytes each) arrive once by two 1-D bulk copies;
//  - down codes: 256 rows x 16 bytes boxes of a 3-D map (f/2, d, slot), four per
//    stage (1024 rows); each row's one down scale for this chunk is read
//    directly, a stage ahead (the 64 chunks of an expert share those sectors).
// Arithmetic: a 16-byte piece of a row is 32 elements = exactly one scale
// group.  cvt.rn.f16x2.e2m1x2 turns each code byte into two exact f16 values;
// the group's products with the f16 activations accumulate in two chains of
// eight HFMA2, the group sum is widened to fp32 and multiplied by the exact
// power of two 2^(E-127), and groups accumulate in fp32.  The intermediate h
// is held in f16 for the down projection, scaled per token and chunk by a
// power of two that puts its largest value in [2^8, 2^9) (undone exactly on
// the fp32 partial sums), so that its range never depends on the weights'
// scales.  (The page keeps DSV4's experts in
// native MXFP4, "bit-identical" to the checkpoint: section "评估结果".)
#include <cuda_fp16.h>
#include <math.h>

#include "decode_bf16.cuh"
#include "decode_mxfp4.cuh"
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int FC = kDecodeChunkFp4;        // 32 rows of f per CTA
constexpr int kConsumers = 512;
constexpr int kThreads = kConsumers + 32;
constexpr int kTile = 16384;
constexpr int kXPre = 4;  // uint4 of a hidden row per consumer (d <= 16384)

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

struct Layout {
  size_t ring, full, empty, scbar, sc, xs, gu, hs, rs, hd, total;
};

template <int TB, int NS>
__host__ __device__ inline Layout smem_layout(int d) {
  Layout L{};
  L.ring = 0;
  L.full = L.ring + (size_t)NS * kTile;
  L.empty = L.full + 8 * NS;
  L.scbar = L.empty + 8 * NS;
  L.sc = (L.scbar + 8 + 127) / 128 * 128;                   // [2][FC][d/32] scale bytes
  L.xs = L.sc + (size_t)2 * FC * (d / 32);                  // [TB][d/2] f16x2 pairs
  L.gu = L.xs + (size_t)TB * (d / 2) * 4;                   // [2 halves][2][FC][TB] fp32 row sums
  L.hs = L.gu + sizeof(float) * 4 * FC * TB;                // [TB][FC/2] f16x2
  L.rs = L.hs + (size_t)TB * (FC / 2) * 4;                  // [TB]
  L.hd = L.rs + sizeof(int) * TB;                           // [TB] 2^(e-8) of each token's h range scale
  L.total = L.hd + sizeof(float) * TB;
  return L;
}

template <int TB, int NS>
__global__ void __launch_bounds__(kThreads, 2)
    decode_mxfp4_kernel(const __grid_constant__ CUtensorMap tmap_gu, const __grid_constant__ CUtensorMap tmap_wd,
                        DecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char dyn[];
  const int d = a.d, f = a.f;
  const Layout Ly = smem_layout<TB, NS>(d);
  unsigned char* ring = dyn + Ly.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + Ly.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(dyn + Ly.empty);
  uint64_t* scbar = reinterpret_cast<uint64_t*>(dyn + Ly.scbar);
  const unsigned char* sc = dyn + Ly.sc;
  unsigned* xs = reinterpret_cast<unsigned*>(dyn + Ly.xs);
  float* gu = reinterpret_cast<float*>(dyn + Ly.gu);
  unsigned* hs = reinterpret_cast<unsigned*>(dyn + Ly.hs);
  float* hdown = reinterpret_cast<float*>(dyn + Ly.hd);
  int* rs = reinterpret_cast<int*>(dyn + Ly.rs);

  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  // Everything below reads what earlier kernels of the stream wrote.
  pdl_wait();
  // One token (TB == 1 is launched for one-token steps): every route reads
  // hidden row 0, so its copy can start now, beside the group values.
  uint4 xpre[kXPre];
  if (TB == 1 && tid < kConsumers) {
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
  const size_t df = (size_t)d * f;
  const unsigned char* ex = a.arena + (size_t)slot * a.Bx;
  const unsigned char* sc_gate = ex + 3 * (df / 2);                 // [f][d/32]
  const unsigned char* sc_down = sc_gate + 2 * (df / 32);           // [d][f/32]
  const int n_batches = (r1 - r0 + TB - 1) / TB;
  const int cb_n = d / 512;              // 256-byte column blocks per gate/up row
  const int gst = (cb_n + 1) / 2;        // gate (or up) stages: two column blocks each
  const int nbox = d / 256;              // 256-row down boxes
  const int dst = (nbox + 3) / 4;        // down stages: four boxes (1024 rows) each
  const int NTL = 2 * gst + dst;         // stages per token batch
  const int total = n_batches * NTL;
  const int sc_row = d / 32;             // scale bytes per gate/up row

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_init(scbar, 1);
    mbar_init_fence();
  }
  __syncthreads();

  if (tid >= kConsumers) {
    if (tid == kConsumers) {
      bool late = false;
      const uint32_t scb = FC * sc_row;
      mbar_expect_tx(scbar, 2 * scb);
      bulk_g2s(dyn + Ly.sc, sc_gate + (size_t)c * FC * sc_row, scb, scbar);
      bulk_g2s(dyn + Ly.sc + scb, sc_gate + df / 32 + (size_t)c * FC * sc_row, scb, scbar);
      int s = 0;
      uint32_t ph = 0;
      for (int n = 0, i = 0; n < total; ++n) {
        if (n >= NS && !mbar_wait(&empty[s], ph ^ 1u, late)) late = true;
        unsigned char* dstp = ring + s * kTile;
        if (i < 2 * gst) {
          const int m = i < gst ? 0 : 1, cb0 = 2 * (i - m * gst), nb = min(2, cb_n - cb0);
          mbar_expect_tx(&full[s], nb * (kTile / 2));
          for (int b = 0; b < nb; ++b)
            tensor_g2s_4d(dstp + b * (kTile / 2), &tmap_gu, (cb0 + b) * 256, c * FC, m, slot, &full[s]);
        } else {
          const int j = i - 2 * gst, box0 = 4 * j, nb = min(4, nbox - box0);
          mbar_expect_tx(&full[s], nb * (kTile / 4));
          for (int b = 0; b < nb; ++b)
            tensor_g2s_3d(dstp + b * (kTile / 4), &tmap_wd, c * (FC / 2), (box0 + b) * 256, slot, &full[s]);
        }
        if (++i == NTL) i = 0;
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
      for (int k = 0; k < NS && k < total; ++k) {
        const int n = total - 1 - k;
        if (!mbar_wait(&full[n % NS], (uint32_t)((n / NS) & 1), late)) late = true;
      }
      if (!mbar_wait(scbar, 0, late)) late = true;
      if (late) atomicOr(a.status, FT_ST_TIMEOUT);
    }
    return;
  }

  const int lane = tid & 31;
  // gate/up: thread = 16-byte column piece p of rows 2rp and 2rp + 1 of the
  // stage's column block hb, so a piece's 32 activations are loaded once per
  // stage for two rows
  const int p = tid & 15, rp = (tid >> 4) & 15, hb = tid >> 8;
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

  if (TB == 1) {
    // the one token's row, for every batch (the first barrier of the batch
    // loop publishes it)
#pragma unroll
    for (int j = 0; j < kXPre; ++j) {
      const int i = tid + j * kConsumers;
      if (i < d / 8) {
        xs[xs_swz(4 * i + 0)] = bf2_to_h2(xpre[j].x);
        xs[xs_swz(4 * i + 1)] = bf2_to_h2(xpre[j].y);
        xs[xs_swz(4 * i + 2)] = bf2_to_h2(xpre[j].z);
        xs[xs_swz(4 * i + 3)] = bf2_to_h2(xpre[j].w);
      }
    }
  }
  for (int b = 0; b < n_batches; ++b) {
    const int tb = r0 + b * TB;
    const int nt = min(TB, r1 - tb);
    // route ids of the batch: needed only for the partial-sum rows, so they
    // reach shared memory after the gate/up pass
    const int my_route = tid < nt ? a.group_routes[tb + tid] : 0;
    consumer_sync();
    if (TB != 1) {
      for (int t = 0; t < nt; ++t) {
        const int tok = a.group_routes[tb + t] / a.k;
        const unsigned* src = reinterpret_cast<const unsigned*>(a.hidden + (size_t)tok * d);  // bf16 pairs
        for (int i = tid; i < d / 2; i += kConsumers) xs[(size_t)t * (d / 2) + xs_swz(i)] = bf2_to_h2(src[i]);
      }
    }
    consumer_sync();
    if (b == 0 && !mbar_wait(scbar, 0, late)) late = true;

    float acc[2][2][TB];  // [gate/up][row 2rp + i][token]
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int t = 0; t < TB; ++t) acc[m][i][t] = 0.f;

#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll 1
      for (int k2 = 0; k2 < gst; ++k2) {
        if (!mbar_wait(&full[s], ph, late)) late = true;
        const int cb = 2 * k2 + hb;
        uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
        if (cb < cb_n) {
          const unsigned char* buf = ring + s * kTile + hb * (kTile / 2) + (2 * rp) * 256 + p * 16;
          w0 = *reinterpret_cast<const uint4*>(buf);
          w1 = *reinterpret_cast<const uint4*>(buf + 256);
        }
        release();
        if (cb < cb_n) {
          const int grp = cb * 16 + p;  // scale group (and global 16-word piece) of this thread
          const float s0 = e8m0(sc[(m * FC + 2 * rp) * sc_row + grp]);
          const float s1 = e8m0(sc[(m * FC + 2 * rp + 1) * sc_row + grp]);
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            if (t < nt) {
              const unsigned* xrow = xs + (size_t)t * (d / 2) + grp * 16;
              uint4 xv[4];
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4)
                xv[c4] = *reinterpret_cast<const uint4*>(xrow + (((c4 + (grp >> 1)) & 3) << 2));
              acc[m][0][t] = fmaf(group_dot(w0, xv), s0, acc[m][0][t]);
              acc[m][1][t] = fmaf(group_dot(w1, xv), s1, acc[m][1][t]);
            }
          }
        }
      }
    }
    // row sums: the 16 pieces of a row pair are 16 consecutive lanes; the two
    // column-block halves are added in the SwiGLU step
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          float v = acc[m][i][t];
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          if (p == 0 && t < nt) gu[((hb * 2 + m) * FC + 2 * rp + i) * TB + t] = v;
        }
    if (tid < nt) rs[tid] = my_route;
    consumer_sync();
    if (tid < 32 * ((FC / 2 * TB + 31) / 32)) {  // whole warps: 16 lanes per token
      const int pr = tid % (FC / 2), t = tid / (FC / 2);
      float h0 = 0.f, h1 = 0.f;
      if (t < nt) {
        auto rsum = [&](int m, int row) { return gu[((0 * 2 + m) * FC + row) * TB + t] + gu[((1 * 2 + m) * FC + row) * TB + t]; };
        const float g0 = rsum(0, 2 * pr), u0 = rsum(1, 2 * pr), g1 = rsum(0, 2 * pr + 1), u1 = rsum(1, 2 * pr + 1);
        h0 = g0 / (1.f + expf(-g0)) * u0;
        h1 = g1 / (1.f + expf(-g1)) * u1;
      }
      float mx = fmaxf(fabsf(h0), fabsf(h1));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float up, down;
      h_range_scale(mx, up, down);
      if (t < nt) {
        const __half2 hv = __floats2half2_rn(h0 * up, h1 * up);
        hs[t * (FC / 2) + pr] = *reinterpret_cast<const unsigned*>(&hv);
        if (pr == 0) hdown[t] = down;
      }
    }
    consumer_sync();

    // down: a stage holds rows 1024 j .. 1024 j + 1023 (16 bytes each, in order);
    // thread = rows tid and tid + 512 of the stage, one scale group each
    const size_t sc_step = (size_t)512 * (f / 32);  // 512 rows of scales
    const unsigned char* scd = sc_down + (size_t)tid * (f / 32) + c;
    unsigned char e0n = tid < d ? __ldg(scd) : 0, e1n = tid + 512 < d ? __ldg(scd + sc_step) : 0;
#pragma unroll 1
    for (int j = 0; j < dst; ++j) {
      const int row0 = j * 1024 + tid, row1 = row0 + 512;
      const float s0 = e8m0(e0n), s1 = e8m0(e1n);
      if (j + 1 < dst) {
        e0n = row0 + 1024 < d ? __ldg(scd + (size_t)(2 * j + 2) * sc_step) : 0;
        e1n = row1 + 1024 < d ? __ldg(scd + (size_t)(2 * j + 3) * sc_step) : 0;
      }
      if (!mbar_wait(&full[s], ph, late)) late = true;
      const unsigned char* buf = ring + s * kTile + tid * 16;
      const uint4 w0 = row0 < d ? *reinterpret_cast<const uint4*>(buf) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 w1 = row1 < d ? *reinterpret_cast<const uint4*>(buf + kTile / 2) : make_uint4(0u, 0u, 0u, 0u);
      release();
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        if (t < nt) {
          const uint4* hp = reinterpret_cast<const uint4*>(hs + t * (FC / 2));
          float* yp = a.ypart + ((size_t)rs[t] * n_chunks + c) * d;
          if (row0 < d) yp[row0] = group_dot(w0, hp) * (s0 * hdown[t]);
          if (row1 < d) yp[row1] = group_dot(w1, hp) * (s1 * hdown[t]);
        }
      }
    }
  }
  if (late) atomicOr(a.status, FT_ST_TIMEOUT);
}

template <int TB, int NS>
cudaError_t launch(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = smem_layout<TB, NS>(a.d).total;
  static thread_local int configured_dev = -1;
  static thread_local size_t configured_smem = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev || configured_smem < smem) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_mxfp4_kernel<TB, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
    configured_smem = smem;
  }
  const dim3 grid(a.f / FC, a.max_groups), block(kThreads);
  if (!a.pdl) {
    decode_mxfp4_kernel<TB, NS><<<grid, block, smem, st>>>(*a.tmap_gu, *a.tmap_wd, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(cfg, attr, grid, block, smem, st);
  return cudaLaunchKernelEx(&cfg, decode_mxfp4_kernel<TB, NS>, *a.tmap_gu, *a.tmap_wd, a);
}

}  // namespace

cudaError_t launch_decode_experts_mxfp4(const DecodeArgs& a, int tokens, cudaStream_t st) {
  if (a.d % 512 || a.d > 16384 || a.f % FC || !a.tmap_wd || !a.tmap_gu) return cudaErrorInvalidValue;
  return tokens == 1 ? launch<1, 5>(a, st) : launch<4, 3>(a, st);
}

}  // namespace ft
