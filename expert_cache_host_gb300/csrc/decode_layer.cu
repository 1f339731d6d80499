// Fused decode layer kernel (bf16 experts): the step's fill and all of its
// routed SwiGLU experts in one cooperative launch, one CTA per SM.
//
// FreeToken article, section "设计：三大机制" 1, Decode bullet: the q filled
// experts are copied from the host pool into their cache slots and then run on
// the GPU beside the experts that were already resident.  Here the two happen
// in one grid with the SMs split by role:
//  - fill CTAs (the first n_fill) stream the fetched experts from the mapped
//    pinned pool into their victim slots, expert after expert; when the last
//    fill CTA finishes its share of fetch entry i it publishes ready[i] = the
//    step's clock (release);
//  - compute CTAs (the rest) run the same per-(expert, 32-row chunk) SwiGLU
//    GEMV as the split decode kernel -- TMA ring of 16 KB tiles, fp32
//    accumulation, one partial sum per (route, chunk) for the merge -- over a
//    persistent list of work items: first every chunk of every expert that was
//    resident before the step, then the chunks of each installed expert in
//    fill order.  Before the first tile of an installed expert the producer
//    warp waits (bounded, %globaltimer) for its ready stamp, so an installed
//    expert starts as soon as its own bytes have landed, from L2.
// The control kernel lists groups by ascending expert and the fetch list is
// ascending too, so the j-th installed group is fetch entry j.
//
// The ring keeps running across a CTA's items, so only the first tile of the
// launch pays the TMA latency; one CTA per SM leaves room for a deep ring.
// Blocks of one cooperative launch are resident together, so the waits of
// compute CTAs on fill CTAs always end; every wait is also bounded in time
// and a wait that runs out records FT_ST_TIMEOUT and carries on.
#include <math.h>

#include "decode_bf16.cuh"
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int FC = kDecodeChunk;           // 32 rows of f per item
constexpr int kConsumers = 512;            // 16 consumer warps
constexpr int kThreads = kConsumers + 32;  // + 1 producer warp
constexpr int kTokBatch = 4;               // tokens per pass over the weights
constexpr int kTile = 16384;               // bytes per ring stage
constexpr int kXPre = 2;                   // uint4 of a hidden row per consumer (d <= 8192)
constexpr int kFillUnroll = 16;            // 16-byte host loads in flight per fill thread

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Generic-proxy writes that another thread released and this thread acquired
// are made visible to this thread's later async-proxy (TMA) reads.
__device__ __forceinline__ void proxy_fence_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

struct Layout {
  size_t ring, full, empty, xs, gu, hs, rs, lists, total;
};

__host__ __device__ inline Layout smem_layout(int d, int ns, int max_groups) {
  Layout L{};
  L.ring = 0;
  L.full = L.ring + (size_t)ns * kTile;
  L.empty = L.full + 8 * (size_t)ns;
  L.xs = (L.empty + 8 * (size_t)ns + 15) / 16 * 16;
  L.gu = L.xs + (size_t)kTokBatch * d * 2;           // [2][FC][kTokBatch] row sums
  L.hs = L.gu + sizeof(float) * 2 * FC * kTokBatch;  // [kTokBatch][FC]
  L.rs = L.hs + sizeof(float) * kTokBatch * FC;      // [kTokBatch]
  L.lists = L.rs + sizeof(int) * kTokBatch;          // [2] counts, then resident / installed group lists
  L.total = L.lists + sizeof(int) * (2 + 2 * (size_t)max_groups);
  return L;
}

// ---------------------------------------------------------------- fill role

__device__ void fill_role(const LayerArgs& la) {
  const DecodeArgs& a = la.d;
  const int q = a.counts[3];
  if (q <= 0) return;  // every fill CTA sees the same q
  const uint32_t now = (uint32_t)a.counts[6];
  const int F = la.n_fill;
  FillMeter* m = la.meter;
  if (threadIdx.x == 0) atomicMin(&m->t0, (unsigned long long)global_ns());
  const size_t bx16 = a.Bx / 16;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nth = (size_t)F * blockDim.x;
  int4* arena = reinterpret_cast<int4*>(const_cast<uint8_t*>(a.arena));
  for (int i = 0; i < q; ++i) {
    const int u = la.fetch[i], s = la.victims[i];
    if ((unsigned)u < (unsigned)la.E_tot && (unsigned)s < (unsigned)a.S) {
      const int4* src = la.pool + (size_t)u * bx16;
      int4* dst = arena + (size_t)s * bx16;
      size_t v = tid;
      for (; v + (kFillUnroll - 1) * nth < bx16; v += kFillUnroll * nth) {
        int4 r[kFillUnroll];
#pragma unroll
        for (int j = 0; j < kFillUnroll; ++j) r[j] = src[v + j * nth];
#pragma unroll
        for (int j = 0; j < kFillUnroll; ++j) dst[v + j * nth] = r[j];
      }
      for (; v < bx16; v += nth) dst[v] = src[v];
    } else if (blockIdx.x == 0 && threadIdx.x == 0) {
      atomicOr(a.status, FT_ST_BAD_SLOT);
    }
    __syncthreads();  // this CTA's share of entry i is written
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(&la.fill_done[i], 1u) == (unsigned)F - 1) {
        atomicExch(&la.fill_done[i], 0u);
        __threadfence();
        atomicExch(&la.ready[i], now);  // every fill CTA's share of entry i is visible
      }
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    atomicMax(&m->t1, (unsigned long long)global_ns());
    __threadfence();
    if (atomicAdd(&m->done, 1u) == (unsigned)F - 1) {
      __threadfence();
      const unsigned long long t0 = atomicAdd(&m->t0, 0ull), t1 = atomicAdd(&m->t1, 0ull);
      atomicAdd(&m->bytes, (unsigned long long)q * a.Bx);
      atomicAdd(&m->ns, t1 > t0 ? t1 - t0 : 0ull);
      atomicAdd(&m->launches, 1ull);
      atomicExch(&m->t0, ~0ull);
      atomicExch(&m->t1, 0ull);
      atomicExch(&m->done, 0u);
    }
  }
}

// ---------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(kThreads, 1)
    decode_layer_bf16_kernel(const __grid_constant__ CUtensorMap tmap_gu, const __grid_constant__ CUtensorMap tmap_wd,
                             const LayerArgs la) {
  if ((int)blockIdx.x < la.n_fill) {
    fill_role(la);
    return;
  }
  const DecodeArgs& a = la.d;
  extern __shared__ __align__(1024) unsigned char dyn[];
  const int d = a.d, f = a.f, ns = la.ns;
  const Layout Ly = smem_layout(d, ns, a.max_groups);
  unsigned char* ring = dyn + Ly.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + Ly.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(dyn + Ly.empty);
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn + Ly.xs);  // [kTokBatch][d]
  float* gu = reinterpret_cast<float*>(dyn + Ly.gu);        // [2][FC][kTokBatch]
  float* hs = reinterpret_cast<float*>(dyn + Ly.hs);        // [kTokBatch][FC]
  int* rs = reinterpret_cast<int*>(dyn + Ly.rs);            // [kTokBatch]
  int* nlist = reinterpret_cast<int*>(dyn + Ly.lists);      // [0] resident, [1] installed
  int* res = nlist + 2;                                     // resident groups, ascending
  int* inst = res + a.max_groups;                           // installed groups = fetch order

  const int tid = threadIdx.x, lane = tid & 31;
  const int C = gridDim.x - la.n_fill, ci = blockIdx.x - la.n_fill;
  if (tid == 0) atomicMin(&la.xmeter->t0, (unsigned long long)global_ns());
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
  if (tid == kConsumers) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_init_fence();
  }
  // work lists: warp 0 splits the groups into resident and installed, in order
  if (tid < 32) {
    const int n_groups = min(a.counts[5], a.max_groups);
    int nr = 0, ni = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int g = base + lane;
      const bool in = g < n_groups;
      const bool isnew = in && a.group_new[g] != 0;
      const unsigned bn = __ballot_sync(0xffffffffu, isnew), br = __ballot_sync(0xffffffffu, in && !isnew);
      const unsigned below = (1u << lane) - 1u;
      if (isnew) inst[ni + __popc(bn & below)] = g;
      else if (in) res[nr + __popc(br & below)] = g;
      ni += __popc(bn);
      nr += __popc(br);
    }
    if (lane == 0) {
      nlist[0] = nr;
      nlist[1] = ni;
    }
  }
  __syncthreads();
  const int nr = nlist[0], ni = nlist[1];
  const int n_chunks = f / FC;
  const int total_items = (nr + ni) * n_chunks;
  const int q = a.counts[3];
  const uint32_t now = (uint32_t)a.counts[6];
  const int cb_n = d / 256;      // column blocks per gate (or up) matrix
  const int P1 = 2 * cb_n;       // gate/up tiles per token batch
  const int NTL = P1 + d / 256;  // + down tiles (256 rows each)

  // item j -> group, chunk, fill index (-1 = resident before the step)
  auto item = [&](int j, int& g, int& c, int& fi) {
    if (j < nr * n_chunks) {
      g = res[j / n_chunks];
      c = j % n_chunks;
      fi = -1;
    } else {
      const int jj = j - nr * n_chunks;
      fi = jj / n_chunks;
      g = inst[fi];
      c = jj % n_chunks;
    }
  };

  if (tid >= kConsumers) {
    // ---------------- producer warp: one ring across all of the CTA's items ----------------
    if (tid == kConsumers) {
      bool late = false;
      int s = 0, n = 0;
      uint32_t ph = 0;
      for (int j = ci; j < total_items; j += C) {
        int g, c, fi;
        item(j, g, c, fi);
        const int slot = a.group_slot[g];
        if ((unsigned)slot >= (unsigned)a.S) continue;  // consumers skip it too
        if (fi >= 0 && fi < q) {
          // the installed expert's bytes: wait for the fill CTAs' stamp
          if (ld_acquire(&la.ready[fi]) != now) {
            const uint64_t t0 = global_ns();
            while (ld_acquire(&la.ready[fi]) != now) {
              if (late || global_ns() - t0 > kWaitNs) {
                late = true;
                break;
              }
              __nanosleep(200);
            }
          }
          proxy_fence_global();
        }
        const int n_batches = (a.group_off[g + 1] - a.group_off[g] + kTokBatch - 1) / kTokBatch;
        for (int t = 0, i = 0; t < n_batches * NTL; ++t) {
          if (n >= ns && !mbar_wait(&empty[s], ph ^ 1u, late)) late = true;
          unsigned char* dst = ring + s * kTile;
          mbar_expect_tx(&full[s], kTile);
          if (i < P1) {
            const int mtx = i < cb_n ? 0 : 1, cb = i - mtx * cb_n;
            tensor_g2s_4d(dst, &tmap_gu, cb * 256, c * FC, mtx, slot, &full[s]);
          } else {
            tensor_g2s_3d(dst, &tmap_wd, c * FC, (i - P1) * 256, slot, &full[s]);
          }
          if (++i == NTL) i = 0;
          if (++s == ns) {
            s = 0;
            ph ^= 1u;
          }
          ++n;
        }
      }
      // drain: the last use of every stage must have landed before the CTA exits
      for (int k = 0; k < ns && k < n; ++k) {
        const int m = n - 1 - k;
        if (!mbar_wait(&full[m % ns], (uint32_t)((m / ns) & 1), late)) late = true;
      }
      if (late) atomicOr(a.status, FT_ST_TIMEOUT);
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int rl = tid >> 4, cq = tid & 15;   // gate/up: row rl, 16-byte columns cq and cq + 16
  const int rowq = tid >> 2, qq = tid & 3;  // down: quarter qq of rows rowq and rowq + 128
  bool late = false;
  int s = 0;
  uint32_t ph = 0;
  auto release = [&]() {
    proxy_fence_reads();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == ns) {
      s = 0;
      ph ^= 1u;
    }
  };
  if (one_tok) {
    for (int t = 0; t < kTokBatch; ++t) {
      uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * d);
#pragma unroll
      for (int j = 0; j < kXPre; ++j) {
        const int i = tid + j * kConsumers;
        if (i < d / 8) dst[i] = xpre[j];
      }
    }
  }
  // End of this CTA's share of the resident experts: the last compute CTA to
  // get there adds the phase (first compute CTA start to last resident item
  // end) and the resident bytes to xmeter.
  bool resident_done = false;
  auto close_resident = [&]() {
    resident_done = true;
    consumer_sync();
    if (tid == 0) {
      FillMeter* m = la.xmeter;
      __threadfence();
      atomicMax(&m->t1, (unsigned long long)global_ns());
      __threadfence();
      if (atomicAdd(&m->done, 1u) == (unsigned)C - 1) {
        __threadfence();
        const unsigned long long t0 = atomicAdd(&m->t0, 0ull), t1 = atomicAdd(&m->t1, 0ull);
        if (nr > 0) {
          atomicAdd(&m->bytes, (unsigned long long)nr * a.Bx);
          atomicAdd(&m->ns, t1 > t0 ? t1 - t0 : 0ull);
          atomicAdd(&m->launches, 1ull);
        }
        atomicExch(&m->t0, ~0ull);
        atomicExch(&m->t1, 0ull);
        atomicExch(&m->done, 0u);
      }
    }
  };
  for (int j = ci; j < total_items; j += C) {
    if (!resident_done && j >= nr * n_chunks) close_resident();
    int g, c, fi;
    item(j, g, c, fi);
    const int slot = a.group_slot[g];
    if ((unsigned)slot >= (unsigned)a.S) {
      if (tid == 0) atomicOr(a.status, FT_ST_BAD_SLOT);
      continue;
    }
    const int r0 = a.group_off[g], r1 = a.group_off[g + 1];
    const int n_batches = (r1 - r0 + kTokBatch - 1) / kTokBatch;
    for (int b = 0; b < n_batches; ++b) {
      const int tb = r0 + b * kTokBatch;
      const int nt = min(kTokBatch, r1 - tb);
      const int my_route = tid < nt ? a.group_routes[tb + tid] : 0;
      consumer_sync();  // the previous batch (or item) is done with xs / rs / hs
      if (!one_tok) {
        for (int t = 0; t < nt; ++t) {
          const int tok = a.group_routes[tb + t] / a.k;
          const uint4* src = reinterpret_cast<const uint4*>(a.hidden + (size_t)tok * d);
          uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * d);
          for (int i = tid; i < d / 8; i += kConsumers) dst[i] = src[i];
        }
      }
      consumer_sync();

      // gate/up: tiles 0 .. P1-1 (tile i: matrix i / cb_n, column block i % cb_n), two per
      // iteration (P1 is even) with independent product chains
      float accg[kTokBatch], accu[kTokBatch];
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) accg[t] = accu[t] = 0.f;
#pragma unroll 1
      for (int i = 0; i < P1; i += 2) {
        const int s1 = s + 1 == ns ? 0 : s + 1;
        const uint32_t ph1 = s + 1 == ns ? ph ^ 1u : ph;
        if (!mbar_wait(&full[s], ph, late)) late = true;
        if (!mbar_wait(&full[s1], ph1, late)) late = true;
        const unsigned char* b0 = ring + s * kTile + rl * 512 + cq * 16;
        const unsigned char* b1 = ring + s1 * kTile + rl * 512 + cq * 16;
        const uint4 wa0 = *reinterpret_cast<const uint4*>(b0), wa1 = *reinterpret_cast<const uint4*>(b0 + 256);
        const uint4 wb0 = *reinterpret_cast<const uint4*>(b1), wb1 = *reinterpret_cast<const uint4*>(b1 + 256);
        release();
        release();
        const int ma = i / cb_n, mb = (i + 1) / cb_n;
        const uint16_t* xa = xs + (i - ma * cb_n) * 256 + cq * 8;
        const uint16_t* xb = xs + (i + 1 - mb * cb_n) * 256 + cq * 8;
#pragma unroll
        for (int t = 0; t < kTokBatch; ++t) {
          if (t < nt) {
            const uint4 xa0 = *reinterpret_cast<const uint4*>(xa + (size_t)t * d);
            const uint4 xa1 = *reinterpret_cast<const uint4*>(xa + (size_t)t * d + 128);
            const uint4 xb0 = *reinterpret_cast<const uint4*>(xb + (size_t)t * d);
            const uint4 xb1 = *reinterpret_cast<const uint4*>(xb + (size_t)t * d + 128);
            const float pa = dot8(wa1, xa1, dot8(wa0, xa0, 0.f));
            const float pb = dot8(wb1, xb1, dot8(wb0, xb0, 0.f));
            accg[t] += (ma == 0 ? pa : 0.f) + (mb == 0 ? pb : 0.f);
            accu[t] += (ma == 1 ? pa : 0.f) + (mb == 1 ? pb : 0.f);
          }
        }
      }
      // row sums: 16 lanes per row
#pragma unroll
      for (int t = 0; t < kTokBatch; ++t) {
        float vg = accg[t], vu = accu[t];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          vg += __shfl_xor_sync(0xffffffffu, vg, o);
          vu += __shfl_xor_sync(0xffffffffu, vu, o);
        }
        if (cq == 0 && t < nt) {
          gu[(0 * FC + rl) * kTokBatch + t] = vg;
          gu[(1 * FC + rl) * kTokBatch + t] = vu;
        }
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
      // down: 256 rows per tile, two tiles per iteration (and one left over when d / 256 is odd)
#pragma unroll 1
      for (int jd = 0; jd < cb_n; jd += 2) {
        const bool two = jd + 1 < cb_n;
        const int s1 = s + 1 == ns ? 0 : s + 1;
        const uint32_t ph1 = s + 1 == ns ? ph ^ 1u : ph;
        if (!mbar_wait(&full[s], ph, late)) late = true;
        if (two && !mbar_wait(&full[s1], ph1, late)) late = true;
        const unsigned char* b0 = ring + s * kTile + tid * 16;
        const unsigned char* b1 = ring + s1 * kTile + tid * 16;
        const uint4 wa0 = *reinterpret_cast<const uint4*>(b0), wa1 = *reinterpret_cast<const uint4*>(b0 + 8192);
        uint4 wb0 = make_uint4(0, 0, 0, 0), wb1 = wb0;
        if (two) {
          wb0 = *reinterpret_cast<const uint4*>(b1);
          wb1 = *reinterpret_cast<const uint4*>(b1 + 8192);
        }
        release();
        if (two) release();
#pragma unroll
        for (int t = 0; t < kTokBatch; ++t) {
          if (t < nt) {
            const float4* hp = reinterpret_cast<const float4*>(hs + t * FC + qq * 8);
            const float4 h0 = hp[0], h1 = hp[1];
            float v0 = dot8h(wa0, h0, h1, 0.f), v1 = dot8h(wa1, h0, h1, 0.f);
            float v2 = dot8h(wb0, h0, h1, 0.f), v3 = dot8h(wb1, h0, h1, 0.f);
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
              v0 += __shfl_xor_sync(0xffffffffu, v0, o);
              v1 += __shfl_xor_sync(0xffffffffu, v1, o);
              v2 += __shfl_xor_sync(0xffffffffu, v2, o);
              v3 += __shfl_xor_sync(0xffffffffu, v3, o);
            }
            if (qq == 0) {
              float* yp = a.ypart + ((size_t)rs[t] * n_chunks + c) * d + jd * 256 + rowq;
              yp[0] = v0;
              yp[128] = v1;
              if (two) {
                yp[256] = v2;
                yp[384] = v3;
              }
            }
          }
        }
      }
    }
  }
  if (!resident_done) close_resident();
  if (late) atomicOr(a.status, FT_ST_TIMEOUT);
}

}  // namespace

int decode_layer_ring_stages(int d, int max_groups, int smem_optin) {
  const size_t fixed = smem_layout(d, 0, max_groups).total + 16 * 16 + 1024;
  if ((size_t)smem_optin <= fixed) return 0;
  return (int)std::min<size_t>(12, ((size_t)smem_optin - fixed) / (kTile + 16));
}

cudaError_t launch_decode_layer(const LayerArgs& la, int grid, cudaStream_t st) {
  const DecodeArgs& a = la.d;
  if (a.dtype != FT_DTYPE_BF16) return cudaErrorNotSupported;
  if (a.d > 8192 || a.d % 256 || a.f % FC || !a.tmap_wd || !a.tmap_gu || la.ns < 2 || la.n_fill < 1 ||
      la.n_fill >= grid)
    return cudaErrorInvalidValue;
  const size_t smem = smem_layout(a.d, la.ns, a.max_groups).total;
  static thread_local int configured_dev = -1;
  static thread_local size_t configured_smem = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev || configured_smem < smem) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_layer_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
    configured_smem = smem;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the compute CTAs wait on the fill CTAs
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_bf16_kernel, *a.tmap_gu, *a.tmap_wd, la);
}

cudaError_t decode_layer_max_blocks_per_sm(int d, int ns, int max_groups, int* out) {
  const size_t smem = smem_layout(d, ns, max_groups).total;
  cudaError_t e = cudaFuncSetAttribute(decode_layer_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, decode_layer_bf16_kernel, kThreads, smem);
}

}  // namespace ft
