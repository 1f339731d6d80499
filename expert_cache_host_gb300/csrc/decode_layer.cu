// Fused decode layer kernel (bf16 or MXFP4 experts): the step's fill and all
// of its routed SwiGLU experts in one cooperative launch, one CTA per SM.
//
// FreeToken article, section "设计：三大机制" 1, Decode bullet: the q filled
// experts are copied from the host pool into their cache slots and then run on
// the GPU beside the experts that were already resident.  Here both happen in
// one grid:
//  - fill: the first n_fill CTAs stream the fetched experts from the mapped
//    pinned pool into their victim slots, expert after expert; when the last
//    of them finishes its share of fetch entry i it publishes ready[i] = the
//    step's clock (release);
//  - experts: every CTA (the fill CTAs once their share is written) takes work
//    items from a device-wide counter.  An item is one expert and 32 rows of
//    f: the same per-chunk SwiGLU GEMV as the split decode kernel --
//        h[t, i] = silu(W_gate[i] . x_t) * (W_up[i] . x_t)   i in the chunk
//        ypart[route(t), chunk, :] = W_down[:, chunk] . h[t, chunk]
//    -- with fp32 accumulation and one partial sum per (route, chunk) for the
//    merge.  Items come in the order: every chunk of every expert resident
//    before the step, then the chunks of each installed expert in fill order
//    (the control kernel lists groups by ascending expert and the fetch list
//    is ascending too, so the j-th installed group is fetch entry j).  Before
//    the first tile of an installed expert's item the producer waits (bounded,
//    %globaltimer) for its ready stamp, so it starts as soon as its own bytes
//    have landed, from L2.  Fill CTAs do not wait on anything, so every wait
//    ends; a wait that runs out records FT_ST_TIMEOUT and carries on.
// Each CTA's producer warp takes the next item when its ring has room and
// passes the index to the consumers through shared memory, published by the
// mbarrier of the item's first stage; the TMA ring (up to 12 16 KB stages)
// runs across a CTA's items.  bf16: gate/up tiles of 32 rows x 256 columns,
// down tiles of 256 rows x 32 columns, two stages per consumer iteration.
// MXFP4 (e2m1 codes, one e8m0 scale per 32 elements of a row): per token
// batch a first stage with the chunk's gate/up scale bytes (two bulk copies,
// copied to shared memory by the consumers so the ring moves on), then
// gate/up stages of two 32-row x 256-byte code boxes and down stages of four
// 256-row x 16-byte boxes; the arithmetic is the split MXFP4 kernel's (f16
// activations, HFMA2 within a scale group, fp32 across groups, h in f16 under a
// per-chunk power-of-two range scale), the
// down scales read through L2 (the fill may have written them in this launch).
#include <math.h>

#include "decode_bf16.cuh"
#include "decode_mxfp4.cuh"
#include "ft_internal.h"
#include "tma.h"

namespace ft {
namespace {

constexpr int FC = kDecodeChunk;           // 32 rows of f per item
static_assert(kDecodeChunk == kDecodeChunkFp4, "both formats use 32-row items");
constexpr int kConsumers = 512;            // 16 consumer warps
constexpr int kThreads = kConsumers + 32;  // + 1 producer warp
constexpr int kQueue = 16;                 // item indices in flight between producer and consumers (> stages)
constexpr int kMaxGroupsWarp = 64;         // groups whose values warp 0 fetches in its first round trip
constexpr int kTile = 16384;               // bytes per ring stage
constexpr int kXPre = 2;                   // uint4 of a hidden row per consumer (d <= 8192)
constexpr int kFillUnroll = 16;            // 16-byte host loads in flight per fill thread
constexpr int kFillTail = 4;               // the same for the last pieces of an expert (predicated)
constexpr int kCtasPerSm = 1;              // CTAs of the grid on each SM (two measured no faster, with spills)

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
  size_t ring, full, empty, xs, gu, hs, sc, queue, lists, total;
};

// TB: tokens per pass over the weights (1 for one-token steps, else 4).
template <bool FP4>
__host__ __device__ inline Layout smem_layout(int d, int ns, int max_groups, int TB) {
  Layout L{};
  L.ring = 0;
  L.full = L.ring + (size_t)ns * kTile;
  L.empty = L.full + 8 * (size_t)ns;
  L.xs = (L.empty + 8 * (size_t)ns + 15) / 16 * 16;  // [TB][d] bf16 hidden rows (MXFP4: [TB][d/2] f16 pairs)
  L.gu = L.xs + (size_t)TB * d * 2;                   // [2][FC][TB] row sums (MXFP4: [2 halves][2][FC][TB])
  L.hs = L.gu + sizeof(float) * (FP4 ? 4 : 2) * FC * TB;  // [TB][FC] h of the chunk (MXFP4: [TB][FC/2] f16 pairs)
  // MXFP4: + [TB] range scales of h; then [2][FC][d/32] gate/up scale bytes
  // (16-byte aligned: the consumers copy the scale bytes in with 16-byte stores)
  L.sc = (L.hs + (FP4 ? 4 * (size_t)TB * (FC / 2) + sizeof(float) * TB : sizeof(float) * TB * FC) + 15) / 16 * 16;
  L.queue = (L.sc + (FP4 ? 2 * (size_t)FC * (d / 32) : 0) + 15) / 16 * 16;  // [kQueue] items, producer -> consumers
  L.lists = L.queue + sizeof(int) * kQueue;           // [2] counts, group lists, group slots, group offsets
  L.total = L.lists + sizeof(int) * (2 + 4 * (size_t)max_groups + 1);
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
      // the rest in predicated batches of kFillTail loads in flight: copying it
      // one piece after the other would cost a host round trip per piece
      for (; v < bx16; v += kFillTail * nth) {
        int4 r[kFillTail];
#pragma unroll
        for (int j = 0; j < kFillTail; ++j)
          if (v + j * nth < bx16) r[j] = src[v + j * nth];
#pragma unroll
        for (int j = 0; j < kFillTail; ++j)
          if (v + j * nth < bx16) dst[v + j * nth] = r[j];
      }
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

template <int TB, bool FP4>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_layer_kernel(const __grid_constant__ CUtensorMap tmap_gu, const __grid_constant__ CUtensorMap tmap_wd,
                        const LayerArgs la) {
  const DecodeArgs& a = la.d;
  extern __shared__ __align__(1024) unsigned char dyn[];
  const int d = a.d, f = a.f, ns = la.ns;
  const Layout Ly = smem_layout<FP4>(d, ns, a.max_groups, TB);
  unsigned char* ring = dyn + Ly.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + Ly.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(dyn + Ly.empty);
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn + Ly.xs);  // [TB][d]
  float* gu = reinterpret_cast<float*>(dyn + Ly.gu);        // [2][FC][TB]
  float* hs = reinterpret_cast<float*>(dyn + Ly.hs);        // [TB][FC]
  unsigned char* sc = dyn + Ly.sc;                          // MXFP4: the chunk's gate/up scale bytes
  volatile int* queue = reinterpret_cast<int*>(dyn + Ly.queue);
  int* nlist = reinterpret_cast<int*>(dyn + Ly.lists);  // [0] resident, [1] installed
  int* res = nlist + 2;                                 // resident groups, ascending
  int* inst = res + a.max_groups;                       // installed groups = fetch order
  int* gslot = inst + a.max_groups;                     // [max_groups] slot of each group
  int* goff = gslot + a.max_groups;                     // [max_groups + 1] route offsets of the groups

  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) atomicMin(&la.xmeter->t0, (unsigned long long)global_ns());
  if (tid == kConsumers) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_init_fence();
  }
  if ((int)blockIdx.x < la.n_fill) {
    fill_role(la);  // then join the expert work below
    __syncthreads();
  }
  // the producer's first item: taken now, so the counter's round trip overlaps the prologue
  int first_item = 0;
  if (tid == kConsumers) first_item = (int)atomicAdd(&la.sched[0], 1u);
  // one token: every route reads hidden row 0, fetched while the lists are built
  uint4 xpre[kXPre];
  if (TB == 1 && tid < kConsumers) {
    const uint4* src = reinterpret_cast<const uint4*>(a.hidden);
#pragma unroll
    for (int j = 0; j < kXPre; ++j) {
      const int i = tid + j * kConsumers;
      if (i < d / 8) xpre[j] = ld_nc_early(src + i);
    }
  }
  // work lists: warp 0 splits the groups into resident and installed, in order,
  // and keeps each group's slot and route offsets in shared memory.  The group
  // arrays hold max_groups (+1) entries, so every group's values are read in
  // the same round trip as the group count.
  if (tid < 32) {
    constexpr int NW = kMaxGroupsWarp / 32;
    const int mg = a.max_groups;
    int cnt = 0, nw[NW], sl[NW], of[NW];
    if (lane == 0) cnt = a.counts[5];
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int g = i * 32 + lane;
      nw[i] = g < mg ? a.group_new[g] : 0;
      sl[i] = g < mg ? a.group_slot[g] : 0;
      of[i] = g <= mg ? a.group_off[g] : 0;
    }
    const int n_groups = min(__shfl_sync(0xffffffffu, cnt, 0), mg);
    int nr = 0, ni = 0;
    auto place = [&](int g, int isn, int slot, int off) {
      const bool in = g < n_groups;
      const bool isnew = in && isn != 0;
      const unsigned bn = __ballot_sync(0xffffffffu, isnew), br = __ballot_sync(0xffffffffu, in && !isnew);
      const unsigned below = (1u << lane) - 1u;
      if (isnew) inst[ni + __popc(bn & below)] = g;
      else if (in) res[nr + __popc(br & below)] = g;
      ni += __popc(bn);
      nr += __popc(br);
      if (in) {
        gslot[g] = slot;
        goff[g] = off;
      }
    };
#pragma unroll
    for (int i = 0; i < NW; ++i)
      if (i * 32 < n_groups) place(i * 32 + lane, nw[i], sl[i], of[i]);
    for (int base = NW * 32; base < n_groups; base += 32) {  // more groups than the first round trip fetched
      const int g = base + lane;
      const bool in = g < n_groups;
      place(g, in ? a.group_new[g] : 0, in ? a.group_slot[g] : 0, in ? a.group_off[g] : 0);
    }
    // the end offset of the last group: already held by lane n_groups % 32 of the first fetch
    int end_off = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int v = __shfl_sync(0xffffffffu, of[i], n_groups & 31);
      if ((n_groups >> 5) == i) end_off = v;
    }
    if (lane == 0) {
      nlist[0] = nr;
      nlist[1] = ni;
      goff[n_groups] = n_groups < NW * 32 ? end_off : a.group_off[n_groups];
    }
  }
  __syncthreads();
  const int nr = nlist[0], ni = nlist[1];
  const int n_chunks = f / FC;
  const int n_res_items = nr * n_chunks;
  const int total_items = (nr + ni) * n_chunks;
  const int q = a.counts[3];
  const uint32_t now = (uint32_t)a.counts[6];
  const int cb_n = d / 256;   // bf16: column blocks of a gate (or up) row; down tiles per batch
  const int P1 = 2 * cb_n;    // bf16: gate/up tiles per token batch
  // MXFP4: 256-byte column blocks of a gate (or up) row, two per stage; 256-row down boxes, four per stage
  const int cb4 = d / 512, gst = (cb4 + 1) / 2, nbox = d / 256, dst4 = (nbox + 3) / 4, sc_row = d / 32;
  const int NTL = FP4 ? 1 + 2 * gst + dst4 : P1 + cb_n;  // stages per token batch

  // item j -> group, chunk, fill index (-1 = resident before the step)
  auto item = [&](int j, int& g, int& c, int& fi) {
    if (j < n_res_items) {
      const int e = j / n_chunks;
      g = res[e];
      c = j - e * n_chunks;
      fi = -1;
    } else {
      const int jj = j - n_res_items;
      fi = jj / n_chunks;
      g = inst[fi];
      c = jj - fi * n_chunks;
    }
  };

  if (tid >= kConsumers) {
    // ---------------- producer warp: takes items from the device-wide counter ----------------
    if (tid == kConsumers) {
      bool late = false;
      int s = 0, n = 0;
      uint32_t ph = 0;
      for (int k = 0;; ++k) {
        const int j = k == 0 ? first_item : (int)atomicAdd(&la.sched[0], 1u);
        int g = 0, c = 0, fi = -1, slot = 0;
        const bool last = j >= total_items;
        if (!last) {
          item(j, g, c, fi);
          slot = gslot[g];
        }
        const bool bad = !last && (unsigned)slot >= (unsigned)a.S;
        if (!last && !bad && fi >= 0 && fi < q) {
          // the installed expert's bytes: wait for the fill CTAs' stamp
          if (ld_acquire(&la.ready[fi]) != now) {
            const uint64_t t0 = global_ns();
            while (ld_acquire(&la.ready[fi]) != now) {
              if (late || global_ns() - t0 > kWaitNs) {
                late = true;
                break;
              }
              __nanosleep(128);
            }
          }
          proxy_fence_global();  // fill-written bytes, read by TMA
        }
        // the item's first stage: free it, then publish the item before the
        // stage can complete (the consumers read it after waiting on the stage)
        if (n >= ns && !mbar_wait(&empty[s], ph ^ 1u, late)) late = true;
        queue[k % kQueue] = last ? -1 : (bad ? -2 - j : j);
        if (last || bad) {
          mbar_arrive_cta(&full[s]);  // no bytes: completes the stage at once
          if (++s == ns) {
            s = 0;
            ph ^= 1u;
          }
          ++n;
          if (last) break;
          continue;
        }
        const int n_batches = (goff[g + 1] - goff[g] + TB - 1) / TB;
        for (int t = 0, i = 0; t < n_batches * NTL; ++t) {
          if (t > 0 && n >= ns && !mbar_wait(&empty[s], ph ^ 1u, late)) late = true;
          unsigned char* dst = ring + s * kTile;
          if constexpr (FP4) {
            if (i == 0) {  // the chunk's gate and up scale rows (FC x d/32 bytes each, contiguous)
              const uint32_t scb = (uint32_t)(FC * sc_row);
              const size_t df = (size_t)d * f;
              const unsigned char* scg = a.arena + (size_t)slot * a.Bx + 3 * (df / 2) + (size_t)c * scb;
              mbar_expect_tx(&full[s], 2 * scb);
              bulk_g2s(dst, scg, scb, &full[s]);
              bulk_g2s(dst + scb, scg + df / 32, scb, &full[s]);
            } else if (i <= 2 * gst) {
              const int ii = i - 1, mtx = ii < gst ? 0 : 1, cb0 = 2 * (ii - mtx * gst), nb = min(2, cb4 - cb0);
              mbar_expect_tx(&full[s], nb * (kTile / 2));
              for (int b2 = 0; b2 < nb; ++b2)
                tensor_g2s_4d(dst + b2 * (kTile / 2), &tmap_gu, (cb0 + b2) * 256, c * FC, mtx, slot, &full[s]);
            } else {
              const int box0 = 4 * (i - 1 - 2 * gst), nb = min(4, nbox - box0);
              mbar_expect_tx(&full[s], nb * (kTile / 4));
              for (int b2 = 0; b2 < nb; ++b2)
                tensor_g2s_3d(dst + b2 * (kTile / 4), &tmap_wd, c * (FC / 2), (box0 + b2) * 256, slot, &full[s]);
            }
          } else {
            mbar_expect_tx(&full[s], kTile);
            if (i < P1) {
              const int mtx = i < cb_n ? 0 : 1, cb = i - mtx * cb_n;
              tensor_g2s_4d(dst, &tmap_gu, cb * 256, c * FC, mtx, slot, &full[s]);
            } else {
              tensor_g2s_3d(dst, &tmap_wd, c * FC, (i - P1) * 256, slot, &full[s]);
            }
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
  auto advance = [&]() {
    if (++s == ns) {
      s = 0;
      ph ^= 1u;
    }
  };
  auto release = [&]() {
    proxy_fence_reads();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    advance();
  };
  if (TB == 1) {
    if constexpr (FP4) {
      unsigned* x4 = reinterpret_cast<unsigned*>(xs);
#pragma unroll
      for (int j = 0; j < kXPre; ++j) {
        const int i = tid + j * kConsumers;
        if (i < d / 8) {
          x4[xs_swz(4 * i + 0)] = bf2_to_h2(xpre[j].x);
          x4[xs_swz(4 * i + 1)] = bf2_to_h2(xpre[j].y);
          x4[xs_swz(4 * i + 2)] = bf2_to_h2(xpre[j].z);
          x4[xs_swz(4 * i + 3)] = bf2_to_h2(xpre[j].w);
        }
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(xs);
#pragma unroll
      for (int j = 0; j < kXPre; ++j) {
        const int i = tid + j * kConsumers;
        if (i < d / 8) dst[i] = xpre[j];
      }
    }
  }
  // resident-phase meter: CTAs that ran resident items stamp the end of their
  // last one; the last CTA of the grid to close adds the phase
  bool resident_done = false, ran_resident = false;
  unsigned long long res_end = 0;
  auto close_resident = [&]() {
    resident_done = true;
    if (tid == 0) {
      FillMeter* m = la.xmeter;
      if (ran_resident) atomicMax(&m->t1, res_end);
      __threadfence();
      if (atomicAdd(&m->done, 1u) == gridDim.x - 1) {
        __threadfence();
        const unsigned long long t0 = atomicAdd(&m->t0, 0ull), t1 = atomicAdd(&m->t1, 0ull);
        if (nr > 0 && t1 > t0) {
          atomicAdd(&m->bytes, (unsigned long long)nr * a.Bx);
          atomicAdd(&m->ns, t1 - t0);
          atomicAdd(&m->launches, 1ull);
        }
        atomicExch(&m->t0, ~0ull);
        atomicExch(&m->t1, 0ull);
        atomicExch(&m->done, 0u);
      }
    }
  };
  for (int k = 0;; ++k) {
    // the item's first stage carries its index (or the end of the work)
    if (!mbar_wait(&full[s], ph, late)) late = true;
    const int j = queue[k % kQueue];
    if (j < -1) {  // an item whose slot id is out of range: no tiles
      if (tid == 0) atomicOr(a.status, FT_ST_BAD_SLOT);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      advance();
      continue;
    }
    if (!resident_done && (j < 0 || j >= n_res_items)) close_resident();
    if (j < 0) break;
    int g, c, fi;
    item(j, g, c, fi);
    const int r0 = goff[g], r1 = goff[g + 1];
    const int n_batches = (r1 - r0 + TB - 1) / TB;
    for (int b = 0; b < n_batches; ++b) {
      const int tb = r0 + b * TB;
      const int nt = TB == 1 ? 1 : min(TB, r1 - tb);
      int rt[TB];  // the batch's route ids (every consumer thread holds them)
#pragma unroll
      for (int t = 0; t < TB; ++t) rt[t] = t < nt ? __ldg(a.group_routes + tb + t) : 0;
      consumer_sync();  // the previous batch (or item) is done with xs / hs
      if constexpr (FP4) {
        unsigned* x4 = reinterpret_cast<unsigned*>(xs);  // [TB][d/2] f16 pairs, swizzled
        unsigned* h4 = reinterpret_cast<unsigned*>(hs);  // [TB][FC/2] f16 pairs
        float* hdown = hs + TB * (FC / 2);                // [TB] 2^(e-8) of each token's h range scale
        if (TB > 1) {
          for (int t = 0; t < nt; ++t) {
            const unsigned* src = reinterpret_cast<const unsigned*>(a.hidden + (size_t)(rt[t] / a.k) * d);
            for (int i = tid; i < d / 2; i += kConsumers) x4[(size_t)t * (d / 2) + xs_swz(i)] = bf2_to_h2(src[i]);
          }
        }
        // the batch's first stage: the chunk's gate/up scales, copied out so the ring moves on
        if (!mbar_wait(&full[s], ph, late)) late = true;
        {
          const uint4* src = reinterpret_cast<const uint4*>(ring + s * kTile);
          uint4* dst = reinterpret_cast<uint4*>(sc);
          for (int i = tid; i < 2 * FC * sc_row / 16; i += kConsumers) dst[i] = src[i];
        }
        release();
        consumer_sync();  // xs and the scales are in place
        // gate/up: thread = 16-byte column piece p of rows 2rp and 2rp + 1 of column block hb of a stage
        const int p = tid & 15, rp = (tid >> 4) & 15, hb = tid >> 8;
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
            if (cb < cb4) {
              const unsigned char* buf = ring + s * kTile + hb * (kTile / 2) + (2 * rp) * 256 + p * 16;
              w0 = *reinterpret_cast<const uint4*>(buf);
              w1 = *reinterpret_cast<const uint4*>(buf + 256);
            }
            release();
            if (cb < cb4) {
              const int grp = cb * 16 + p;  // scale group (and global 16-word piece) of this thread
              const float s0 = e8m0(sc[(m * FC + 2 * rp) * sc_row + grp]);
              const float s1 = e8m0(sc[(m * FC + 2 * rp + 1) * sc_row + grp]);
#pragma unroll
              for (int t = 0; t < TB; ++t) {
                if (t < nt) {
                  const unsigned* xrow = x4 + (size_t)t * (d / 2) + grp * 16;
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
        consumer_sync();
        if (tid < 32 * ((FC / 2 * TB + 31) / 32)) {  // whole warps: 16 lanes per token
          const int pr = tid % (FC / 2), t = tid / (FC / 2);
          float h0 = 0.f, h1 = 0.f;
          if (t < nt) {
            auto rsum = [&](int m, int row) { return gu[(m * FC + row) * TB + t] + gu[((2 + m) * FC + row) * TB + t]; };
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
            h4[t * (FC / 2) + pr] = *reinterpret_cast<const unsigned*>(&hv);
            if (pr == 0) hdown[t] = down;
          }
        }
        consumer_sync();
        // down: a stage holds rows 1024 j .. 1024 j + 1023 (16 bytes each, in order);
        // thread = rows tid and tid + 512 of the stage, one scale group each
        const size_t df = (size_t)d * f;
        const size_t sc_step = (size_t)512 * (f / 32);  // 512 rows of scales
        const unsigned char* scd =
            a.arena + (size_t)gslot[g] * a.Bx + 3 * (df / 2) + 2 * (df / 32) + (size_t)tid * (f / 32) + c;
        unsigned e0n = tid < d ? __ldcg(scd) : 0u, e1n = tid + 512 < d ? __ldcg(scd + sc_step) : 0u;
#pragma unroll 1
        for (int jd = 0; jd < dst4; ++jd) {
          const int row0 = jd * 1024 + tid, row1 = row0 + 512;
          const float s0 = e8m0(e0n), s1 = e8m0(e1n);
          if (jd + 1 < dst4) {
            e0n = row0 + 1024 < d ? __ldcg(scd + (size_t)(2 * jd + 2) * sc_step) : 0u;
            e1n = row1 + 1024 < d ? __ldcg(scd + (size_t)(2 * jd + 3) * sc_step) : 0u;
          }
          if (!mbar_wait(&full[s], ph, late)) late = true;
          const unsigned char* buf = ring + s * kTile + tid * 16;
          const uint4 w0 = row0 < d ? *reinterpret_cast<const uint4*>(buf) : make_uint4(0u, 0u, 0u, 0u);
          const uint4 w1 = row1 < d ? *reinterpret_cast<const uint4*>(buf + kTile / 2) : make_uint4(0u, 0u, 0u, 0u);
          release();
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            if (t < nt) {
              const uint4* hp = reinterpret_cast<const uint4*>(h4 + t * (FC / 2));
              float* yp = a.ypart + ((size_t)rt[t] * n_chunks + c) * d;
              if (row0 < d) yp[row0] = group_dot(w0, hp) * (s0 * hdown[t]);
              if (row1 < d) yp[row1] = group_dot(w1, hp) * (s1 * hdown[t]);
            }
          }
        }
      } else {
      if (TB > 1) {
        for (int t = 0; t < nt; ++t) {
          const int tok = rt[t] / a.k;
          const uint4* src = reinterpret_cast<const uint4*>(a.hidden + (size_t)tok * d);
          uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * d);
          for (int i = tid; i < d / 8; i += kConsumers) dst[i] = src[i];
        }
        consumer_sync();
      }

      // gate/up: tiles 0 .. P1-1 (tile i: matrix i >= cb_n, column block i mod cb_n), two per
      // iteration (P1 is even) with independent product chains
      float accg[TB], accu[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) accg[t] = accu[t] = 0.f;
      int cba = 0;  // column block of the first tile of the pair
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
        const bool ua = i >= cb_n, ub = i + 1 >= cb_n;
        const int cbb = cba + 1 == cb_n ? 0 : cba + 1;
        const uint16_t* xa = xs + cba * 256 + cq * 8;
        const uint16_t* xb = xs + cbb * 256 + cq * 8;
        cba = cbb + 1 == cb_n ? 0 : cbb + 1;
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          if (t < nt) {
            const uint4 xa0 = *reinterpret_cast<const uint4*>(xa + (size_t)t * d);
            const uint4 xa1 = *reinterpret_cast<const uint4*>(xa + (size_t)t * d + 128);
            const uint4 xb0 = *reinterpret_cast<const uint4*>(xb + (size_t)t * d);
            const uint4 xb1 = *reinterpret_cast<const uint4*>(xb + (size_t)t * d + 128);
            const float pa = dot8(wa1, xa1, dot8(wa0, xa0, 0.f));
            const float pb = dot8(wb1, xb1, dot8(wb0, xb0, 0.f));
            accg[t] += (ua ? 0.f : pa) + (ub ? 0.f : pb);
            accu[t] += (ua ? pa : 0.f) + (ub ? pb : 0.f);
          }
        }
      }
      // row sums: 16 lanes per row
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        float vg = accg[t], vu = accu[t];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          vg += __shfl_xor_sync(0xffffffffu, vg, o);
          vu += __shfl_xor_sync(0xffffffffu, vu, o);
        }
        if (cq == 0 && t < nt) {
          gu[(0 * FC + rl) * TB + t] = vg;
          gu[(1 * FC + rl) * TB + t] = vu;
        }
      }
      consumer_sync();
      if (tid < FC * TB) {
        const int row = tid % FC, t = tid / FC;
        if (t < nt) {
          const float gs = gu[(0 * FC + row) * TB + t], us = gu[(1 * FC + row) * TB + t];
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
        for (int t = 0; t < TB; ++t) {
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
              float* yp = a.ypart + ((size_t)rt[t] * n_chunks + c) * d + jd * 256 + rowq;
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
    if (j < n_res_items) {  // stamp the end of a resident item (thread 0 stands for the CTA)
      ran_resident = true;
      if (tid == 0) res_end = global_ns();
    }
  }
  // every item of the launch has been taken (this CTA's producer took its last
  // one before publishing the end): the last CTA out resets the counter
  consumer_sync();
  if (tid == 0) {
    if (late) atomicOr(a.status, FT_ST_TIMEOUT);
    __threadfence();
    if (atomicAdd(&la.sched[1], 1u) == gridDim.x - 1) {
      atomicExch(&la.sched[0], 0u);
      atomicExch(&la.sched[1], 0u);
    }
  } else if (late) {
    atomicOr(a.status, FT_ST_TIMEOUT);
  }
}

}  // namespace

int decode_layer_ring_stages(int d, int max_groups, int smem_optin, int ctas_per_sm, int dtype) {
  // the shared memory of an SM holds ctas_per_sm CTAs (1 KB of it reserved per CTA)
  const size_t per_cta = (size_t)(smem_optin + 1024) / ctas_per_sm - 1024;
  const size_t fixed = (dtype == FT_DTYPE_MXFP4 ? smem_layout<true>(d, 0, max_groups, 4).total
                                                : smem_layout<false>(d, 0, max_groups, 4).total) +
                       16 * 16 + 1024;
  if (per_cta <= fixed) return 0;
  return (int)std::min<size_t>(12, (per_cta - fixed) / (kTile + 16));
}

int decode_layer_ctas_per_sm() { return kCtasPerSm; }

namespace {
template <int TB, bool FP4>
cudaError_t launch_tb(const LayerArgs& la, int grid, cudaStream_t st) {
  const DecodeArgs& a = la.d;
  const size_t smem = smem_layout<FP4>(a.d, la.ns, a.max_groups, TB).total;
  static thread_local int configured_dev = -1;
  static thread_local size_t configured_smem = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev || configured_smem < smem) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_layer_kernel<TB, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  attr[0].id = cudaLaunchAttributeCooperative;  // CTAs wait on each other's fills
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<TB, FP4>, *a.tmap_gu, *a.tmap_wd, la);
}

template <bool FP4>
cudaError_t max_blocks(int d, int ns, int max_groups, int* out) {
  const size_t smem4 = smem_layout<FP4>(d, ns, max_groups, 4).total;
  cudaError_t e =
      cudaFuncSetAttribute(decode_layer_kernel<4, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem4);
  if (e != cudaSuccess) return e;
  int b4 = 0, b1 = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b4, decode_layer_kernel<4, FP4>, kThreads, smem4);
  if (e != cudaSuccess) return e;
  const size_t smem1 = smem_layout<FP4>(d, ns, max_groups, 1).total;
  e = cudaFuncSetAttribute(decode_layer_kernel<1, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, decode_layer_kernel<1, FP4>, kThreads, smem1);
  *out = std::min(b1, b4);
  return e;
}
}  // namespace

cudaError_t launch_decode_layer(const LayerArgs& la, int grid, cudaStream_t st) {
  const DecodeArgs& a = la.d;
  const bool fp4 = a.dtype == FT_DTYPE_MXFP4;
  if (a.dtype != FT_DTYPE_BF16 && !fp4) return cudaErrorNotSupported;
  if (a.d > 8192 || a.d % (fp4 ? 512 : 256) || a.f % FC || !a.tmap_wd || !a.tmap_gu || la.ns < 2 ||
      la.ns >= kQueue || la.n_fill < 1 || la.n_fill >= grid || !la.sched)
    return cudaErrorInvalidValue;
  if (fp4) return a.T == 1 ? launch_tb<1, true>(la, grid, st) : launch_tb<4, true>(la, grid, st);
  return a.T == 1 ? launch_tb<1, false>(la, grid, st) : launch_tb<4, false>(la, grid, st);
}

cudaError_t decode_layer_max_blocks_per_sm(int d, int ns, int max_groups, int* out, int dtype) {
  return dtype == FT_DTYPE_MXFP4 ? max_blocks<true>(d, ns, max_groups, out) : max_blocks<false>(d, ns, max_groups, out);
}

}  // namespace ft
