// Prefill path: full-layer double buffer, dispatch and grouped expert GEMMs.
//
// FreeToken article, section "设计 1" Prefill bullet: a long prompt routes to
// most experts of every layer, so prefill fetches nothing on demand; while the
// GPU computes layer l, a dedicated transfer stream loads the complete expert
// set of layer l+1 into the other buffer, and the buffers then swap roles.
// Prefill neither reads nor updates the decode cache.
//
// One layer on the compute stream:
//   route (top-k + per-expert histogram) -> scan (segment offsets, M-tile
//   list) -> scatter (counting sort of the routes by expert) -> gather (rows
//   of the hidden states in expert order) -> GEMM gate/up + SwiGLU (tcgen05)
//   -> GEMM down (tcgen05) -> combine: out[t] = partial[t] + sum_j w[t,j] y[t,j]
//   in a fixed order over j.
// The upload of a layer is one copy-engine cudaMemcpyAsync of E*B_x
// contiguous bytes of the pinned pool (the canonical layout keeps a layer's
// experts adjacent), ordered after the last GEMM that read the buffer.
#include <cstdio>
#include <cstring>
#include <new>

#include "grouped_gemm.h"
#include "prefill.h"
#include "tma.h"

namespace ft {

struct PrefillState {
  PrefillConfig cfg{};
  cudaStream_t xfer = nullptr;
  cudaEvent_t ev_up[2] = {nullptr, nullptr};
  cudaEvent_t ev_free[2] = {nullptr, nullptr};
  bool free_recorded[2] = {false, false};
  uint8_t* lbuf[2] = {nullptr, nullptr};
  int lbuf_layer[2] = {-1, -1};
  CUtensorMap map_w1[2], map_w2[2], map_x, map_h;  // bf16 weights; MXFP4: the code maps
  CUtensorMap map_s1[2], map_s2[2];                 // MXFP4: the scale maps
  CUtensorMap map_h_out, map_y_out;  // epilogue store maps (32-row boxes)
  int rows_cap = 0, max_mtiles = 0;
  int32_t* ids = nullptr;
  float* w = nullptr;
  int32_t* hist = nullptr;
  int32_t* seg_start = nullptr;
  int32_t* cursor = nullptr;
  int32_t* n_mtiles = nullptr;
  int32_t* tile_expert = nullptr;
  int32_t* tile_row0 = nullptr;
  // tiles of two 128-row M tiles of one expert (an expert's last tile holds
  // one when its M-tile count is odd): the MXFP4 GEMMs
  int32_t* n_mtiles2 = nullptr;
  int32_t* tile2_expert = nullptr;
  int32_t* tile2_row0 = nullptr;
  int32_t* tile2_mcnt = nullptr;
  int max_mtiles2 = 0;
  int32_t* perm = nullptr;
  int32_t* inv = nullptr;
  uint16_t* xs = nullptr;
  uint16_t* hbuf = nullptr;
  float* ybuf = nullptr;
};

namespace {

constexpr int kScanThreads = 1024;

// Segment offsets of the counting sort, the list of 128-row M tiles and the
// list of tiles of two M tiles (an expert's last one holds one when its
// M-tile count is odd).
__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(const int32_t* __restrict__ hist, int E, int32_t* __restrict__ seg_start, int32_t* __restrict__ cursor,
                int32_t* __restrict__ n_mtiles, int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row0,
                int32_t* __restrict__ n_mtiles2, int32_t* __restrict__ tile2_expert, int32_t* __restrict__ tile2_row0,
                int32_t* __restrict__ tile2_mcnt) {
  __shared__ int wsum[32];
  const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
  const int c = e < E ? hist[e] : 0;
  const int mt = (c + 127) / 128, mt2 = (c + 255) / 256;
  int res[3];
  const int v[3] = {c, mt, mt2};
  for (int p = 0; p < 3; ++p) {
    int x = v[p];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int s = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      wsum[lane] = s;
    }
    __syncthreads();
    res[p] = (wid ? wsum[wid - 1] : 0) + x - v[p];
    if (e == kScanThreads - 1) {
      if (p == 0) seg_start[E] = wsum[31];
      else if (p == 1) *n_mtiles = wsum[31];
      else *n_mtiles2 = wsum[31];
    }
    __syncthreads();
  }
  if (e < E) {
    seg_start[e] = res[0];
    cursor[e] = 0;
    for (int i = 0; i < mt; ++i) {
      tile_expert[res[1] + i] = e;
      tile_row0[res[1] + i] = res[0] + 128 * i;
    }
    for (int i = 0; i < mt2; ++i) {
      tile2_expert[res[2] + i] = e;
      tile2_row0[res[2] + i] = res[0] + 256 * i;
      tile2_mcnt[res[2] + i] = mt - 2 * i >= 2 ? 2 : 1;
    }
  }
}

__global__ void scatter_kernel(const int32_t* __restrict__ ids, int n_routes, const int32_t* __restrict__ seg_start,
                               int32_t* __restrict__ cursor, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_routes) return;
  const int e = ids[r];
  const int pos = seg_start[e] + atomicAdd(&cursor[e], 1);
  perm[pos] = r;
  inv[r] = pos;
}

// xs[pos] = hidden[perm[pos] / k]: one warp per row, 16-byte copies.
__global__ void gather_kernel(const uint4* __restrict__ hidden, const int32_t* __restrict__ perm, int n_rows, int k,
                              int d8, uint4* __restrict__ xs) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const uint4* src = hidden + (size_t)(perm[row] / k) * d8;
  uint4* dst = xs + (size_t)row * d8;
  for (int i = threadIdx.x & 31; i < d8; i += 32) dst[i] = src[i];
}

// out[t] = partial[t] + sum_j w[t,j] * y[inv[t,j]], j ascending.
__global__ void combine_kernel(const float4* __restrict__ y, const int32_t* __restrict__ inv,
                               const float* __restrict__ w, const float4* __restrict__ partial, float4* __restrict__ out,
                               int k, int d4) {
  const int t = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d4) return;
  float4 acc = partial ? partial[(size_t)t * d4 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float wj = w[t * k + j];
    const float4 v = y[(size_t)inv[t * k + j] * d4 + i];
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  out[(size_t)t * d4 + i] = acc;
}

bool make_weight_maps(PrefillState* p, int b, char* msg, size_t n) {
  const uint64_t d = p->cfg.d, f = p->cfg.f, E = p->cfg.E, Bx = p->cfg.Bx;
  uint8_t* lb = p->lbuf[b];
  if (p->cfg.dtype == FT_DTYPE_MXFP4) {
    // canonical MXFP4 expert: [codes gate | up | down | scales gate | up | down]
    const uint64_t df = d * f;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    // boxes: 64 gate (up) rows per gate/up tile, 128 W_down rows per down tile
    const uint64_t c1_dims[4] = {d / 2, f, 2, E}, c1_str[3] = {d / 2, df / 2, Bx};
    const uint32_t c1_box[4] = {32, 64, 1, 1};
    const uint64_t s1_dims[4] = {d / 32, f, 2, E}, s1_str[3] = {d / 32, df / 32, Bx};
    const uint32_t s1_box[4] = {16, 64, 1, 1};
    const uint64_t c2_dims[3] = {f / 2, d, E}, c2_str[2] = {f / 2, Bx};
    const uint32_t c2_box[3] = {32, 128, 1};
    const uint64_t s2_dims[3] = {f / 32, d, E}, s2_str[2] = {f / 32, Bx};
    const uint32_t s2_box[3] = {16, 128, 1};
    return encode_tensor_map(&p->map_w1[b], u8, 4, lb, c1_dims, c1_str, c1_box, msg, n) &&
           encode_tensor_map(&p->map_s1[b], u8, 4, lb + 3 * df / 2, s1_dims, s1_str, s1_box, msg, n) &&
           encode_tensor_map(&p->map_w2[b], u8, 3, lb + df, c2_dims, c2_str, c2_box, msg, n) &&
           encode_tensor_map(&p->map_s2[b], u8, 3, lb + 3 * df / 2 + 2 * df / 32, s2_dims, s2_str, s2_box, msg, n);
  }
  {
    const uint64_t dims[4] = {d, f, 2, E};
    const uint64_t strides[3] = {d * 2, d * f * 2, Bx};
    const uint32_t box[4] = {64, 128, 1, 1};
    if (!encode_tensor_map(&p->map_w1[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, lb, dims, strides, box, msg, n, true))
      return false;
  }
  {
    const uint64_t dims[3] = {f, d, E};
    const uint64_t strides[2] = {f * 2, Bx};
    const uint32_t box[3] = {64, 256, 1};
    if (!encode_tensor_map(&p->map_w2[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, lb + 4 * d * f, dims, strides, box, msg,
                           n, true))
      return false;
  }
  return true;
}

template <typename T>
bool dalloc(T** p, size_t count) {
  if (cudaMalloc(reinterpret_cast<void**>(p), sizeof(T) * (count ? count : 1)) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return false;
  }
  return true;
}

int upload(PrefillState* p, int layer, int b, Profiler* prof) {
  if (p->free_recorded[b] && cudaStreamWaitEvent(p->xfer, p->ev_free[b], 0) != cudaSuccess) return FT_E_CUDA;
  const size_t bytes = (size_t)p->cfg.E * p->cfg.Bx;
  const uint8_t* src = static_cast<const uint8_t*>(p->cfg.pool_host) + (size_t)layer * bytes;
  cudaEvent_t pb = prof ? prof->begin(p->xfer) : nullptr;
  if (cudaMemcpyAsync(p->lbuf[b], src, bytes, cudaMemcpyHostToDevice, p->xfer) != cudaSuccess) return FT_E_CUDA;
  if (prof) prof->end(p->xfer, FT_K_UPLOAD, pb);
  if (cudaEventRecord(p->ev_up[b], p->xfer) != cudaSuccess) return FT_E_CUDA;
  p->lbuf_layer[b] = layer;
  return FT_OK;
}

}  // namespace

void prefill_destroy(PrefillState* p) {
  if (!p) return;
  if (p->xfer) cudaStreamSynchronize(p->xfer);
  for (int b = 0; b < 2; ++b) {
    cudaFree(p->lbuf[b]);
    if (p->ev_up[b]) cudaEventDestroy(p->ev_up[b]);
    if (p->ev_free[b]) cudaEventDestroy(p->ev_free[b]);
  }
  cudaFree(p->ids);
  cudaFree(p->w);
  cudaFree(p->hist);
  cudaFree(p->seg_start);
  cudaFree(p->cursor);
  cudaFree(p->n_mtiles);
  cudaFree(p->tile_expert);
  cudaFree(p->tile_row0);
  cudaFree(p->n_mtiles2);
  cudaFree(p->tile2_expert);
  cudaFree(p->tile2_row0);
  cudaFree(p->tile2_mcnt);
  cudaFree(p->perm);
  cudaFree(p->inv);
  cudaFree(p->xs);
  cudaFree(p->hbuf);
  cudaFree(p->ybuf);
  if (p->xfer) cudaStreamDestroy(p->xfer);
  delete p;
}

PrefillState* prefill_create(const PrefillConfig& cfg, char* msg, size_t msg_len) {
  if (cfg.dtype == FT_DTYPE_MXFP4 ? (cfg.d % 512 || cfg.f % 512) : (cfg.d % 256 || cfg.f % 128)) {
    snprintf(msg, msg_len, "prefill GEMMs need d %% 256 == 0 and f %% 128 == 0 (bf16), or d and f multiples of 512 (MXFP4)");
    return nullptr;
  }
  PrefillState* p = new (std::nothrow) PrefillState();
  if (!p) return nullptr;
  p->cfg = cfg;
  p->rows_cap = cfg.t_max * cfg.k;
  p->max_mtiles = (p->rows_cap + 127) / 128 + cfg.E;
  p->max_mtiles2 = (p->rows_cap + 255) / 256 + cfg.E;
  const size_t layer_bytes = (size_t)cfg.E * cfg.Bx;
  bool ok = true;
  for (int b = 0; b < cfg.buffers; ++b) ok = ok && dalloc(&p->lbuf[b], layer_bytes);
  ok = ok && dalloc(&p->ids, p->rows_cap) && dalloc(&p->w, p->rows_cap) && dalloc(&p->hist, cfg.E) &&
       dalloc(&p->seg_start, cfg.E + 1) && dalloc(&p->cursor, cfg.E) && dalloc(&p->n_mtiles, 1) &&
       dalloc(&p->tile_expert, p->max_mtiles) && dalloc(&p->tile_row0, p->max_mtiles) &&
       dalloc(&p->n_mtiles2, 1) && dalloc(&p->tile2_expert, p->max_mtiles2) && dalloc(&p->tile2_row0, p->max_mtiles2) &&
       dalloc(&p->tile2_mcnt, p->max_mtiles2) &&
       dalloc(&p->perm, p->rows_cap) && dalloc(&p->inv, p->rows_cap) &&
       dalloc(&p->xs, (size_t)p->rows_cap * cfg.d) && dalloc(&p->hbuf, (size_t)p->rows_cap * cfg.f) &&
       dalloc(&p->ybuf, (size_t)p->rows_cap * cfg.d);
  if (!ok) {
    snprintf(msg, msg_len, "device allocation of %zu-byte layer buffers and work buffers failed", layer_bytes);
    prefill_destroy(p);
    return nullptr;
  }
  int lo = 0, hi = 0;
  cudaDeviceGetStreamPriorityRange(&lo, &hi);
  if (cudaStreamCreateWithPriority(&p->xfer, cudaStreamNonBlocking, hi) != cudaSuccess) ok = false;
  for (int b = 0; b < 2 && ok; ++b)
    ok = cudaEventCreateWithFlags(&p->ev_up[b], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_free[b], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    snprintf(msg, msg_len, "stream/event creation failed");
    prefill_destroy(p);
    return nullptr;
  }
  for (int b = 0; b < cfg.buffers; ++b)
    if (!make_weight_maps(p, b, msg, msg_len)) {
      prefill_destroy(p);
      return nullptr;
    }
  {
    const uint64_t dims[2] = {(uint64_t)cfg.d, (uint64_t)p->rows_cap};
    const uint64_t strides[1] = {(uint64_t)cfg.d * 2};
    const uint32_t box[2] = {64, 128};
    ok = encode_tensor_map(&p->map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->xs, dims, strides, box, msg, msg_len, true);
  }
  if (ok) {
    const uint64_t dims[2] = {(uint64_t)cfg.f, (uint64_t)p->rows_cap};
    const uint64_t strides[1] = {(uint64_t)cfg.f * 2};
    const uint32_t box[2] = {64, 128};
    ok = encode_tensor_map(&p->map_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->hbuf, dims, strides, box, msg, msg_len,
                           true);
  }
  if (ok) {
    const uint64_t dims[2] = {(uint64_t)cfg.f, (uint64_t)p->rows_cap};
    const uint64_t strides[1] = {(uint64_t)cfg.f * 2};
    const uint32_t box[2] = {64, 32};
    ok = encode_tensor_map(&p->map_h_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->hbuf, dims, strides, box, msg,
                           msg_len, true);
  }
  if (ok) {
    const uint64_t dims[2] = {(uint64_t)cfg.d, (uint64_t)p->rows_cap};
    const uint64_t strides[1] = {(uint64_t)cfg.d * 4};
    const uint32_t box[2] = {32, 32};
    ok = encode_tensor_map(&p->map_y_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p->ybuf, dims, strides, box, msg,
                           msg_len, true);
  }
  if (!ok) {
    prefill_destroy(p);
    return nullptr;
  }
  return p;
}

int prefill_forward(PrefillState* p, int layer, const float* logits, const uint16_t* hidden, int T,
                    const float* partial, float* out, cudaStream_t st, Profiler* prof, char* msg, size_t msg_len) {
  const PrefillConfig& c = p->cfg;
  const int b = c.buffers == 2 ? (layer & 1) : 0;
  int rc = FT_OK;
  if (p->lbuf_layer[b] != layer && (rc = upload(p, layer, b, prof))) {
    snprintf(msg, msg_len, "layer upload failed");
    return rc;
  }
  if (cudaStreamWaitEvent(st, p->ev_up[b], 0) != cudaSuccess) return FT_E_CUDA;

  const int n_routes = T * c.k;
  cudaEvent_t pb = prof ? prof->begin(st) : nullptr;
  cudaError_t e = cudaMemsetAsync(p->hist, 0, sizeof(int32_t) * c.E, st);
  if (e == cudaSuccess) e = launch_route(logits, T, c.E, c.k, p->ids, p->w, c.status, p->hist, st);
  if (e == cudaSuccess) {
    scan_kernel<<<1, kScanThreads, 0, st>>>(p->hist, c.E, p->seg_start, p->cursor, p->n_mtiles, p->tile_expert,
                                            p->tile_row0, p->n_mtiles2, p->tile2_expert, p->tile2_row0, p->tile2_mcnt);
    scatter_kernel<<<(n_routes + 255) / 256, 256, 0, st>>>(p->ids, n_routes, p->seg_start, p->cursor, p->perm, p->inv);
    gather_kernel<<<(n_routes + 7) / 8, 256, 0, st>>>(reinterpret_cast<const uint4*>(hidden), p->perm, n_routes, c.k,
                                                      c.d / 8, reinterpret_cast<uint4*>(p->xs));
    e = cudaGetLastError();
  }
  GemmArgs ga{};  // 128-row tiles (bf16)
  ga.n_mtiles = p->n_mtiles;
  ga.tile_expert = p->tile_expert;
  ga.tile_row0 = p->tile_row0;
  ga.seg_start = p->seg_start;
  ga.status = c.status;
  GemmArgs ga2 = ga;  // tiles of two M tiles (MXFP4)
  ga2.n_mtiles = p->n_mtiles2;
  ga2.tile_expert = p->tile2_expert;
  ga2.tile_row0 = p->tile2_row0;
  ga2.tile_mcnt = p->tile2_mcnt;
  const bool fp4 = c.dtype == FT_DTYPE_MXFP4;
  const int max_mt = (n_routes + 127) / 128 + c.E, max_mt2 = (n_routes + 255) / 256 + c.E;
  if (prof) prof->end(st, FT_K_PREFILL, pb);
  pb = prof ? prof->begin(st) : nullptr;
  if (e == cudaSuccess) {
    GemmArgs& gu = fp4 ? ga2 : ga;
    gu.out = p->hbuf;
    gu.out_ld = c.f;
    gu.K = c.d;
    e = fp4 ? launch_gemm_gateup_mxfp4(&p->map_x, &p->map_w1[b], &p->map_s1[b], &p->map_h_out, gu, max_mt2, c.f, st)
            : launch_gemm_gateup(&p->map_x, &p->map_w1[b], &p->map_h_out, gu, max_mt, c.f, st);
  }
  if (e == cudaSuccess) {
    GemmArgs& gd = fp4 ? ga2 : ga;
    gd.out = p->ybuf;
    gd.out_ld = c.d;
    gd.K = c.f;
    e = fp4 ? launch_gemm_down_mxfp4(&p->map_h, &p->map_w2[b], &p->map_s2[b], &p->map_y_out, gd, max_mt2, c.d, st)
            : launch_gemm_down(&p->map_h, &p->map_w2[b], &p->map_y_out, gd, max_mt, c.d, st);
  }
  if (prof) prof->end(st, FT_K_GEMM, pb);
  pb = prof ? prof->begin(st) : nullptr;
  if (e == cudaSuccess && cudaEventRecord(p->ev_free[b], st) == cudaSuccess) p->free_recorded[b] = true;
  if (e == cudaSuccess) {
    const int d4 = c.d / 4;
    dim3 grid((d4 + 255) / 256, T);
    combine_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4*>(p->ybuf), p->inv, p->w,
                                         reinterpret_cast<const float4*>(partial), reinterpret_cast<float4*>(out), c.k,
                                         d4);
    e = cudaGetLastError();
  }
  if (prof) prof->end(st, FT_K_PREFILL, pb);
  if (e != cudaSuccess) {
    snprintf(msg, msg_len, "launch failed: %s", cudaGetErrorString(e));
    return FT_E_CUDA;
  }
  if (c.buffers == 2 && layer + 1 < c.L) {
    const int b2 = (layer + 1) & 1;
    if (p->lbuf_layer[b2] != layer + 1 && (rc = upload(p, layer + 1, b2, prof))) {
      snprintf(msg, msg_len, "next-layer upload failed");
      return rc;
    }
  }
  return FT_OK;
}

}  // namespace ft
