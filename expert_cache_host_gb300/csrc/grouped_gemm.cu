// Grouped expert GEMMs of the prefill path on the fifth-generation tensor
// cores (tcgen05 + tensor memory), fed by TMA.
//
// The routes of a prefill chunk are sorted by expert (counting sort), so the
// rows of each expert form one contiguous segment of the gathered activation
// matrix; segments are cut into 128-row M tiles (the last one ragged), listed
// on the device.  An output tile is one (M tile, N tile):
//   mode 1 (gate/up): G = X W_gate^T and U = X W_up^T for the same 128 N
//     columns into two tensor-memory accumulators, then H = silu(G) * U,
//     rounded to bf16 (the operand of the next GEMM);
//   mode 2 (down):    Y = H W_down^T, 256 N columns, fp32 out.
// Persistent: one CTA per SM walks the tiles (N tiles of an M tile adjacent,
// so the activation tile is re-read from L2).  Warp roles: warp 0 lane 0
// issues TMA loads into a 4-stage ring (A tile 128 x 64 and the B tiles,
// 128-byte swizzled), running ahead across tile boundaries; warp 1 allocates
// all 512 tensor-memory columns as two accumulator buffers and its lane 0
// issues tcgen05.mma (M=128, K=16 steps), committing each stage back to the
// producer and each finished tile to the epilogue; warps 2-5 drain a buffer
// with tcgen05.ld (one row per thread), store the rows that belong to the
// segment and hand the buffer back -- so the epilogue of one tile overlaps
// the MMAs of the next.  All waits are bounded (FT_ST_TIMEOUT).
#include <cuda_bf16.h>
#include <math.h>

#include "grouped_gemm.h"
#include "tcgen05.h"

namespace ft {
namespace {

constexpr int BM = 128, BK = 64, NSTAGE = 4, kThreads = 192, kEpiWarps = 4;

template <int MODE>
struct Cfg {
  static constexpr int BN = MODE == 1 ? 128 : 256;
  static constexpr int NB = MODE == 1 ? 2 : 1;  // B tiles per stage
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + NB * B_BYTES;
  static constexpr uint32_t ACC_COLS = 256;          // fp32 columns of one accumulator buffer
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;  // double buffer: all 512 columns
  // epilogue staging (mode 2): per epilogue warp, two 32-row x 128-byte boxes (4 KB each)
  static constexpr int OUT_COLS = MODE == 1 ? 64 : 32;  // output columns per 128-byte row piece (bf16 / fp32)
  static constexpr int STG_BYTES = MODE == 2 ? kEpiWarps * 2 * 4096 : 0;
  static constexpr size_t SMEM = (size_t)NSTAGE * STAGE + STG_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

// Position of 16-byte chunk j of row r (0..31) inside a 32 x 128-byte staging
// box in the 128-byte swizzle layout the store tensor map expects.
__device__ __forceinline__ int stg_off(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_out, GemmArgs a, int n_ntiles) {
  using C = Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg = smem + NSTAGE * C::STAGE;  // epilogue staging (1024-byte aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + C::STG_BYTES);
  uint64_t* empty = full + NSTAGE;
  uint64_t* accf = empty + NSTAGE;  // [2] accumulator buffer holds a finished tile
  uint64_t* acce = accf + 2;        // [2] accumulator buffer drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);

  const int n_tiles = *a.n_mtiles * n_ntiles;
  const int KB = a.K / BK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps);
    }
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool late = false;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;  // k blocks issued so far (ring position)
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int mt = t / n_ntiles, n0 = (t - mt * n_ntiles) * C::BN;
        const int e = a.tile_expert[mt], r0 = a.tile_row0[mt];
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NSTAGE;
          if (it >= NSTAGE && !mbar_wait(&empty[s], (uint32_t)(((it / NSTAGE) - 1) & 1), late)) late = true;
          uint8_t* sa = smem + s * C::STAGE;
          uint8_t* sb = sa + C::A_BYTES;
          mbar_expect_tx(&full[s], C::STAGE);
          tensor_g2s_2d(sa, &map_a, kb * BK, r0, &full[s]);
          if (MODE == 1) {
            tensor_g2s_4d(sb, &map_b, kb * BK, n0, 0, e, &full[s]);
            tensor_g2s_4d(sb + C::B_BYTES, &map_b, kb * BK, n0, 1, e, &full[s]);
          } else {
            tensor_g2s_3d(sb, &map_b, kb * BK, n0, e, &full[s]);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(BM, C::BN);
      uint32_t it = 0;
      int i = 0;  // tiles of this CTA so far
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
        const int b = i & 1;
        // the epilogue must have drained this buffer (tile i - 2)
        if (i >= 2 && !mbar_wait(&acce[b], (uint32_t)(((i >> 1) - 1) & 1), late)) late = true;
        tc_fence_after();
        const uint32_t acc_tm = tmem + (uint32_t)b * C::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NSTAGE;
          if (!mbar_wait(&full[s], (uint32_t)((it / NSTAGE) & 1), late)) late = true;
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE), sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = umma_desc_sw128(sa + kk * 32);
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            umma_bf16(acc_tm, ad, umma_desc_sw128(sb + kk * 32), idesc, acc);
            if (MODE == 1) umma_bf16(acc_tm + C::BN, ad, umma_desc_sw128(sb + C::B_BYTES + kk * 32), idesc, acc);
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&accf[b]);
      }
    }
  } else {
    // epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31 (one row each).
    // Mode 2: a warp whose 32 rows all belong to the segment stages them in
    // shared memory (128-byte swizzle) and writes each 32-row x 128-byte box
    // with one TMA store (32 scattered 16-byte row pieces per store
    // instruction were bound by L2 write requests); otherwise valid rows are
    // stored directly.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    uint8_t* my_stg = stg + q * 2 * 4096;
    int nbuf = 0;  // staging buffer to fill next (0/1)
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      const int mt = t / n_ntiles, n0 = (t - mt * n_ntiles) * C::BN;
      const int e = a.tile_expert[mt], r0 = a.tile_row0[mt], r_end = a.seg_start[e + 1];
      const int grow = r0 + row;
      const bool valid = grow < r_end;
      // every row of this warp is valid (warp-uniform); the bf16 H rows of
      // mode 1 are small and go out directly, the fp32 Y rows through TMA
      const bool whole = MODE == 2 && r0 + q * 32 + 31 < r_end;
      if (!mbar_wait(&accf[b], (uint32_t)((i >> 1) & 1), late)) late = true;
      tc_fence_after();
      const uint32_t lane_addr = tmem + (uint32_t)b * C::ACC_COLS + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < C::BN; c0 += C::OUT_COLS) {
        uint4 packed[8];  // 128 bytes of this row's output columns c0 .. c0 + OUT_COLS
        if (MODE == 1) {
          uint32_t* pw = reinterpret_cast<uint32_t*>(packed);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float gv[32], uv[32];
            tmem_ld32(lane_addr + c0 + 32 * half, gv);
            tmem_ld32(lane_addr + C::BN + c0 + 32 * half, uv);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float g0 = gv[2 * j], g1 = gv[2 * j + 1];
              // H is rounded to bf16 (8-bit mantissa) right after: the fast exp and
              // divide (relative error ~1e-6) cannot change it beyond that rounding
              const float h0 = __fdividef(g0, 1.f + __expf(-g0)) * uv[2 * j];
              const float h1 = __fdividef(g1, 1.f + __expf(-g1)) * uv[2 * j + 1];
              __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
              pw[16 * half + j] = *reinterpret_cast<uint32_t*>(&b2);
            }
          }
        } else {
          float yv[32];
          tmem_ld32(lane_addr + c0, yv);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            packed[j] = make_uint4(__float_as_uint(yv[4 * j]), __float_as_uint(yv[4 * j + 1]),
                                   __float_as_uint(yv[4 * j + 2]), __float_as_uint(yv[4 * j + 3]));
        }
        if (whole) {
          uint8_t* buf = my_stg + nbuf * 4096;
          if (lane == 0) bulk_wait_read<1>();  // the store issued from this buffer two boxes ago has read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(buf + stg_off(lane, j)) = packed[j];
          proxy_fence_writes();
          __syncwarp();
          if (lane == 0) {
            tensor_s2g_2d(&map_out, n0 + c0, r0 + q * 32, buf);
            bulk_commit();
          }
          nbuf ^= 1;
        } else if (valid) {
          uint8_t* dst = reinterpret_cast<uint8_t*>(a.out) + ((size_t)grow * a.out_ld + n0 + c0) * (MODE == 1 ? 2 : 4);
#pragma unroll
          for (int j = 0; j < 8; ++j) reinterpret_cast<uint4*>(dst)[j] = packed[j];
        }
      }
      // this warp's reads of the buffer are done: hand it back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acce[b]);
    }
    if (lane == 0) bulk_wait_all();  // every store of this warp has landed before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (late) atomicOr(a.status, FT_ST_TIMEOUT);
}

template <int MODE>
cudaError_t launch(const CUtensorMap* map_a, const CUtensorMap* map_b, const CUtensorMap* map_out, const GemmArgs& a,
                   int max_mtiles, int N, cudaStream_t st) {
  using C = Cfg<MODE>;
  if (N % C::BN || a.K % BK) return cudaErrorInvalidValue;
  static thread_local int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int n_ntiles = N / C::BN;
  const int grid = max_mtiles * n_ntiles < sms ? max_mtiles * n_ntiles : sms;  // persistent: one CTA per SM
  grouped_gemm_kernel<MODE><<<grid, kThreads, C::SMEM, st>>>(*map_a, *map_b, *map_out, a, n_ntiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gateup(const CUtensorMap* map_x, const CUtensorMap* map_w1, const CUtensorMap* map_h_out,
                               const GemmArgs& a, int max_mtiles, int f, cudaStream_t st) {
  return launch<1>(map_x, map_w1, map_h_out, a, max_mtiles, f, st);
}

cudaError_t launch_gemm_down(const CUtensorMap* map_h, const CUtensorMap* map_w2, const CUtensorMap* map_y_out,
                             const GemmArgs& a, int max_mtiles, int d, cudaStream_t st) {
  return launch<2>(map_h, map_w2, map_y_out, a, max_mtiles, d, st);
}

}  // namespace ft
