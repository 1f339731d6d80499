// Grouped expert GEMMs of the prefill path on the fifth-generation tensor
// cores (tcgen05 + tensor memory), fed by TMA.
//
// The routes of a prefill chunk are sorted by expert (counting sort), so the
// rows of each expert form one contiguous segment of the gathered activation
// matrix; segments are cut into 128-row M tiles (the last one ragged), listed
// on the device.  One CTA computes one (M tile, N tile):
//   mode 1 (gate/up): G = X W_gate^T and U = X W_up^T for the same 128 N
//     columns into two tensor-memory accumulators, then H = silu(G) * U,
//     rounded to bf16 (the operand of the next GEMM);
//   mode 2 (down):    Y = H W_down^T, 256 N columns, fp32 out.
// Warp roles: warp 0 lane 0 issues TMA loads into a 4-stage ring (A tile
// 128 x 64 and the B tiles, 128-byte swizzled), warp 1 allocates tensor
// memory and its lane 0 issues tcgen05.mma (M=128, K=16 steps), committing
// each stage back to the producer and finally to the epilogue, warps 2-5 read
// the accumulators with tcgen05.ld (one row per thread) and store the rows
// that belong to the segment.  All waits are bounded (FT_ST_TIMEOUT).
#include <cuda_bf16.h>
#include <math.h>

#include "grouped_gemm.h"
#include "tcgen05.h"

namespace ft {
namespace {

constexpr int BM = 128, BK = 64, NSTAGE = 4, kThreads = 192;

template <int MODE>
struct Cfg {
  static constexpr int BN = MODE == 1 ? 128 : 256;
  static constexpr int NB = MODE == 1 ? 2 : 1;  // B tiles per stage
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + NB * B_BYTES;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr size_t SMEM = (size_t)NSTAGE * STAGE + 1024 /*align*/ + 256 /*barriers*/;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        GemmArgs a) {
  using C = Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * C::STAGE);
  uint64_t* empty = full + NSTAGE;
  uint64_t* accb = empty + NSTAGE;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);

  // N tiles of one M tile are adjacent in launch order (the activation tile is
  // re-read from L2, not DRAM), and the few M tiles of one expert follow each
  // other (its weight tiles stay in L2 too).
  const int nt = blockIdx.x, mt = blockIdx.y;
  if (mt >= *a.n_mtiles) return;
  const int e = a.tile_expert[mt], r0 = a.tile_row0[mt], r_end = a.seg_start[e + 1];
  const int n0 = nt * C::BN;
  const int KB = a.K / BK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
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
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % NSTAGE;
        if (kb >= NSTAGE && !mbar_wait(&empty[s], (uint32_t)(((kb / NSTAGE) - 1) & 1), late)) late = true;
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
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(BM, C::BN);
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % NSTAGE;
        if (!mbar_wait(&full[s], (uint32_t)((kb / NSTAGE) & 1), late)) late = true;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * C::STAGE), sb = sa + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(sa + kk * 32);
          const uint32_t acc = (kb | kk) ? 1u : 0u;
          umma_bf16(tmem, ad, umma_desc_sw128(sb + kk * 32), idesc, acc);
          if (MODE == 1) umma_bf16(tmem + C::BN, ad, umma_desc_sw128(sb + C::B_BYTES + kk * 32), idesc, acc);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(accb);
    }
  } else {
    // epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31 (one row each)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int grow = r0 + row;
    const bool valid = grow < r_end;
    if (!mbar_wait(accb, 0, late)) late = true;
    tc_fence_after();
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
    if (MODE == 1) {
      __nv_bfloat16* H = reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)grow * a.out_ld + n0;
#pragma unroll 1
      for (int c0 = 0; c0 < C::BN; c0 += 32) {
        float gv[32], uv[32];
        tmem_ld32(lane_addr + c0, gv);
        tmem_ld32(lane_addr + C::BN + c0, uv);
        if (valid) {
          uint4 packed[4];
          uint32_t* pw = reinterpret_cast<uint32_t*>(packed);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = gv[2 * i], g1 = gv[2 * i + 1];
            const float h0 = g0 / (1.f + expf(-g0)) * uv[2 * i];
            const float h1 = g1 / (1.f + expf(-g1)) * uv[2 * i + 1];
            __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
            pw[i] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(H + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = packed[i];
        }
      }
    } else {
      float* Y = reinterpret_cast<float*>(a.out) + (size_t)grow * a.out_ld + n0;
#pragma unroll 1
      for (int c0 = 0; c0 < C::BN; c0 += 32) {
        float yv[32];
        tmem_ld32(lane_addr + c0, yv);
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(Y + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(yv[4 * i], yv[4 * i + 1], yv[4 * i + 2], yv[4 * i + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (late) atomicOr(a.status, FT_ST_TIMEOUT);
}

template <int MODE>
cudaError_t launch(const CUtensorMap* map_a, const CUtensorMap* map_b, const GemmArgs& a, int max_mtiles, int N,
                   cudaStream_t st) {
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
  dim3 grid(N / C::BN, max_mtiles);
  grouped_gemm_kernel<MODE><<<grid, kThreads, C::SMEM, st>>>(*map_a, *map_b, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gateup(const CUtensorMap* map_x, const CUtensorMap* map_w1, const GemmArgs& a, int max_mtiles,
                               int f, cudaStream_t st) {
  return launch<1>(map_x, map_w1, a, max_mtiles, f, st);
}

cudaError_t launch_gemm_down(const CUtensorMap* map_h, const CUtensorMap* map_w2, const GemmArgs& a, int max_mtiles,
                             int d, cudaStream_t st) {
  return launch<2>(map_h, map_w2, a, max_mtiles, d, st);
}

}  // namespace ft
