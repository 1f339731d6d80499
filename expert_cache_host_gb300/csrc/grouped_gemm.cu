// Grouped expert GEMMs of the prefill path on the fifth-generation tensor
// cores (tcgen05 + tensor memory), fed by TMA.
//
// The routes of a prefill chunk are sorted by expert (counting sort), so the
// rows of each expert form one contiguous segment of the gathered activation
// matrix; segments are cut into 128-row M tiles (the last one ragged), listed
// on the device.  An output tile is one (M tile, N tile):
//   mode 1 (gate/up): [G | U] = X [W_gate; W_up]^T for the same 128 rows of
//     W_gate and W_up, stacked into one 256-row B operand (one M=128, N=256
//     MMA per K step), then H = silu(G) * U, rounded to bf16 (the operand of
//     the next GEMM);
//   mode 2 (down):    Y = H W_down^T, 256 N columns, fp32 out.
// Persistent: one CTA per SM walks the tiles (N tiles of an M tile adjacent,
// so the activation tile is re-read from L2).  Warp roles: warp 0 lane 0
// issues TMA loads into the stage ring (A tile 128 x 64 and the B tile,
// 128-byte swizzled), running ahead across tile boundaries; warp 1 allocates
// all 512 tensor-memory columns as two accumulator buffers and its lane 0
// issues tcgen05.mma (M=128, N=256, K=16 steps), committing each stage back
// to the producer and each finished tile to the epilogue; warps 2-5 drain a
// buffer with tcgen05.ld (one row per thread), store the rows that belong to
// the segment and hand the buffer back -- so the epilogue of one tile overlaps
// the MMAs of the next.  All waits are bounded (FT_ST_TIMEOUT).
//
// MXFP4 weights (e2m1 codes, one e8m0 scale per 32 elements of a row): the
// producer loads the B tile's raw codes (32 bytes of each of its 256 rows per
// K step) and the scale bytes of the next 8 K steps (16 bytes per row) into
// a staging area of the stage; eight converter warps (6-13) turn every
// 32-element group into bf16 -- each e2m1 value times 2^(s-127) is exact in
// bf16 across the e8m0 range, saturating only where the product leaves it
// (|value| > 3.4e38) -- write it into the B tile in the same 128-byte swizzle
// layout TMA produces, and arrive on the stage's full barrier.  The MMA is
// then the bf16 one: activations are never quantised.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "grouped_gemm.h"
#include "tcgen05.h"

namespace ft {
namespace {

constexpr int BM = 128, BK = 64, kConvWarps = 8;

// A tile is up to MT 128-row M tiles of one expert (the tile list says how
// many) x B_ROWS rows of the B operand:
//   bf16: 1 M tile x 256 B rows (gate/up: 128 gate + 128 up; down: 256 rows
//     of W_down), accumulators double-buffered;
//   MXFP4: 2 M tiles x 128 B rows (64 gate + 64 up; 128 rows of W_down): every
//     dequantised B tile feeds two MMAs, accumulators double-buffered.
// Either way a tile's accumulators take 256 tensor-memory columns, so two
// buffers fill the 512 and the epilogue of a tile overlaps the next tile's MMAs.
template <int MODE, bool FP4>
struct Cfg {
  static constexpr int MT = FP4 ? 2 : 1;                                   // max 128-row M tiles per tile
  static constexpr int B_ROWS = FP4 ? 128 : 256;                           // B operand rows
  static constexpr int BN = MODE == 1 ? B_ROWS / 2 : B_ROWS;               // output columns of a tile
  static constexpr uint32_t ACC_COLS = MT * B_ROWS;                        // fp32 columns of one buffer
  static constexpr int NBUF = 2;                                           // accumulator buffers
  static constexpr uint32_t TMEM_COLS = NBUF * ACC_COLS;                   // all 512 columns
  static constexpr int EPI = 4;                                            // epilogue warps, one per lane quarter
  static constexpr int kThreads = 64 + 32 * EPI + (FP4 ? 32 * kConvWarps : 0);
  static constexpr int CONV0 = 2 + EPI;                                    // first converter warp
  static constexpr int A_TILE = BM * BK * 2;
  static constexpr int A_BYTES = MT * A_TILE;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int RAW_CODES = FP4 ? B_ROWS * BK / 2 : 0;  // 32 code bytes per row per K step
  static constexpr int RAW_SC = FP4 ? B_ROWS * 16 : 0;          // scale bytes of 8 K steps per row
  static constexpr int STAGE = A_BYTES + B_BYTES + RAW_CODES + RAW_SC;  // a multiple of 1024
  static constexpr int NSTAGE = FP4 && MODE == 2 ? 3 : 4;  // MXFP4 down: room for the epilogue staging
  // epilogue staging (mode 2): per epilogue warp, two 32-row x 128-byte boxes (4 KB each)
  static constexpr int OUT_COLS = MODE == 1 ? 64 : 32;  // output columns per 128-byte row piece (bf16 / fp32)
  static constexpr int STG_BYTES = MODE == 2 ? EPI * 2 * 4096 : 0;
  static constexpr size_t SMEM = (size_t)NSTAGE * STAGE + STG_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(STAGE % 1024 == 0, "stage tiles must stay 1024-byte aligned for the 128-byte swizzle");
  static_assert(TMEM_COLS == 512, "two accumulator buffers fill the tensor memory");
};

// Exact 2^(s-127) for an e8m0 byte (s = 255 is NaN, s = 0 the fp32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_scale(unsigned s) {
  return s == 255u ? __int_as_float(0x7FC00000) : (s ? __int_as_float((int)(s << 23)) : __int_as_float(0x00400000));
}

// Eight e2m1 codes (four bytes, element 2i in the low nibble of byte i) times
// the group scale -> eight bf16 values (one 16-byte chunk of a B row).  The
// code -> f16 conversion and the fp32 product are exact; so is the rounding
// to bf16, since the product carries at most two significant bits.
__device__ __forceinline__ uint4 e2m1x8_to_bf16(unsigned w, float sc) {
  unsigned p[4];
  asm("{ .reg .b8 a0, a1, a2, a3; mov.b32 {a0, a1, a2, a3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a0; cvt.rn.f16x2.e2m1x2 %1, a1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, a2; cvt.rn.f16x2.e2m1x2 %3, a3; }"
      : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3])
      : "r"(w));
  unsigned o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&p[i]));
    __nv_bfloat162 b = __floats2bfloat162_rn(v.x * sc, v.y * sc);
    o[i] = *reinterpret_cast<unsigned*>(&b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Position of 16-byte chunk j of row r inside a tile of 128-byte rows in the
// 128-byte swizzle layout (the one TMA reads and writes and the MMA
// descriptors name), the tile 1024-byte aligned.
__device__ __forceinline__ int stg_off(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

template <int MODE, bool FP4>
__global__ void __launch_bounds__(Cfg<MODE, FP4>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_out,
                        GemmArgs a, int n_ntiles) {
  using C = Cfg<MODE, FP4>;
  constexpr int NSTAGE = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg = smem + NSTAGE * C::STAGE;  // epilogue staging (1024-byte aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + C::STG_BYTES);
  uint64_t* empty = full + NSTAGE;
  uint64_t* rawf = empty + NSTAGE;  // [NSTAGE] MXFP4: the stage's codes and scales have landed
  uint64_t* accf = rawf + NSTAGE;   // [2] accumulator buffer holds a finished tile
  uint64_t* acce = accf + 2;        // [2] accumulator buffer drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);

  const int n_tiles = *a.n_mtiles * n_ntiles;
  const int KB = a.K / BK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      // MXFP4: the A tile's bytes plus one arrival per converter warp
      mbar_init(&full[s], FP4 ? 1 + kConvWarps : 1);
      mbar_init(&empty[s], 1);
      mbar_init(&rawf[s], 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], C::EPI);
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
        const int mc = C::MT == 1 ? 1 : (a.tile_mcnt ? a.tile_mcnt[mt] : C::MT);  // M tiles of this tile (1 .. MT)
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NSTAGE;
          if (it >= NSTAGE && !mbar_wait(&empty[s], (uint32_t)(((it / NSTAGE) - 1) & 1), late)) late = true;
          uint8_t* sa = smem + s * C::STAGE;
          uint8_t* sb = sa + C::A_BYTES;
          if (FP4) {
            uint8_t* rc = sb + C::B_BYTES;    // [B_ROWS][32 code bytes]
            uint8_t* rs = rc + C::RAW_CODES;  // [B_ROWS][16 scale bytes]
            const int xs = (kb >> 3) * 16;  // the 16 scale bytes that cover K steps 8*(kb/8) .. +7
            mbar_expect_tx(&rawf[s], C::RAW_CODES + C::RAW_SC);
            if (MODE == 1) {
              tensor_g2s_4d(rc, &map_b, kb * (BK / 2), n0, 0, e, &rawf[s]);
              tensor_g2s_4d(rc + C::RAW_CODES / 2, &map_b, kb * (BK / 2), n0, 1, e, &rawf[s]);
              tensor_g2s_4d(rs, &map_s, xs, n0, 0, e, &rawf[s]);
              tensor_g2s_4d(rs + C::RAW_SC / 2, &map_s, xs, n0, 1, e, &rawf[s]);
            } else {
              tensor_g2s_3d(rc, &map_b, kb * (BK / 2), n0, e, &rawf[s]);
              tensor_g2s_3d(rs, &map_s, xs, n0, e, &rawf[s]);
            }
            mbar_expect_tx(&full[s], mc * C::A_TILE);
            for (int h = 0; h < mc; ++h) tensor_g2s_2d(sa + h * C::A_TILE, &map_a, kb * BK, r0 + BM * h, &full[s]);
          } else {
            mbar_expect_tx(&full[s], mc * C::A_TILE + C::B_BYTES);
            for (int h = 0; h < mc; ++h) tensor_g2s_2d(sa + h * C::A_TILE, &map_a, kb * BK, r0 + BM * h, &full[s]);
            if (MODE == 1) {
              tensor_g2s_4d(sb, &map_b, kb * BK, n0, 0, e, &full[s]);
              tensor_g2s_4d(sb + C::B_BYTES / 2, &map_b, kb * BK, n0, 1, e, &full[s]);
            } else {
              tensor_g2s_3d(sb, &map_b, kb * BK, n0, e, &full[s]);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(BM, C::B_ROWS);
      uint32_t it = 0;
      int i = 0;  // tiles of this CTA so far
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
        const int b = i % C::NBUF;
        const int mc = C::MT == 1 ? 1 : (a.tile_mcnt ? a.tile_mcnt[t / n_ntiles] : C::MT);
        // the epilogue must have drained this buffer (tile i - NBUF)
        if (i >= C::NBUF && !mbar_wait(&acce[b], (uint32_t)(((i / C::NBUF) - 1) & 1), late)) late = true;
        tc_fence_after();
        const uint32_t acc_tm = tmem + (uint32_t)b * C::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NSTAGE;
          if (!mbar_wait(&full[s], (uint32_t)((it / NSTAGE) & 1), late)) late = true;
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE), sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
#pragma unroll
            for (int h = 0; h < C::MT; ++h)
              if (h < mc)
                umma_bf16(acc_tm + (uint32_t)(h * C::B_ROWS), umma_desc_sw128(sa + h * C::A_TILE + kk * 32),
                          umma_desc_sw128(sb + kk * 32), idesc, (kb | kk) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        umma_commit(&accf[b]);
      }
    }
  } else if (warp < C::CONV0) {
    // epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31 (one row each).
    // Mode 2: a warp whose 32 rows all belong to the segment stages them in
    // shared memory (128-byte swizzle) and writes each 32-row x 128-byte box
    // with one TMA store (32 scattered 16-byte row pieces per store
    // instruction were bound by L2 write requests); otherwise valid rows are
    // stored directly.
    const int q = warp & 3;  // the tensor-memory lane quarter this warp may read
    const int row = q * 32 + lane;
    uint8_t* my_stg = stg + q * 2 * 4096;
    int nbuf = 0;  // staging buffer to fill next (0/1)
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
      const int b = i % C::NBUF;
      const int mt = t / n_ntiles, n0 = (t - mt * n_ntiles) * C::BN;
      const int e = a.tile_expert[mt], r_end = a.seg_start[e + 1];
      const int mc = C::MT == 1 ? 1 : (a.tile_mcnt ? a.tile_mcnt[mt] : C::MT);
      if (!mbar_wait(&accf[b], (uint32_t)((i / C::NBUF) & 1), late)) late = true;
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < mc; ++h) {  // the tile's M tiles, one accumulator each
        const int r0 = a.tile_row0[mt] + BM * h;
        const int grow = r0 + row;
        const bool valid = grow < r_end;
        // every row of this warp is valid (warp-uniform); the bf16 H rows of
        // mode 1 are small and go out directly, the fp32 Y rows through TMA
        const bool whole = MODE == 2 && r0 + q * 32 + 31 < r_end;
        const uint32_t lane_addr =
            tmem + (uint32_t)b * C::ACC_COLS + (uint32_t)(h * C::B_ROWS) + ((uint32_t)(q * 32) << 16);
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
      }
      // this warp's reads of the buffer are done: hand it back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acce[b]);
    }
    if (lane == 0) bulk_wait_all();  // every store of this warp has landed before the CTA exits
  } else if (FP4) {
    // converters: 256 threads, B_ROWS * 2 / 256 (row, 32-element group) units
    // each per K step; a warp covers 16 rows, so its 16-byte code reads are
    // contiguous and each quarter-warp's four 16-byte chunk stores hit
    // distinct banks.
    const int ct = threadIdx.x - 32 * C::CONV0;
    uint32_t it = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % NSTAGE;
        if (!mbar_wait(&rawf[s], (uint32_t)((it / NSTAGE) & 1), late)) late = true;
        uint8_t* sb = smem + s * C::STAGE + C::A_BYTES;
        const uint8_t* rc = sb + C::B_BYTES;
        const uint8_t* rs = rc + C::RAW_CODES;
#pragma unroll
        for (int u2 = 0; u2 < C::B_ROWS * 2 / 256; ++u2) {
          const int u = ct + 256 * u2, r = u >> 1, h = u & 1;
          const uint4 cw = *reinterpret_cast<const uint4*>(rc + r * 32 + h * 16);
          const float sc = e8m0_scale(rs[r * 16 + (kb & 7) * 2 + h]);
          const unsigned wv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(sb + stg_off(r, 4 * h + q)) = e2m1x8_to_bf16(wv[q], sc);
        }
        // the B tile is read by the tensor core (async proxy), and the codes'
        // staging is rewritten by TMA once the MMAs have consumed the stage
        proxy_fence_writes();
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(&full[s]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (late) atomicOr(a.status, FT_ST_TIMEOUT);
}

template <int MODE, bool FP4>
cudaError_t launch(const CUtensorMap* map_a, const CUtensorMap* map_b, const CUtensorMap* map_s,
                   const CUtensorMap* map_out, const GemmArgs& a, int max_mtiles, int N, cudaStream_t st) {
  using C = Cfg<MODE, FP4>;
  if (N % C::BN || a.K % BK || (FP4 && a.K % 512)) return cudaErrorInvalidValue;
  static thread_local int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int n_ntiles = N / C::BN;
  const int grid = max_mtiles * n_ntiles < sms ? max_mtiles * n_ntiles : sms;  // persistent: one CTA per SM
  grouped_gemm_kernel<MODE, FP4>
      <<<grid, C::kThreads, C::SMEM, st>>>(*map_a, *map_b, map_s ? *map_s : *map_b, *map_out, a, n_ntiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gateup(const CUtensorMap* map_x, const CUtensorMap* map_w1, const CUtensorMap* map_h_out,
                               const GemmArgs& a, int max_mtiles, int f, cudaStream_t st) {
  return launch<1, false>(map_x, map_w1, nullptr, map_h_out, a, max_mtiles, f, st);
}

cudaError_t launch_gemm_down(const CUtensorMap* map_h, const CUtensorMap* map_w2, const CUtensorMap* map_y_out,
                             const GemmArgs& a, int max_mtiles, int d, cudaStream_t st) {
  return launch<2, false>(map_h, map_w2, nullptr, map_y_out, a, max_mtiles, d, st);
}

cudaError_t launch_gemm_gateup_mxfp4(const CUtensorMap* map_x, const CUtensorMap* map_c1, const CUtensorMap* map_s1,
                                     const CUtensorMap* map_h_out, const GemmArgs& a, int max_mtiles, int f,
                                     cudaStream_t st) {
  return launch<1, true>(map_x, map_c1, map_s1, map_h_out, a, max_mtiles, f, st);
}

cudaError_t launch_gemm_down_mxfp4(const CUtensorMap* map_h, const CUtensorMap* map_c2, const CUtensorMap* map_s2,
                                   const CUtensorMap* map_y_out, const GemmArgs& a, int max_mtiles, int d,
                                   cudaStream_t st) {
  return launch<2, true>(map_h, map_c2, map_s2, map_y_out, a, max_mtiles, d, st);
}

}  // namespace ft
