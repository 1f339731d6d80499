// Grouped expert GEMMs (tcgen05) for the prefill path.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ft_internal.h"

namespace ft {

struct GemmArgs {
  const int32_t* n_mtiles;     // device: number of valid tiles (up to 256 rows for the two-M-tile GEMMs)
  const int32_t* tile_expert;  // [max_mtiles] expert of each tile
  const int32_t* tile_row0;    // [max_mtiles] first sorted row of each tile
  const int32_t* tile_mcnt;    // [max_mtiles] 128-row M tiles in each tile (1 or 2); null: the kernel's maximum
  const int32_t* seg_start;    // [E + 1] first sorted row of each expert's segment
  void* out;                   // mode 1: H bf16 [rows, f]; mode 2: Y fp32 [rows, d]
  int out_ld;                  // elements per output row
  int K;                       // reduction length: d (mode 1) or f (mode 2)
  uint32_t* status;
};

// H[rows, f] = silu(X W_gate^T) * (X W_up^T) per expert segment; tiles of one
// 128-row M tile.
// map_x: 2-D (d, rows) bf16, box 64 x 128, 128-byte swizzle.
// map_w1: 4-D (d, f, {gate, up}, expert) bf16, box 64 x 128 x 1 x 1, 128-byte swizzle.
// map_h_out: 2-D (f, rows) bf16, box 64 x 32, 128-byte swizzle (epilogue stores).
cudaError_t launch_gemm_gateup(const CUtensorMap* map_x, const CUtensorMap* map_w1, const CUtensorMap* map_h_out,
                               const GemmArgs& a, int max_mtiles, int f, cudaStream_t st);

// Y[rows, d] = H W_down^T per expert segment; tiles of one 128-row M tile.
// map_h: 2-D (f, rows) bf16, box 64 x 128; map_w2: 3-D (f, d, expert), box 64 x 256; both 128-byte swizzle.
// map_y_out: 2-D (d, rows) fp32, box 32 x 32, 128-byte swizzle (epilogue stores).
cudaError_t launch_gemm_down(const CUtensorMap* map_h, const CUtensorMap* map_w2, const CUtensorMap* map_y_out,
                             const GemmArgs& a, int max_mtiles, int d, cudaStream_t st);

// MXFP4 weights (e2m1 codes + e8m0 scales, the canonical expert layout),
// dequantised to bf16 in shared memory; d and f multiples of 512.  Both
// GEMMs take tiles of up to two 128-row M tiles (tile_mcnt).
// map_c1: 4-D uint8 (d/2, f, {gate, up}, expert), box 32 x 64 x 1 x 1;
// map_s1: 4-D uint8 (d/32, f, {gate, up}, expert), box 16 x 64 x 1 x 1.
cudaError_t launch_gemm_gateup_mxfp4(const CUtensorMap* map_x, const CUtensorMap* map_c1, const CUtensorMap* map_s1,
                                     const CUtensorMap* map_h_out, const GemmArgs& a, int max_mtiles, int f,
                                     cudaStream_t st);

// map_c2: 3-D uint8 (f/2, d, expert), box 32 x 128 x 1; map_s2: 3-D uint8 (f/32, d, expert), box 16 x 128 x 1.
cudaError_t launch_gemm_down_mxfp4(const CUtensorMap* map_h, const CUtensorMap* map_c2, const CUtensorMap* map_s2,
                                   const CUtensorMap* map_y_out, const GemmArgs& a, int max_mtiles, int d,
                                   cudaStream_t st);

}  // namespace ft
