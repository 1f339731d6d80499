// Prefill path: full-layer double buffer and grouped expert GEMMs.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ft_internal.h"

namespace ft {

struct PrefillConfig {
  int L, E, k, d, f, dtype;
  int buffers;  // 1 or 2
  int t_max;
  size_t Bx;
  const uint8_t* pool_dev;  // mapped device view of the pool
  const void* pool_host;    // host address of the pool (copy engine source)
  uint32_t* status;
  int sm_count;
};

struct PrefillState;

PrefillState* prefill_create(const PrefillConfig& cfg, char* msg, size_t msg_len);
void prefill_destroy(PrefillState* p);
int prefill_forward(PrefillState* p, int layer, const float* logits, const uint16_t* hidden, int T,
                    const float* partial, float* out, cudaStream_t st, Profiler* prof, char* msg,
                    size_t msg_len);

}  // namespace ft
