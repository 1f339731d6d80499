// Prefill path (not built yet).
#include <cstdio>
#include "prefill.h"
#include "ft_internal.h"

namespace ft {

struct PrefillState {
  int dummy;
};

PrefillState* prefill_create(const PrefillConfig&, char* msg, size_t msg_len) {
  snprintf(msg, msg_len, "prefill is not built in this library version");
  return nullptr;
}
void prefill_destroy(PrefillState*) {}
int prefill_forward(PrefillState*, int, const float*, const uint16_t*, int, const float*, float*, cudaStream_t, Profiler*,
                    char* msg, size_t msg_len) {
  snprintf(msg, msg_len, "prefill is not built");
  return FT_E_UNSUPPORTED;
}

}  // namespace ft
