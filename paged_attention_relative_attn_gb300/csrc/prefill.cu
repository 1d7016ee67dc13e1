// Chunked / paged prefill (placeholder until the tcgen05 kernel lands).
#include "internal.h"

namespace ira {
int launch_prefill(const PrefillCall& c) {
  (void)c;
  return INKLING_ERR_CUDA;
}
}  // namespace ira
