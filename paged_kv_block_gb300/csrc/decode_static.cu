// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call in: code running inside a
// custom allocator or an out-of-memory handler, plugins whose host framework owns every
// device allocation, or runtimes whose memory pool forbids allocations after start-up.
// For them this file keeps the decode scratch (plan, split partials, status word) in one
// fixed array in the library's own device memory.  The array is reserved on every GPU that
// loads the library and stays reserved until the process exits.
#include <mutex>

#include "../../include/paged_attn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = PAGED_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up on first use (host code
// cannot use the symbol itself as an address).  Returns a status code.
int scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return PAGED_ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PAGED_ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PAGED_ATTN_OK;
}

}  // namespace

extern "C" int paged_decode_run_static(const paged_decode_params* params, const void* query,
                                       const void* k, const void* v, const int32_t* kv_indptr,
                                       const int32_t* kv_indices, const int32_t* seq_lens,
                                       const int32_t* qo_indptr, void* out, float* lse,
                                       void* stream) {
  const size_t need = paged_decode_workspace_size(params);
  if (need == 0) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (need > kScratchBytes) return PAGED_ATTN_ERR_WORKSPACE;   // over the fixed maximum
  void* scratch = nullptr;
  const int rc = scratch_of_current_device(&scratch);
  if (rc != PAGED_ATTN_OK) return rc;
  // The regular decode path clears the status word itself and overwrites every other part
  // of the scratch it reads, so stale contents from an earlier call do not leak in.
  return paged_decode_run(params, query, k, v, kv_indptr, kv_indices, seq_lens, qo_indptr, out,
                          lse, scratch, kScratchBytes, stream);
}

// The status word opens every decode scratch layout (byte offset 0), so the word of the last
// paged_decode_run_static call on this device sits at the start of the array.
extern "C" int paged_decode_static_status(void* stream, uint32_t* raw_word) {
  void* scratch = nullptr;
  const int rc = scratch_of_current_device(&scratch);
  if (rc != PAGED_ATTN_OK) return rc;
  return paged_attn_workspace_status(scratch, stream, raw_word);
}
