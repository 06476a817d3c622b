// Benchmark hook: the rate at which this GPU's SMs read an L2-resident buffer.
//
// The bitmap form gathers the K/V rows of every selected block for every query, so most of
// its input reads hit L2 (each key row is read by hundreds of queries).  Its second roofline
// is the rate of such reads; this probe measures it with plain 16-byte loads that bypass L1
// (ld.global.cg), every thread streaming a grid-strided share of the buffer `reps` times.
#include <cstdint>

#include "../../include/paged_attn.h"
#include "internal.h"

namespace pa {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeCtasPerSm = 4;

__device__ __forceinline__ uint4 ld_cg16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kProbeThreads)
l2_read_probe_kernel(const uint4* __restrict__ buf, long long n16, int reps,
                     uint32_t* __restrict__ sink) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long t0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0u;
  for (int r = 0; r < reps; ++r) {
    long long i = t0;
    // four independent loads in flight per thread
    for (; i + 3 * stride < n16; i += 4 * stride) {
      const uint4 a = ld_cg16(buf + i), b = ld_cg16(buf + i + stride);
      const uint4 c = ld_cg16(buf + i + 2 * stride), d = ld_cg16(buf + i + 3 * stride);
      acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^
             d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
      const uint4 a = ld_cg16(buf + i);
      acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
  }
  // a store that depends on every load, taken (almost) never, keeps the loads alive
  if (acc == 0x9e3779b9u) sink[0] = acc;
}

}  // namespace
}  // namespace pa

extern "C" int paged_attn_l2_read_probe(const void* buf_dev, size_t bytes, int reps,
                                        uint32_t* sink_dev, void* stream) {
  if (!buf_dev || !sink_dev || bytes < 16 || bytes % 16 || reps <= 0 ||
      (reinterpret_cast<uintptr_t>(buf_dev) & 15))
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const int sms = pa::current_sm_count();
  if (sms <= 0) return PAGED_ATTN_ERR_CUDA;
  pa::l2_read_probe_kernel<<<sms * pa::kProbeCtasPerSm, pa::kProbeThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf_dev), static_cast<long long>(bytes / 16), reps, sink_dev);
  pa::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}
