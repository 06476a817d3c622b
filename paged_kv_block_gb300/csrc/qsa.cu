// Per-query block-bitmap attention forward (FlashInfer page qsa_forward) on tcgen05.
//
// One CTA per (query token t, KV head g).  The planner has already turned row t of the
// bitmap into the ascending list of selected blocks that meet [lo[t], hi[t]]; every block
// holds block_size = 4 key tokens, so a tile of 32 blocks is 128 key slots.  The work per
// (t, g) is a gather of ~1 MB of scattered K/V rows used by only G query heads, so the path
// is bound by the L2 -> SM gather rather than by the tensor pipe.  The MMAs therefore take
// the keys as the M dimension:
//   S^T [128 keys x 16]  = K_tile [128 x 256] * Q^T        (Q: G heads padded to 16 rows)
//   O^T [256 d x 16]    += V_tile^T [256 x 128] * P^T        (two M = 128 halves of d)
// Roles (288 threads):
//   warps 0-3  producers: cp.async gathers (zero-filled for dead slots) of 32 KB stages
//              (K d0-127, K d128-255, V d0-127, V d128-255 of each tile) into a 3-stage ring
//   warp  4    TMEM owner and MMA issuer (one thread)
//   warps 5-8  softmax: thread = key slot (TMEM lane) for S^T and = d row for O^T; the
//              column maxima over the 128 keys come from redux.sync plus a shared-memory
//              exchange, the row sums are accumulated per thread and reduced at the end.
#include <cstdint>
#include <cuda_bf16.h>

#include "../../include/paged_attn.h"
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kD = 256;
constexpr int kN = 16;                 // query heads of one KV head, padded (MMA N)
constexpr int kSlots = 128;            // key slots per tile = 32 blocks of 4
constexpr int kStageBytes = 32768;     // [128 keys][128 d] bf16 as two 64-column halves
constexpr int kRing = 3;
constexpr int kThreads = 288;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

struct QsaCtrl {
  uint64_t full[kRing];
  uint64_t empty[kRing];
  uint64_t q_full, s_full, p_full, o_full;
  uint32_t tmem_base;
  int abort_flag;
  int tok_tab[kSlots];
  float red[2][4][kN];
  float lred[4][kN];
};

constexpr int kQBytes = 4 * kN * 128;          // 4 chunks of [16 rows][128 B]
constexpr int kPBytes = 2 * kN * 128;          // 2 halves of [16 rows][128 B]
constexpr int kSmemBytes = kRing * kStageBytes + kQBytes + kPBytes + sizeof(QsaCtrl) + 1024;

struct QsaLaunch {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* out;
  float* out32;
  float* lse;
  const int* indptr;
  const int* indices;
  const int* bfirst;
  const int* blast;
  const int* lo;
  const int* hi;
  uint32_t* status;
  int T, Hq, Hkv, G;
  float scale_log2;
};

__device__ __forceinline__ int f2ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

__global__ void __launch_bounds__(kThreads, 2) qsa_kernel(QsaLaunch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = base;
  uint8_t* q_s = ring + kRing * kStageBytes;
  uint8_t* p_s = q_s + kQBytes;
  QsaCtrl* ctl = reinterpret_cast<QsaCtrl*>(p_s + kPBytes);

  if (launch_aborted(a.status)) return;
  const int t = blockIdx.x / a.Hkv, g = blockIdx.x % a.Hkv;
  const int G = a.G;
  const int beg = __ldg(a.indptr + t);
  const int nblk = __ldg(a.indptr + t + 1) - beg;
  const int N = nblk > 0 ? (nblk + 31) / 32 : 0;     // tiles
  const int S = 4 * N;                                // stages
  const int lo = __ldg(a.lo + t), hi = __ldg(a.hi + t);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&ctl->full[i], 128);
      mbar_init(&ctl->empty[i], 1);
    }
    mbar_init(&ctl->q_full, 128);
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->p_full, 128);
    mbar_init(&ctl->o_full, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&ctl->tmem_base, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp < 4) {
    // ================================ producers ===========================================
    const int p = threadIdx.x;                         // 0..127
    const uint32_t q_addr = smem_u32(q_s);
    for (int i = 0; i < 4; ++i) {                      // Q: 16 rows x 32 chunks of 16 B
      const int c = p + 128 * i, r = c >> 5, cc = c & 31;
      const int head = g * G + (r < G ? r : G - 1);
      const __nv_bfloat16* src = a.q + (static_cast<long long>(t) * a.Hq + head) * kD + cc * 8;
      cp_async16(q_addr + (cc >> 3) * (kN * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4), src,
                 r < G ? 16u : 0u);
    }
    cp_async_arrive_noinc(&ctl->q_full);
    const uint32_t ring_addr = smem_u32(ring);
    bool ok = true;
    for (int s = 0; s < S && ok; ++s) {
      const int n = s >> 2, part = s & 3, slot = s % kRing;
      if (part == 0) {                                 // key tokens of tile n
        named_bar(2, 128);
        const int i = n * 32 + (p >> 2);
        int tok = -1;
        if (i < nblk) {
          const int b = __ldg(a.indices + beg + i);
          const int tk = __ldg(a.bfirst + b) + (p & 3);
          if (tk <= __ldg(a.blast + b) && tk >= lo && tk <= hi) tok = tk;
        }
        ctl->tok_tab[p] = tok;
        named_bar(2, 128);
      }
      if (s >= kRing && !mbar_wait(&ctl->empty[slot], ((s / kRing) - 1) & 1, a.status, abort_flag)) {
        ok = false;
        break;
      }
      const __nv_bfloat16* src_base = part < 2 ? a.k : a.v;
      const int col0 = (part & 1) * 128;
      const uint32_t stage = ring_addr + slot * kStageBytes;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int c = p + 128 * i, row = c >> 4, cc = c & 15;
        const int tok = ctl->tok_tab[row];
        const __nv_bfloat16* src =
            src_base + (static_cast<long long>(tok >= 0 ? tok : 0) * a.Hkv + g) * kD + col0 + cc * 8;
        cp_async16(stage + (cc >> 3) * 16384 + row * 128 + (((cc & 7) ^ (row & 7)) << 4), src,
                   tok >= 0 ? 16u : 0u);
      }
      // the stage's barrier completes when this thread's copies (and the other 127's) land
      cp_async_arrive_noinc(&ctl->full[slot]);
    }
    cp_async_wait<0>();
  } else if (warp == 4) {
    // ================================ MMA issuer ==========================================
    if (lane == 0 && N > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, kN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, kN, true, false);
      const uint32_t ring_addr = smem_u32(ring), q_addr = smem_u32(q_s), p_addr = smem_u32(p_s);
      bool ok = mbar_wait(&ctl->q_full, 0, a.status, abort_flag);
      fence_proxy_async_smem();   // cp.async (generic proxy) writes -> tensor-core reads
      for (int n = 0; ok && n < N; ++n) {
        const int s0 = 4 * n;
        if (!mbar_wait(&ctl->full[s0 % kRing], (s0 / kRing) & 1, a.status, abort_flag) ||
            !mbar_wait(&ctl->full[(s0 + 1) % kRing], ((s0 + 1) / kRing) & 1, a.status, abort_flag))
          break;
        fence_proxy_async_smem();
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const int st = (s0 + (ks >> 3)) % kRing, kk = ks & 7;
          const uint32_t ka = ring_addr + st * kStageBytes + (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t qa = q_addr + (ks >> 2) * (kN * 128) + (ks & 3) * 32;
          mma_ss(tmem, sdesc_sw128(ka, 16, 1024), sdesc_sw128(qa, 16, 1024), idesc_qk, ks > 0);
        }
        mma_commit(&ctl->s_full);
        mma_commit(&ctl->empty[s0 % kRing]);
        mma_commit(&ctl->empty[(s0 + 1) % kRing]);
        if (!mbar_wait(&ctl->p_full, n & 1, a.status, abort_flag) ||
            !mbar_wait(&ctl->full[(s0 + 2) % kRing], ((s0 + 2) / kRing) & 1, a.status, abort_flag) ||
            !mbar_wait(&ctl->full[(s0 + 3) % kRing], ((s0 + 3) / kRing) & 1, a.status, abort_flag))
          break;
        fence_proxy_async_smem();
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int st = (s0 + 2 + h) % kRing;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t va = ring_addr + st * kStageBytes + ks * 2048;
            const uint32_t pa = p_addr + (ks >> 2) * (kN * 128) + (ks & 3) * 32;
            mma_ss(tmem + 16 + 16 * h, sdesc_sw128(va, 16384, 1024), sdesc_sw128(pa, 16, 1024),
                   idesc_pv, (n > 0 || ks > 0));
          }
        }
        mma_commit(&ctl->empty[(s0 + 2) % kRing]);
        mma_commit(&ctl->empty[(s0 + 3) % kRing]);
        if (n == N - 1) mma_commit(&ctl->o_full);
      }
    }
  } else {
    // ================================ softmax =============================================
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                      // key slot of S^T, d row of O^T
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    float m[kN], l[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    for (int n = 0; n < N; ++n) {
      if (!mbar_wait_warp(&ctl->s_full, n & 1, a.status, abort_flag)) break;
      tc_fence_after();
      uint32_t sv[16];
      tmem_ld16(tmem + lane_base, sv);
      tmem_ld_wait();
      const int i = n * 32 + (r >> 2);
      bool valid = false;
      if (i < nblk) {
        const int b = __ldg(a.indices + beg + i);
        const int tk = __ldg(a.bfirst + b) + (r & 3);
        valid = tk <= __ldg(a.blast + b) && tk >= lo && tk <= hi;
      }
      float x[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h)
        x[h] = (valid && h < G) ? __uint_as_float(sv[h]) * sl2 : -INFINITY;
      float (*red)[kN] = ctl->red[n & 1];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const int wm = __reduce_max_sync(0xffffffffu, f2ord(x[h]));
        if (lane == 0) red[wq][h] = ord2f(wm);
      }
      named_bar(1, 128);
      bool need = false;
      float alpha[kN], mu[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const float M = fmaxf(fmaxf(red[0][h], red[1][h]), fmaxf(red[2][h], red[3][h]));
        alpha[h] = 1.f;
        if (M > m[h] + kRescaleThreshold || (m[h] == -INFINITY && M > -INFINITY)) {
          alpha[h] = m[h] == -INFINITY ? 0.f : fast_exp2(m[h] - M);
          m[h] = M;
          need = true;
        }
        mu[h] = m[h] == -INFINITY ? 0.f : m[h];
      }
      // P^T [16 heads][128 keys], K-major with the 128-byte swizzle (two 64-key halves)
      uint8_t* prow = p_s + (r >> 6) * (kN * 128);
      const int rr = r & 63;
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const float pv = fast_exp2(x[h] - mu[h]);
        l[h] = l[h] * alpha[h] + pv;
        *reinterpret_cast<__nv_bfloat16*>(prow + h * 128 + ((((rr >> 3) ^ (h & 7)) & 7) << 4) +
                                          (rr & 7) * 2) = __float2bfloat16_rn(pv);
      }
      if (n > 0 && need) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t ov[16];
          tmem_ld16(tmem + lane_base + 16 + 16 * hh, ov);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kN; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
          tmem_st16(tmem + lane_base + 16 + 16 * hh, ov);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->p_full);
    }
    // ---- epilogue: column sums, normalise, write out / out_fp32 / lse ---------------------
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      float v = l[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) ctl->lred[wq][h] = v;
    }
    named_bar(1, 128);
    const bool have_o = N > 0 && mbar_wait_warp(&ctl->o_full, 0, a.status, abort_flag);
    uint32_t olo[16], ohi[16];
    if (have_o) {
      tc_fence_after();
      tmem_ld16(tmem + lane_base + 16, olo);
      tmem_ld16(tmem + lane_base + 32, ohi);
      tmem_ld_wait();
    }
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      if (h >= G) break;
      const float L = ctl->lred[0][h] + ctl->lred[1][h] + ctl->lred[2][h] + ctl->lred[3][h];
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float v0 = have_o ? __uint_as_float(olo[h]) * inv : 0.f;
      const float v1 = have_o ? __uint_as_float(ohi[h]) * inv : 0.f;
      const long long o = (static_cast<long long>(t) * a.Hq + g * G + h) * kD;
      a.out[o + r] = __float2bfloat16_rn(v0);
      a.out[o + 128 + r] = __float2bfloat16_rn(v1);
      if (a.out32) {
        a.out32[o + r] = v0;
        a.out32[o + 128 + r] = v1;
      }
      if (r == 0 && a.lse)
        a.lse[static_cast<long long>(g * G + h) * a.T + t] =
            L > 0.f ? (m[h] + fast_log2(L)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

int launch_qsa(const paged_attn_params* p, const paged_attn_meta* m, const void* q, const void* k,
               const void* v, void* out, float* out_fp32, float* lse, const int* indptr,
               const int* indices, uint32_t* status, cudaStream_t st) {
  const int G = p->num_qo_heads / p->num_kv_heads;
  if (G > kN || p->head_dim != kD) return PAGED_ATTN_ERR_UNSUPPORTED;
  if (!out || !m->lo_dev || !m->hi_dev || !m->block_first_dev || !m->block_last_dev)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v)) & 15u)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const long long units = static_cast<long long>(p->q_len) * p->num_kv_heads;
  if (units == 0) return PAGED_ATTN_OK;
  if (units >= (1LL << 31)) return PAGED_ATTN_ERR_UNSUPPORTED;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(qsa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return PAGED_ATTN_ERR_CUDA;
    attr_set = true;
  }
  QsaLaunch a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.out32 = out_fp32;
  a.lse = lse;
  a.indptr = indptr;
  a.indices = indices;
  a.bfirst = m->block_first_dev;
  a.blast = m->block_last_dev;
  a.lo = m->lo_dev;
  a.hi = m->hi_dev;
  a.status = status;
  a.T = p->q_len;
  a.Hq = p->num_qo_heads;
  a.Hkv = p->num_kv_heads;
  a.G = G;
  a.scale_log2 = p->sm_scale * 1.4426950408889634f;
  void* tok;
  timer_begin(st, &tok);
  qsa_kernel<<<static_cast<unsigned>(units), kThreads, kSmemBytes, st>>>(a);
  timer_end(st, tok);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

}  // namespace pa
