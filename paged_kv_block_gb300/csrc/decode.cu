// Single-token paged decode with split-KV (FlashInfer page prims_ts_batch_decode_with_kv_cache):
// one CTA per (request, KV head, key split).  A producer warp streams the split's K/V pages
// into a 3-stage shared-memory ring with TMA (128-byte swizzled boxes, one box per page
// piece and 64-column half); four consumer warps each take 16 keys of every 64-key stage
// and run S = Q K^T and O += P V with warp MMAs (the G query heads of the KV head are the
// rows of the 16-row A operand).  Each CTA writes its normalised fp32 partial output and
// natural-log LSE; a merge kernel combines the splits of every (request, head).
//
// The kernel is bound by HBM bandwidth: every K/V byte is read once and used by G heads.
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kStageKeys = 64;
constexpr int kStages = 3;
constexpr int kHalfBytes = kStageKeys * 128;         // 64 keys x 64 dims x bf16
constexpr int kTileBytes = 2 * kHalfBytes;            // one K (or V) stage tile
constexpr int kStageBytes = 2 * kTileBytes;           // K + V
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeSmem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
};

constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256;

__device__ __forceinline__ uint32_t swz(uint32_t key, uint32_t chunk) {
  return key * 128u + (((chunk ^ (key & 7u)) & 7u) << 4);
}

__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, DecodeLaunch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  DecodeSmem* sm = reinterpret_cast<DecodeSmem*>(tiles + kStages * kStageBytes);

  const int n_items = a.Hkv * a.split_offset[a.B];
  const int item_id = blockIdx.x;
  if (item_id >= n_items || launch_aborted(a.status)) return;
  const SplitItem it = a.items[item_id];
  const int b = it.b, g = it.g;
  const int G = a.Hq / a.Hkv;
  const int L = a.seq_lens[b];
  const int kv_begin = it.kv_begin, kv_end = it.kv_end;
  const int first_key = (kv_begin / kStageKeys) * kStageKeys;
  const int n_stages = kv_end > first_key ? (kv_end - first_key + kStageKeys - 1) / kStageKeys : 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], kConsumerWarps);
    }
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &sm->abort_flag;

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      const int ps = a.page_size;
      const int R = ps < kStageKeys ? ps : kStageKeys;
      const int* pages = a.kv_indices + a.kv_indptr[b];
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % kStages;
        if (s >= kStages) {
          if (!mbar_wait(&sm->empty[slot], ((s / kStages) - 1) & 1, a.status, abort_flag)) break;
        }
        uint8_t* kt = tiles + slot * kStageBytes;
        uint8_t* vt = kt + kTileBytes;
        const int key0 = first_key + s * kStageKeys;
        uint32_t bytes = 0;
        int n_load = 0;
        int rows_k[kStageKeys / 8], rows_v[kStageKeys / 8];
        for (int p = 0; p * R < kStageKeys; ++p) {
          const int key = key0 + p * R;
          if (key >= L || key >= kv_end) continue;
          const int page = pages[key / ps];
          if (page < 0 || page >= a.num_pages) {
            report_error(a.status, kErrMetadata);
            continue;
          }
          const int row = page * a.page_rows + key % ps;
          rows_k[p] = row + a.k_head_off + g * ps;
          rows_v[p] = row + a.v_head_off + g * ps;
          bytes += 4u * R * 128u;
          n_load |= 1 << p;
        }
        mbar_arrive_expect_tx(&sm->full[slot], bytes);
        for (int p = 0; p * R < kStageKeys; ++p) {
          if (!((n_load >> p) & 1)) continue;
          const uint32_t off = static_cast<uint32_t>(p * R) * 128u;
          tma_load_2d(kt + off, &kmap, &sm->full[slot], 0, rows_k[p]);
          tma_load_2d(kt + kHalfBytes + off, &kmap, &sm->full[slot], 64, rows_k[p]);
          tma_load_2d(vt + off, &vmap, &sm->full[slot], 0, rows_v[p]);
          tma_load_2d(vt + kHalfBytes + off, &vmap, &sm->full[slot], 64, rows_v[p]);
        }
      }
    }
  } else {
    // ------------------------------ consumers ------------------------------------------
    const int gr = lane >> 2, tq = lane & 3;   // fragment row group, thread-in-quad
    // Q as the A operand: rows = heads of the group (rows >= G are zero).
    uint32_t qa[kD / 16][4];
    const __nv_bfloat16* qb = a.q + (static_cast<long long>(b) * a.Hq + g * G) * kD;
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      const int c0 = ks * 16 + tq * 2;
      auto ld = [&](int row, int col) -> uint32_t {
        if (row >= G) return 0u;
        return *reinterpret_cast<const uint32_t*>(qb + row * kD + col);
      };
      qa[ks][0] = ld(gr, c0);
      qa[ks][1] = ld(gr + 8, c0);
      qa[ks][2] = ld(gr, c0 + 8);
      qa[ks][3] = ld(gr + 8, c0 + 8);
    }
    float o[kD / 8][4];
#pragma unroll
    for (int j = 0; j < kD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const float sl2 = a.scale_log2;

    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % kStages;
      if (!mbar_wait_warp(&sm->full[slot], (s / kStages) & 1, a.status, abort_flag)) break;
      const uint32_t kt = smem_u32(tiles + slot * kStageBytes);
      const uint32_t vt = kt + kTileBytes;
      const int kbase = first_key + s * kStageKeys + warp * 16;   // first key of this warp

      // ---- S = Q K^T over this warp's 16 keys --------------------------------------
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      {
        const int mi = lane >> 3, r = lane & 7;
        const uint32_t key_local = warp * 16 + (mi >> 1) * 8 + r;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const int dim = ks * 16 + (mi & 1) * 8;
          const uint32_t addr = kt + (dim >> 6) * kHalfBytes + swz(key_local, (dim & 63) >> 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_16816(sc[0], qa[ks], b0, b1);
          mma_16816(sc[1], qa[ks], b2, b3);
        }
      }
      // ---- mask + online softmax (rows gr and gr + 8) ----------------------------------
      bool vk[2][2];
      bool any_invalid = false;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kbase + nt * 8 + tq * 2 + e;
          vk[nt][e] = key >= kv_begin && key < kv_end;
          any_invalid |= !vk[nt][e];
        }
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = vk[nt][e & 1] ? sc[nt][e] * sl2 : -INFINITY;
          sc[nt][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      float alpha[2], muse[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mnew = fmaxf(m_run[h], mx[h]);
        muse[h] = mnew == -INFINITY ? 0.f : mnew;
        alpha[h] = fast_exp2(m_run[h] - muse[h]);
        m_run[h] = mnew;
      }
      float rs[2] = {0.f, 0.f};
      uint32_t pa_[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p0 = fast_exp2(sc[nt][0] - muse[0]);
        const float p1 = fast_exp2(sc[nt][1] - muse[0]);
        const float p2 = fast_exp2(sc[nt][2] - muse[1]);
        const float p3 = fast_exp2(sc[nt][3] - muse[1]);
        rs[0] += p0 + p1;
        rs[1] += p2 + p3;
        pa_[nt * 2 + 0] = pack_bf16(p0, p1);
        pa_[nt * 2 + 1] = pack_bf16(p2, p3);
      }
      l_run[0] = l_run[0] * alpha[0] + rs[0];
      l_run[1] = l_run[1] * alpha[1] + rs[1];
#pragma unroll
      for (int j = 0; j < kD / 8; ++j) {
        o[j][0] *= alpha[0];
        o[j][1] *= alpha[0];
        o[j][2] *= alpha[1];
        o[j][3] *= alpha[1];
      }
      // ---- O += P V ---------------------------------------------------------------
      const uint32_t aP[4] = {pa_[0], pa_[1], pa_[2], pa_[3]};
      // keys of this lane inside the B fragments: 2tq, 2tq+1 (b0) and 8+2tq, 8+2tq+1 (b1)
      const uint32_t m_lo = (vk[0][0] ? 0x0000FFFFu : 0u) | (vk[0][1] ? 0xFFFF0000u : 0u);
      const uint32_t m_hi = (vk[1][0] ? 0x0000FFFFu : 0u) | (vk[1][1] ? 0xFFFF0000u : 0u);
      {
        const int mi = lane >> 3, r = lane & 7;
        const uint32_t key_local = warp * 16 + (mi & 1) * 8 + r;
#pragma unroll
        for (int j = 0; j < kD / 8; j += 2) {
          const int dim = (j + (mi >> 1)) * 8;
          const uint32_t addr = vt + (dim >> 6) * kHalfBytes + swz(key_local, (dim & 63) >> 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          if (any_invalid) {   // stale or unused rows may hold non-finite values
            b0 &= m_lo;
            b1 &= m_hi;
            b2 &= m_lo;
            b3 &= m_hi;
          }
          mma_16816(o[j], aP, b0, b1);
          mma_16816(o[j + 1], aP, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->empty[slot]);
    }

    // ---- combine the four warps -------------------------------------------------------
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    // consumers are done with the stage ring once all of them pass this barrier
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    float* red_o = reinterpret_cast<float*>(tiles);                     // [4][16][128]
    float* red_m = red_o + kConsumerWarps * 16 * kD;                    // [4][16]
    float* red_l = red_m + kConsumerWarps * 16;                         // [4][16]
#pragma unroll
    for (int j = 0; j < kD / 8; ++j) {
      const int col = j * 8 + tq * 2;
      float* r0 = red_o + (warp * 16 + gr) * kD + col;
      float* r1 = red_o + (warp * 16 + gr + 8) * kD + col;
      r0[0] = o[j][0];
      r0[1] = o[j][1];
      r1[0] = o[j][2];
      r1[1] = o[j][3];
    }
    if (tq == 0) {
      red_m[warp * 16 + gr] = m_run[0];
      red_m[warp * 16 + gr + 8] = m_run[1];
      red_l[warp * 16 + gr] = l_run[0];
      red_l[warp * 16 + gr + 8] = l_run[1];
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    const int d = threadIdx.x;   // 0..127: one output column
    for (int h = 0; h < G; ++h) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * 16 + h]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float Lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = fast_exp2(red_m[w * 16 + h] - Mu);
        Lsum += f * red_l[w * 16 + h];
        acc += f * red_o[(w * 16 + h) * kD + d];
      }
      const long long prow = static_cast<long long>(item_id) * G + h;
      a.part_o[prow * kD + d] = Lsum > 0.f ? acc / Lsum : 0.f;
      if (d == 0) a.part_lse[prow] = Lsum > 0.f ? (Mu + fast_log2(Lsum)) * kLn2 : -INFINITY;
    }
  }
}

// One CTA of 128 threads per (request, query head): combine the request's splits.
__global__ void decode_merge_kernel(DecodeLaunch a) {
  const int bh = blockIdx.x;
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int G = a.Hq / a.Hkv, g = h / G, hg = h % G;
  const int n = a.split_offset[b + 1] - a.split_offset[b];
  const long long base = static_cast<long long>(a.Hkv) * a.split_offset[b] + g * n;
  const int d = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < n; ++s) M = fmaxf(M, a.part_lse[(base + s) * G + hg]);
  const float Mu = M == -INFINITY ? 0.f : M;
  float wsum = 0.f, acc = 0.f;
  for (int s = 0; s < n; ++s) {
    const float lse_s = a.part_lse[(base + s) * G + hg];
    const float w = __expf(lse_s - Mu);
    wsum += w;
    if (w > 0.f) acc += w * a.part_o[((base + s) * G + hg) * kD + d];
  }
  const float outv = wsum > 0.f ? acc / wsum * a.out_scale : 0.f;
  a.out[(static_cast<long long>(b) * a.Hq + h) * kD + d] = __float2bfloat16_rn(outv);
  if (a.lse && d == 0)
    a.lse[static_cast<long long>(b) * a.Hq + h] = wsum > 0.f ? Mu + __logf(wsum) : -INFINITY;
}

}  // namespace

int launch_decode(const DecodeLaunch& a, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  if (a.capacity > 0) {
    void* tok;
    timer_begin(st, &tok);
    decode_split_kernel<<<a.capacity, kThreads, kSmemBytes, st>>>(*a.kmap, *a.vmap, a);
    timer_end(st, tok);
    count_launches(1);
  }
  if (a.B > 0) {
    decode_merge_kernel<<<a.B * a.Hq, kD, 0, st>>>(a);
    count_launches(1);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace pa
