// Single-token paged decode with split-KV (FlashInfer page prims_ts_batch_decode_with_kv_cache).
//
// Persistent: two CTAs per SM pull (request, KV head, key split) work items from a counter.
// In each CTA a producer warp fetches the item's query rows (one TMA box per 64-column half)
// and streams the split's K/V pages into a 3-stage shared-memory ring with TMA (128-byte
// swizzled boxes, one per page piece and half), running ahead across items so the ring never
// drains between them.  Four consumer warps each take 16 keys of every 64-key stage and run
// S = Q K^T and O += P V with warp MMAs (the G query heads of the KV head are the rows of the
// 16-row A operand).  At the end of an item the warps combine their states; a request with a
// single split writes its output directly, otherwise the split's normalised fp32 partial and
// natural-log LSE go to the workspace and the last split of the (request, KV head) to finish
// merges them.
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
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMergeWarp = kConsumerWarps + 1;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kMergeSlots = 2;
constexpr int kItemSlots = 2;
constexpr int kMaxG = 16;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeSmem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t item_full[kItemSlots];
  uint64_t item_empty[kItemSlots];
  int item_id[kItemSlots];
  uint64_t merge_full[kMergeSlots];
  uint64_t merge_empty[kMergeSlots];
  int4 merge_job[kMergeSlots];   // (request, KV head, item, splits); request -1 ends the queue
  int abort_flag;
  float red_m[kConsumerWarps][kMaxG];
  float red_l[kConsumerWarps][kMaxG];
};

// Shared memory: ring | Q slots (two 64-column halves of G rows, each half in its own
// 1 KB-aligned swizzle span) | per-warp O rows of the combine | control.  Sized by G so that
// two CTAs fit on an SM for G <= 8.
__host__ __device__ constexpr int q_half_bytes(int G) { return G <= 8 ? 1024 : 2048; }
__host__ __device__ constexpr int red_bytes(int G) { return kConsumerWarps * G * kD * 4; }
__host__ __device__ constexpr int smem_bytes(int G) {
  return kStages * kStageBytes + kItemSlots * 2 * q_half_bytes(G) + red_bytes(G) +
         static_cast<int>(sizeof(DecodeSmem)) + 1024;
}

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}

__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap qmap, DecodeLaunch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = smem_align<1024>(smem_raw);
  const int G = a.Hq / a.Hkv;
  const int qhalf = q_half_bytes(G);
  uint8_t* qslots = tiles + kStages * kStageBytes;
  float* red_o = reinterpret_cast<float*>(qslots + kItemSlots * 2 * qhalf);
  DecodeSmem* sm =
      reinterpret_cast<DecodeSmem*>(reinterpret_cast<uint8_t*>(red_o) + red_bytes(G));

  if (launch_aborted(a.status)) return;
  const int n_items = a.Hkv * a.split_offset[a.B];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], kConsumerWarps);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&sm->item_full[s], 1);
      mbar_init(&sm->item_empty[s], kConsumerWarps);
    }
    for (int s = 0; s < kMergeSlots; ++s) {
      mbar_init(&sm->merge_full[s], 1);
      mbar_init(&sm->merge_empty[s], 1);
    }
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &sm->abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------ producer (whole warp) -----------------------------
    // Lane p handles page piece p of every stage (R keys of one page); the page ids of the
    // next stage are loaded while the current stage is issued.
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      tma_prefetch_desc(&qmap);
    }
    const int ps = a.page_size;
    const int R = ps < kStageKeys ? ps : kStageKeys;
    const int pieces = kStageKeys / R;                       // <= 8 (page size >= 8)
    int sg = 0;
    for (int icount = 0;; ++icount) {
      int item = 0;
      if (lane == 0) item = atomicAdd(a.work_counter, 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      const int islot = icount % kItemSlots;
      if (icount >= kItemSlots &&
          !mbar_wait_warp(&sm->item_empty[islot], ((icount / kItemSlots) - 1) & 1, a.status,
                          abort_flag))
        break;
      if (item >= n_items) {
        if (lane == 0) {
          sm->item_id[islot] = -1;
          mbar_arrive(&sm->item_full[islot]);
        }
        break;
      }
      const SplitItem it = a.items[item];
      if (lane == 0) {
        sm->item_id[islot] = item;
        uint8_t* qdst = qslots + islot * 2 * qhalf;
        mbar_arrive_expect_tx(&sm->item_full[islot], 2u * G * 128u);
        tma_load_2d(qdst, &qmap, &sm->item_full[islot], 0, it.b * a.Hq + it.g * G);
        tma_load_2d(qdst + qhalf, &qmap, &sm->item_full[islot], 64, it.b * a.Hq + it.g * G);
      }
      const int L = a.seq_lens[it.b];
      const int first_key = (it.kv_begin / kStageKeys) * kStageKeys;
      const int n_stages =
          it.kv_end > first_key ? (it.kv_end - first_key + kStageKeys - 1) / kStageKeys : 0;
      const int* pages = a.kv_indices + a.kv_indptr[it.b];
      auto page_of = [&](int s) -> int {      // page id of this lane's piece of stage s, or -1
        const int key = first_key + s * kStageKeys + lane * R;
        if (lane >= pieces || s >= n_stages || key >= L || key >= it.kv_end) return -1;
        return __ldg(pages + key / ps);
      };
      int page_next = page_of(0);
      bool ok = true;
      for (int s = 0; s < n_stages; ++s, ++sg) {
        const int page = page_next;
        page_next = page_of(s + 1);
        const int slot = sg % kStages;
        if (sg >= kStages &&
            !mbar_wait_warp(&sm->empty[slot], ((sg / kStages) - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        bool live = page >= 0;
        if (live && page >= a.num_pages) {
          report_error(a.status, kErrMetadata);
          live = false;
        }
        const uint32_t n_live = __popc(__ballot_sync(0xffffffffu, live));
        if (lane == 0) mbar_arrive_expect_tx(&sm->full[slot], n_live * 4u * R * 128u);
        __syncwarp();
        if (live) {
          const int key = first_key + s * kStageKeys + lane * R;
          const int row = page * a.page_rows + key % ps;
          const int rk = row + a.k_head_off + it.g * ps;
          const int rv = row + a.v_head_off + it.g * ps;
          uint8_t* kt = tiles + slot * kStageBytes;
          uint8_t* vt = kt + kTileBytes;
          const uint32_t off = static_cast<uint32_t>(lane * R) * 128u;
          tma_load_2d(kt + off, &kmap, &sm->full[slot], 0, rk);
          tma_load_2d(kt + kHalfBytes + off, &kmap, &sm->full[slot], 64, rk);
          tma_load_2d(vt + off, &vmap, &sm->full[slot], 0, rv);
          tma_load_2d(vt + kHalfBytes + off, &vmap, &sm->full[slot], 64, rv);
        }
      }
      if (!ok) break;
    }
  } else if (warp == kMergeWarp) {
    // ------------------------------ split merger ---------------------------------------
    // For each item of a multi-split request: make its partials visible GPU-wide, count the
    // split, and if it is the last of (b, g) to finish, merge all splits (lane -> 4 columns).
    for (int jcount = 0;; ++jcount) {
      const int js = jcount % kMergeSlots;
      if (!mbar_wait_warp(&sm->merge_full[js], (jcount / kMergeSlots) & 1, a.status, abort_flag))
        break;
      const int4 job = sm->merge_job[js];
      if (job.x < 0) break;
      const int b = job.x, g = job.y, n_split = job.w;
      __threadfence();   // the consumers' partials (ordered before the hand-off) -> GPU scope
      int prev = 0;
      if (lane == 0) prev = atomicAdd(a.counters + b * a.Hkv + g, 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == n_split - 1) {
        __threadfence();
        const long long base = static_cast<long long>(a.Hkv) * a.split_offset[b] +
                               static_cast<long long>(g) * n_split;
        for (int h = 0; h < G; ++h) {
          float M = -INFINITY;
          for (int s = lane; s < n_split; s += 32)
            M = fmaxf(M, __ldcg(a.part_lse + (base + s) * G + h));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          const float Mu = M == -INFINITY ? 0.f : M;
          float wsum = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s = 0; s < n_split; ++s) {
            const float wgt = __expf(__ldcg(a.part_lse + (base + s) * G + h) - Mu);
            wsum += wgt;
            if (wgt > 0.f) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                   a.part_o + ((base + s) * G + h) * kD) + lane);
              acc.x += wgt * v.x;
              acc.y += wgt * v.y;
              acc.z += wgt * v.z;
              acc.w += wgt * v.w;
            }
          }
          const float sc = wsum > 0.f ? a.out_scale / wsum : 0.f;
          const long long orow = static_cast<long long>(b) * a.Hq + g * G + h;
          __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(a.out + orow * kD) + lane * 2;
          dst[0] = __floats2bfloat162_rn(acc.x * sc, acc.y * sc);
          dst[1] = __floats2bfloat162_rn(acc.z * sc, acc.w * sc);
          if (a.lse && lane == 0) a.lse[orow] = wsum > 0.f ? Mu + __logf(wsum) : -INFINITY;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->merge_empty[js]);
    }
  } else {
    // ------------------------------ consumers ------------------------------------------
    const int gr = lane >> 2, tq = lane & 3;   // fragment row group, thread-in-quad
    const float sl2 = a.scale_log2;
    int sg = 0;
    int jcount = 0;                            // merge jobs handed to the merge warp
    for (int icount = 0;; ++icount) {
      const int islot = icount % kItemSlots;
      if (!mbar_wait_warp(&sm->item_full[islot], (icount / kItemSlots) & 1, a.status, abort_flag))
        break;
      const int item = sm->item_id[islot];
      if (item < 0) {
        if (threadIdx.x == 0) {                  // end of the merge queue
          const int js = jcount % kMergeSlots;
          if (jcount < kMergeSlots ||
              mbar_wait(&sm->merge_empty[js], ((jcount / kMergeSlots) - 1) & 1, a.status, abort_flag)) {
            sm->merge_job[js] = make_int4(-1, 0, 0, 0);
            mbar_arrive(&sm->merge_full[js]);
          }
        }
        break;
      }
      const SplitItem it = a.items[item];
      const int b = it.b, g = it.g;
      const int kv_begin = it.kv_begin, kv_end = it.kv_end;
      const int first_key = (kv_begin / kStageKeys) * kStageKeys;
      const int n_stages =
          kv_end > first_key ? (kv_end - first_key + kStageKeys - 1) / kStageKeys : 0;
      // Q as the A operand from the item's Q slot: rows = heads of the group (rows >= G: 0).
      uint32_t qa[kD / 16][4];
      {
        const uint8_t* qs = qslots + islot * 2 * qhalf;
        auto ld = [&](int row, int col) -> uint32_t {
          if (row >= G) return 0u;
          return *reinterpret_cast<const uint32_t*>(
              qs + (col >> 6) * qhalf + swz(row, (col & 63) >> 3) + (col & 7) * 2);
        };
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const int c0 = ks * 16 + tq * 2;
          qa[ks][0] = ld(gr, c0);
          qa[ks][1] = ld(gr + 8, c0);
          qa[ks][2] = ld(gr, c0 + 8);
          qa[ks][3] = ld(gr + 8, c0 + 8);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->item_empty[islot]);

      float o[kD / 8][4];
#pragma unroll
      for (int j = 0; j < kD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY};
      float l_run[2] = {0.f, 0.f};
      bool ok = true;
      for (int s = 0; s < n_stages; ++s, ++sg) {
        const int slot = sg % kStages;
        if (!mbar_wait_warp(&sm->full[slot], (sg / kStages) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t kt = smem_u32(tiles + slot * kStageBytes);
        const uint32_t vt = kt + kTileBytes;
        const int kbase = first_key + s * kStageKeys + warp * 16;   // first key of this warp

        // ---- this warp's 16 keys of K and V into registers; the stage is released at once,
        // so the producer refills it while the warp computes -----------------------------
        const int mi = lane >> 3, r8 = lane & 7;
        uint32_t kb[kD / 16][4], vb[kD / 16][4];
        {
          const uint32_t key_local = warp * 16 + (mi >> 1) * 8 + r8;
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const int dim = ks * 16 + (mi & 1) * 8;
            ldsm_x4(kt + (dim >> 6) * kHalfBytes + swz(key_local, (dim & 63) >> 3), kb[ks][0],
                    kb[ks][1], kb[ks][2], kb[ks][3]);
          }
        }
        {
          const uint32_t key_local = warp * 16 + (mi & 1) * 8 + r8;
#pragma unroll
          for (int j = 0; j < kD / 8; j += 2) {
            const int dim = (j + (mi >> 1)) * 8;
            ldsm_x4_t(vt + (dim >> 6) * kHalfBytes + swz(key_local, (dim & 63) >> 3),
                      vb[j >> 1][0], vb[j >> 1][1], vb[j >> 1][2], vb[j >> 1][3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[slot]);

        // ---- S = Q K^T over this warp's 16 keys --------------------------------------
        // even and odd k-steps accumulate separately: two independent MMA chains per tile
        float sc[2][4], sd[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] = sd[nt][e] = 0.f;
        {
#pragma unroll
          for (int ks = 0; ks < kD / 16; ks += 2) {
            mma_16816(sc[0], qa[ks], kb[ks][0], kb[ks][1]);
            mma_16816(sc[1], qa[ks], kb[ks][2], kb[ks][3]);
            mma_16816(sd[0], qa[ks + 1], kb[ks + 1][0], kb[ks + 1][1]);
            mma_16816(sd[1], qa[ks + 1], kb[ks + 1][2], kb[ks + 1][3]);
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
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
        // lazily moved maximum: the reference only moves when a stage exceeds it by more
        // than 8 (log2 units), so O is rarely rescaled; the final division is unaffected
        float alpha[2] = {1.f, 1.f}, muse[2];
        bool moved = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          if (mx[h] > m_run[h] + 8.f) {
            alpha[h] = m_run[h] == -INFINITY ? 0.f : fast_exp2(m_run[h] - mx[h]);
            m_run[h] = mx[h];
            moved = true;
          }
          muse[h] = m_run[h] == -INFINITY ? 0.f : m_run[h];
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
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int j = 0; j < kD / 8; ++j) {
            o[j][0] *= alpha[0];
            o[j][1] *= alpha[0];
            o[j][2] *= alpha[1];
            o[j][3] *= alpha[1];
          }
        }
        // ---- O += P V ---------------------------------------------------------------
        const uint32_t aP[4] = {pa_[0], pa_[1], pa_[2], pa_[3]};
        // keys of this lane inside the B fragments: 2tq, 2tq+1 (b0) and 8+2tq, 8+2tq+1 (b1)
        const uint32_t m_lo = (vk[0][0] ? 0x0000FFFFu : 0u) | (vk[0][1] ? 0xFFFF0000u : 0u);
        const uint32_t m_hi = (vk[1][0] ? 0x0000FFFFu : 0u) | (vk[1][1] ? 0xFFFF0000u : 0u);
        {
#pragma unroll
          for (int j = 0; j < kD / 8; j += 2) {
            uint32_t b0 = vb[j >> 1][0], b1 = vb[j >> 1][1], b2 = vb[j >> 1][2], b3 = vb[j >> 1][3];
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
      }
      if (!ok) break;

      // ---- combine the four warps -------------------------------------------------------
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
      }
#pragma unroll
      for (int j = 0; j < kD / 8; ++j) {
        const int col = j * 8 + tq * 2;
        if (gr < G) {
          float* r0 = red_o + (warp * G + gr) * kD + col;
          r0[0] = o[j][0];
          r0[1] = o[j][1];
        }
        if (gr + 8 < G) {
          float* r1 = red_o + (warp * G + gr + 8) * kD + col;
          r1[0] = o[j][2];
          r1[1] = o[j][3];
        }
      }
      if (tq == 0) {
        if (gr < G) {
          sm->red_m[warp][gr] = m_run[0];
          sm->red_l[warp][gr] = l_run[0];
        }
        if (gr + 8 < G) {
          sm->red_m[warp][gr + 8] = m_run[1];
          sm->red_l[warp][gr + 8] = l_run[1];
        }
      }
      named_bar(1, kConsumerWarps * 32);
      const int d = threadIdx.x;   // 0..127: one output column
      const int n_split = a.split_offset[b + 1] - a.split_offset[b];
      for (int h = 0; h < G; ++h) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm->red_m[w][h]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float Lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float f = fast_exp2(sm->red_m[w][h] - Mu);
          Lsum += f * sm->red_l[w][h];
          acc += f * red_o[(w * G + h) * kD + d];
        }
        const float on = Lsum > 0.f ? acc / Lsum : 0.f;
        const float lse_nat = Lsum > 0.f ? (Mu + fast_log2(Lsum)) * kLn2 : -INFINITY;
        if (n_split == 1) {
          const long long orow = static_cast<long long>(b) * a.Hq + g * G + h;
          a.out[orow * kD + d] = __float2bfloat16_rn(on * a.out_scale);
          if (a.lse && d == 0) a.lse[orow] = lse_nat;
        } else {
          const long long prow = static_cast<long long>(item) * G + h;
          a.part_o[prow * kD + d] = on;
          if (d == 0) a.part_lse[prow] = lse_nat;
        }
      }
      if (n_split > 1) {
        // the fence, the split counter and, for the last split of (b, g), the merge run on the
        // merge warp, so the consumers go on to the next item at once
        named_bar(1, kConsumerWarps * 32);         // every partial of this item is written
        if (threadIdx.x == 0) {
          const int js = jcount % kMergeSlots;
          if (jcount < kMergeSlots ||
              mbar_wait(&sm->merge_empty[js], ((jcount / kMergeSlots) - 1) & 1, a.status, abort_flag)) {
            sm->merge_job[js] = make_int4(b, g, item, n_split);
            mbar_arrive(&sm->merge_full[js]);
          }
        }
        ++jcount;
      }
      named_bar(1, kConsumerWarps * 32);   // the combine buffers are free again
    }
  }
}

int g_num_sms = 0;

}  // namespace

int launch_decode(const DecodeLaunch& a, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes(kMaxG)) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  const int G = a.Hq / a.Hkv;
  const int smem = smem_bytes(G);
  const int per_sm = 2 * (smem + 1024) <= 228 * 1024 ? 2 : 1;
  if (g_num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return -1;
  }
  if (a.capacity > 0) {
    const int grid = a.capacity < per_sm * g_num_sms ? a.capacity : per_sm * g_num_sms;
    void* tok;
    timer_begin(st, &tok);
    decode_split_kernel<<<grid, kThreads, smem, st>>>(*a.kmap, *a.vmap, *a.qmap, a);
    timer_end(st, tok);
    count_launches(1);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace pa
