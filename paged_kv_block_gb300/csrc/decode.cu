// Paged decode with split-KV (FlashInfer page prims_ts_batch_decode_with_kv_cache): one
// query per request, SQ fixed queries per request ([B, SQ, Hq, D]) or packed queries
// (qo_indptr), each query at position len - nq + i under the causal / window mask.
//
// Persistent: two CTAs per SM pull (request, KV head, key split) work items from a counter.
// An item's rows are the M = (queries per request) x G (query, head) pairs of its KV head,
// row m = (query m / G, head m % G), M <= 64, in R = 1, 2 or 4 blocks of 16 rows.  In each
// CTA a producer warp fetches the item's query rows (one TMA box of G heads x queries per
// 64-column half) and streams the split's K/V pages into a 3-stage shared-memory ring with
// TMA (128-byte swizzled boxes, one per page piece and half), running ahead across items so
// the ring never drains between them.  Four consumer warps split each 64-key stage: warp w
// takes row block w / (4 / R) and a (16 R)-key slice, 16 keys at a time, and runs
// S = Q K^T and O += P V with warp MMAs (16 rows of the A operand).  At the end of an item
// the warps combine their states in the shared memory of the item's last stage, which they
// release only afterwards; a request with a single split writes its output directly,
// otherwise the split's normalised fp32 partial and natural-log LSE go to the workspace and
// the last split of the (request, KV head) to finish merges them.
//
// The kernel is bound by HBM bandwidth: every K/V byte is read once and used by all M rows.
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
constexpr int kMaxRows = 64;   // rows (query, head pairs) of one item
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
  int skip;                // an earlier CTA recorded a timeout: this CTA does nothing
  float red_m[kMaxRows];   // per (key slice, row) maxima and sums of the combine
  float red_l[kMaxRows];
};

// Shared memory: ring | Q slots (two 64-column halves of M rows, each half in its own
// 1 KB-aligned swizzle span) | control.  The combine at the end of an item borrows the
// item's last ring stage (32 KB = 64 rows x 128 fp32 columns), so two CTAs fit on an SM
// for M <= 16.
__host__ __device__ constexpr int q_half_bytes(int M) { return (M * 128 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int smem_bytes(int M) {
  return kStages * kStageBytes + kItemSlots * 2 * q_half_bytes(M) +
         static_cast<int>(sizeof(DecodeSmem)) + 1024;
}
static_assert(kMaxRows * kD * 4 <= kStageBytes, "the combine must fit in one ring stage");

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}

// Merge of the split partials of rows m0 .. m0 + 7 (those below live_rows) of one (request,
// KV head), by one warp: lane l owns columns 4l .. 4l + 3.  The merge sits on the critical
// path at the end of a launch, so it is written for few dependent L2 round trips: lane j
// loads split s0 + j's LSE of all 8 rows at once, and the partial rows of two splits are
// loaded together (16 loads in flight) before they are accumulated.  Every live row of
// every split has a partial (an empty split writes O = 0 and LSE = -inf), so no load is
// conditional on the data.
constexpr int kMergeRows = 8;
__device__ __forceinline__ void merge_rows(const DecodeLaunch& a, long long base, int n_split, int M,
                                        int G, int m0, int live_rows, int q_row0, int g,
                                        int lane) {
  const int nr = live_rows - m0 < kMergeRows ? live_rows - m0 : kMergeRows;
  float Mx[kMergeRows], wsum[kMergeRows];
  float4 acc[kMergeRows];
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
    Mx[r] = -INFINITY;
    wsum[r] = 0.f;
    acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // row maxima over all splits (one pass of loads when n_split <= 32)
  float lse_own[kMergeRows];
  for (int s0 = 0; s0 < n_split; s0 += 32) {
    const int s = s0 + lane;
#pragma unroll
    for (int r = 0; r < kMergeRows; ++r) {
      lse_own[r] = (s < n_split && r < nr) ? __ldcg(a.part_lse + (base + s) * M + m0 + r)
                                           : -INFINITY;
      Mx[r] = fmaxf(Mx[r], lse_own[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mx[r] = fmaxf(Mx[r], __shfl_xor_sync(0xffffffffu, Mx[r], o));
    if (Mx[r] == -INFINITY) Mx[r] = 0.f;
  }
  for (int s0 = 0; s0 < n_split; s0 += 32) {
    const int s = s0 + lane;
    float wl[kMergeRows];
#pragma unroll
    for (int r = 0; r < kMergeRows; ++r) {
      // the LSEs of the last group of 32 splits are still in registers
      const float l = (s0 + 32 >= n_split) ? lse_own[r]
                      : ((s < n_split && r < nr) ? __ldcg(a.part_lse + (base + s) * M + m0 + r)
                                                 : -INFINITY);
      wl[r] = __expf(l - Mx[r]);
      wsum[r] += wl[r];
    }
    const int ns = n_split - s0 < 32 ? n_split - s0 : 32;
    for (int j = 0; j < ns; j += 2) {
      const bool two = j + 1 < ns;
      const float* po0 = a.part_o + ((base + s0 + j) * M + m0) * kD;
      const float* po1 = po0 + static_cast<long long>(M) * kD;
      float4 v0[kMergeRows], v1[kMergeRows];
#pragma unroll
      for (int r = 0; r < kMergeRows; ++r) {
        if (r < nr) {
          v0[r] = __ldcg(reinterpret_cast<const float4*>(po0 + r * kD) + lane);
          if (two) v1[r] = __ldcg(reinterpret_cast<const float4*>(po1 + r * kD) + lane);
        }
      }
#pragma unroll
      for (int r = 0; r < kMergeRows; ++r) {
        const float w0 = __shfl_sync(0xffffffffu, wl[r], j);
        const float w1 = __shfl_sync(0xffffffffu, wl[r], two ? j + 1 : j);
        if (r < nr) {
          acc[r].x += w0 * v0[r].x;
          acc[r].y += w0 * v0[r].y;
          acc[r].z += w0 * v0[r].z;
          acc[r].w += w0 * v0[r].w;
          if (two) {
            acc[r].x += w1 * v1[r].x;
            acc[r].y += w1 * v1[r].y;
            acc[r].z += w1 * v1[r].z;
            acc[r].w += w1 * v1[r].w;
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum[r] += __shfl_xor_sync(0xffffffffu, wsum[r], o);
    if (r >= nr) continue;
    const int m = m0 + r;
    const int qrow = q_row0 + m / G;
    if (qrow < 0 || qrow >= a.q_rows) continue;
    const float sc = wsum[r] > 0.f ? a.out_scale / wsum[r] : 0.f;
    const long long orow = static_cast<long long>(qrow) * a.Hq + g * G + m % G;
    store_out4(a.out, orow * kD + lane * 4,
               make_float4(acc[r].x * sc, acc[r].y * sc, acc[r].z * sc, acc[r].w * sc),
               a.out_dtype);
    if (a.lse && lane == 0) a.lse[orow] = wsum[r] > 0.f ? Mx[r] + __logf(wsum[r]) : -INFINITY;
  }
}

// NRB: 16-row blocks per item (1, 2 or 4).  ROWMASK: rows differ in their visible keys
// (causal mask with several queries per item); otherwise every row sees the whole split.
template <int NRB, bool ROWMASK>
__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap qmap, DecodeLaunch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = smem_align<1024>(smem_raw);
  const int G = a.Hq / a.Hkv;
  const int M = a.rows;
  const int qhalf = q_half_bytes(M);
  uint8_t* qslots = tiles + kStages * kStageBytes;
  DecodeSmem* sm = reinterpret_cast<DecodeSmem*>(qslots + kItemSlots * 2 * qhalf);

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
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
  }
  // everything below reads the plan, which the launch before this one writes
  grid_dependency_wait();
  if (threadIdx.x == 0) sm->skip = launch_aborted(a.status) ? 1 : 0;
  __syncthreads();
  if (sm->skip) return;
  const int n_items = a.Hkv * a.split_offset[a.B];
  volatile int* abort_flag = &sm->abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------ producer (whole warp) -----------------------------
    // Lane p handles page piece p of every stage (R keys of one page); the page ids of the
    // next stage are loaded while the current stage is issued.
    const int ps = a.page_size;
    const int R = page_piece_rows(ps, kStageKeys);
    const int pieces = kStageKeys / R;                       // <= 8 (pieces of >= 8 keys)
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
      item = __ldg(a.order + item);
      const SplitItem it = a.items[item];
      if (lane == 0) {
        sm->item_id[islot] = item;
        uint8_t* qdst = qslots + islot * 2 * qhalf;
        // box: 64 columns x G heads x (M / G) queries; rows past the tensor read as zero
        const int q_row0 = a.qo_indptr ? __ldg(a.qo_indptr + it.b) : it.b * a.q_len;
        mbar_arrive_expect_tx(&sm->item_full[islot], 2u * M * 128u);
        tma_load_3d(qdst, &qmap, &sm->item_full[islot], 0, it.g * G, q_row0);
        tma_load_3d(qdst + qhalf, &qmap, &sm->item_full[islot], 64, it.g * G, q_row0);
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
        const int nq = a.qo_indptr ? a.qo_indptr[b + 1] - a.qo_indptr[b] : a.q_len;
        const int q_row0 = a.qo_indptr ? a.qo_indptr[b] : b * a.q_len;
        const int live_rows = nq <= 0 ? 0 : (nq * G < M ? nq * G : M);
        for (int m0 = 0; m0 < live_rows; m0 += kMergeRows)
          merge_rows(a, base, n_split, M, G, m0, live_rows, q_row0, g, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->merge_empty[js]);
    }
  } else {
    // ------------------------------ consumers ------------------------------------------
    const int gr = lane >> 2, tq = lane & 3;   // fragment row group, thread-in-quad
    const float sl2 = a.scale_log2;
    constexpr int nrb = NRB;
    constexpr int kg = kConsumerWarps / NRB;    // key slices per stage
    const int rb = warp / kg, kq = warp % kg;   // this warp's row block and key slice
    constexpr int slice_keys = kStageKeys / kg; // 16 * NRB
    int sg = 0;
    int jcount = 0;                            // merge jobs handed to the merge warp
    // The consumer warps meet at named barriers every item, so they leave the item loop
    // only together: each failed wait is carried to a barrier whose reduction (bar.red.or)
    // tells every warp.
    for (int icount = 0;; ++icount) {
      const int islot = icount % kItemSlots;
      const bool got = mbar_wait_warp(&sm->item_full[islot], (icount / kItemSlots) & 1,
                                      a.status, abort_flag);
      if (named_bar_or(1, kConsumerWarps * 32, !got)) break;
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
      const int nq = a.qo_indptr ? a.qo_indptr[b + 1] - a.qo_indptr[b] : a.q_len;
      const int q_row0 = a.qo_indptr ? a.qo_indptr[b] : b * a.q_len;
      const int L = a.seq_lens[b];
      // keys [klo, khi) of the split that each of this lane's two rows sees: query i sits at
      // L - nq + i; rows past the item's queries keep the split range (never written)
      int klo[2], khi[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = rb * 16 + gr + r * 8;
        const int i = row / G;
        klo[r] = kv_begin;
        khi[r] = kv_end;
        if (ROWMASK && row < M && i < nq) {
          const long long pos = static_cast<long long>(L) - nq + i;
          if (a.causal && pos + 1 < khi[r]) khi[r] = static_cast<int>(pos + 1);
          if (a.window_left >= 0 && pos - a.window_left > klo[r])
            klo[r] = static_cast<int>(pos - a.window_left);
        }
      }
      // Q as the A operand from the item's Q slot: rows rb * 16 .. + 15 (rows >= M: 0)
      uint32_t qa[kD / 16][4];
      {
        const uint8_t* qs = qslots + islot * 2 * qhalf;
        auto ld = [&](int row, int col) -> uint32_t {
          if (row >= M) return 0u;
          return *reinterpret_cast<const uint32_t*>(
              qs + (col >> 6) * qhalf + swz(row, (col & 63) >> 3) + (col & 7) * 2);
        };
        const int r0 = rb * 16 + gr;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const int c0 = ks * 16 + tq * 2;
          qa[ks][0] = ld(r0, c0);
          qa[ks][1] = ld(r0 + 8, c0);
          qa[ks][2] = ld(r0, c0 + 8);
          qa[ks][3] = ld(r0 + 8, c0 + 8);
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
#pragma unroll 1
        for (int sub = 0; sub < nrb; ++sub) {
          const int key0 = kq * slice_keys + sub * 16;          // within the stage
          const int kbase = first_key + s * kStageKeys + key0;   // first key of the step

          // ---- 16 keys of K and V into registers; after the slice's last step the stage
          // is released at once (except the item's last stage, which the combine reuses),
          // so the producer refills it while the warp computes --------------------------
          const int mi = lane >> 3, r8 = lane & 7;
          uint32_t kb[kD / 16][4], vb[kD / 16][4];
          {
            const uint32_t key_local = key0 + (mi >> 1) * 8 + r8;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
              const int dim = ks * 16 + (mi & 1) * 8;
              ldsm_x4(kt + (dim >> 6) * kHalfBytes + swz(key_local, (dim & 63) >> 3), kb[ks][0],
                      kb[ks][1], kb[ks][2], kb[ks][3]);
            }
          }
          {
            const uint32_t key_local = key0 + (mi & 1) * 8 + r8;
#pragma unroll
            for (int j = 0; j < kD / 8; j += 2) {
              const int dim = (j + (mi >> 1)) * 8;
              ldsm_x4_t(vt + (dim >> 6) * kHalfBytes + swz(key_local, (dim & 63) >> 3),
                        vb[j >> 1][0], vb[j >> 1][1], vb[j >> 1][2], vb[j >> 1][3]);
            }
          }
          __syncwarp();
          if (lane == 0 && sub == nrb - 1 && s + 1 < n_stages) mbar_arrive(&sm->empty[slot]);

          // ---- S = Q K^T over the step's 16 keys ----------------------------------------
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
          // ---- mask + online softmax (rows gr and gr + 8) --------------------------------
          // V rows outside the split may be stale or unused pool rows: zeroed for the MMA
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
              const int r = e >> 1;
              const int key = kbase + nt * 8 + tq * 2 + (e & 1);
              const float x = key >= klo[r] && key < khi[r] ? sc[nt][e] * sl2 : -INFINITY;
              sc[nt][e] = x;
              mx[r] = fmaxf(mx[r], x);
            }
          // lazily moved maximum: the reference only moves when a step exceeds it by more
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
          // ---- O += P V -------------------------------------------------------------
          const uint32_t aP[4] = {pa_[0], pa_[1], pa_[2], pa_[3]};
          // keys of this lane inside the B fragments: 2tq, 2tq+1 (b0) and 8+2tq, 8+2tq+1 (b1)
          const uint32_t m_lo = (vk[0][0] ? 0x0000FFFFu : 0u) | (vk[0][1] ? 0xFFFF0000u : 0u);
          const uint32_t m_hi = (vk[1][0] ? 0x0000FFFFu : 0u) | (vk[1][1] ? 0xFFFF0000u : 0u);
          {
#pragma unroll
            for (int j = 0; j < kD / 8; j += 2) {
              uint32_t b0 = vb[j >> 1][0], b1 = vb[j >> 1][1], b2 = vb[j >> 1][2],
                       b3 = vb[j >> 1][3];
              if (any_invalid) {
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
      }
      if (named_bar_or(1, kConsumerWarps * 32, !ok)) break;   // some warp's stage wait failed

      // ---- combine the key slices of each row ---------------------------------------------
      // red_o [kg][M][128] fp32 in the item's last stage, which no warp reads any more once
      // all have passed the first barrier; the stage is released after the last one.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
      }
      const bool have_stage = n_stages > 0;
      const int last_slot = have_stage ? (sg - 1) % kStages : 0;
      float* red_o = reinterpret_cast<float*>(tiles + last_slot * kStageBytes);
      if (have_stage) {
        named_bar(1, kConsumerWarps * 32);   // every warp is done with the last stage's K/V
        const int r0 = rb * 16 + gr;
#pragma unroll
        for (int j = 0; j < kD / 8; ++j) {
          const int col = j * 8 + tq * 2;
          if (r0 < M) {
            float* p0 = red_o + (kq * M + r0) * kD + col;
            p0[0] = o[j][0];
            p0[1] = o[j][1];
          }
          if (r0 + 8 < M) {
            float* p1 = red_o + (kq * M + r0 + 8) * kD + col;
            p1[0] = o[j][2];
            p1[1] = o[j][3];
          }
        }
        if (tq == 0) {
          if (r0 < M) {
            sm->red_m[kq * M + r0] = m_run[0];
            sm->red_l[kq * M + r0] = l_run[0];
          }
          if (r0 + 8 < M) {
            sm->red_m[kq * M + r0 + 8] = m_run[1];
            sm->red_l[kq * M + r0 + 8] = l_run[1];
          }
        }
      }
      named_bar(1, kConsumerWarps * 32);
      const int d = threadIdx.x;   // 0..127: one output column
      const int n_split = a.split_offset[b + 1] - a.split_offset[b];
      const int live_rows = nq <= 0 ? 0 : (nq * G < M ? nq * G : M);
      for (int m = 0; m < live_rows; ++m) {
        float Mx = -INFINITY;
        float Lsum = 0.f, acc = 0.f;
        if (have_stage) {
          for (int w = 0; w < kg; ++w) Mx = fmaxf(Mx, sm->red_m[w * M + m]);
          const float Mu = Mx == -INFINITY ? 0.f : Mx;
          for (int w = 0; w < kg; ++w) {
            const float f = fast_exp2(sm->red_m[w * M + m] - Mu);
            Lsum += f * sm->red_l[w * M + m];
            acc += f * red_o[(w * M + m) * kD + d];
          }
          Mx = Mu;
        }
        const float on = Lsum > 0.f ? acc / Lsum : 0.f;
        const float lse_nat = Lsum > 0.f ? (Mx + fast_log2(Lsum)) * kLn2 : -INFINITY;
        if (n_split == 1) {
          const int qrow = q_row0 + m / G;
          if (qrow < 0 || qrow >= a.q_rows) continue;
          const long long orow = static_cast<long long>(qrow) * a.Hq + g * G + m % G;
          store_out1(a.out, orow * kD + d, on * a.out_scale, a.out_dtype);
          if (a.lse && d == 0) a.lse[orow] = lse_nat;
        } else {
          const long long prow = static_cast<long long>(item) * M + m;
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
      named_bar(1, kConsumerWarps * 32);   // the combine is read: the stage goes back
      if (have_stage && lane == 0) mbar_arrive(&sm->empty[last_slot]);
    }
  }
}

template <int NRB, bool ROWMASK>
int launch_decode_t(const DecodeLaunch& a, cudaStream_t st) {
  static std::atomic<uint64_t> smem_set{0};
  if (!kernel_smem_ready(decode_split_kernel<NRB, ROWMASK>, smem_bytes(kMaxRows), smem_set))
    return -1;
  const int smem = smem_bytes(a.rows);
  const int per_sm = 2 * (smem + 1024) <= 228 * 1024 ? 2 : 1;
  const int sms = current_sm_count();
  if (sms <= 0) return -1;
  if (a.capacity > 0) {
    const int grid = a.capacity < per_sm * sms ? a.capacity : per_sm * sms;
    void* tok;
    timer_begin(st, &tok);
    // programmatic dependent launch: the CTAs start their prologue while the planner runs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_split_kernel<NRB, ROWMASK>, *a.kmap, *a.vmap, *a.qmap,
                           a) != cudaSuccess)
      return -1;
    timer_end(st, tok);
    count_launches(1);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_decode(const DecodeLaunch& a, cudaStream_t st) {
  if (a.rows < 1 || a.rows > kMaxRows || (a.nrb != 1 && a.nrb != 2 && a.nrb != 4) ||
      a.rows > 16 * a.nrb)
    return -1;
  const int G = a.Hq / a.Hkv;
  const bool rowmask = a.causal && a.rows > G;   // several queries per item
  switch (a.nrb * 2 + (rowmask ? 1 : 0)) {
    case 2: return launch_decode_t<1, false>(a, st);
    case 3: return launch_decode_t<1, true>(a, st);
    case 4: return launch_decode_t<2, false>(a, st);
    case 5: return launch_decode_t<2, true>(a, st);
    case 8: return launch_decode_t<4, false>(a, st);
    default: return launch_decode_t<4, true>(a, st);
  }
}

}  // namespace pa
