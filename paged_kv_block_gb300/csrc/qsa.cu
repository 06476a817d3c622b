// Per-query block-bitmap attention forward (FlashInfer page qsa_forward) on tcgen05.
//
// One CTA per (query token t, pair of KV heads g0, g0 + 1).  The planner has already turned
// row t of the bitmap into the ascending list of selected blocks that meet [lo[t], hi[t]];
// every block holds block_size = 4 key tokens.  With the cache laid out [T, Hkv, D], the
// rows of one block for two neighbouring KV heads, 64 columns of d at a time, form a
// [4 tokens][2 heads][64 d] box of 8 rows x 128 B: one 128-byte-swizzle atom.  One copy
// (a 4-D box) brings the four such atoms (the four 64-column chunks) of a block, so the
// gather is one 4 KB copy per block landing directly in the layout the tensor core reads.  The key
// rows of a tile are (block, token, head) triples; the MMA's N dimension holds the query
// heads of both KV heads, and the cross pairs (a key row of one head against a query head
// of the other) are masked out of the softmax, so each head sees exactly its own attention.
// The work is bound by the L2 -> SM gather (the unique K/V is a few tens of MB, read many
// times), so the MMAs take the key rows as the M dimension:
//   S^T [128 rows x 32] = K_tile [128 x 256] * Q^T        (Q: 2 x G heads, each group
//                                                            padded to 16)
//   O^T [256 d x 32]   += V_tile^T [256 x 128] * P^T      (two M = 128 halves of d)
// A tile is K then V, each 64 KB laid out [16 blocks][4 chunks][8 rows][128 B], so the MMAs
// see 16 blocks at a 4 KB stride.  The copies run as two independent pipelines, one per half
// of the blocks (0-7 and 8-15), each with its own full barriers: the copy rate of one
// pipeline (one chain of stage barriers) saturates well below the SM's, and two pipelines
// nearly double it.  A slot is released to both pipelines by one barrier.  The two
// pipelines' 32 KB slots interleave into three 64 KB pair slots.  Units are copied in the
// order the MMAs consume them, K(0), K(1), V(0), K(2), V(1), ..., V(N - 1):
// S^T(n + 1) is computed before PV(n), so K(n + 1) can be in flight two tiles ahead and the
// softmax of one tile follows the previous one without waiting for a copy.
// Roles (288 threads):
//   warps 0-3  producers: per tile publish the key-row table (token of each row, or dead),
//              fetching the next tile's block spans a tile ahead; warps 2p and 2p + 1 form
//              pipeline p and copy blocks 8p .. 8p + 3 and 8p + 4 .. 8p + 7
//   warps 4-7  softmax: thread = key row (TMEM lane) of S^T and = d row of O^T; column
//              maxima per head group from redux.sync plus a shared-memory exchange; rows
//              that are dead but were loaded from memory get their V row zeroed, so
//              non-finite data outside the selection cannot reach the output.
//   warp 8     TMEM owner and MMA issuer (one thread)
#include <cstdint>
#include <cuda_bf16.h>

#include "../../include/paged_attn.h"
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kD = 256;
constexpr int kGroupCols = 16;                // query heads of one KV head, padded
constexpr int kN = 2 * kGroupCols;            // MMA N: the query heads of both KV heads
constexpr int kBlocksPerTile = 16;
constexpr int kRows = kBlocksPerTile * 8;     // key rows per tile (MMA M)
constexpr int kBlockBytes = 4096;             // one block: four 8-row atoms (64-column chunks)
constexpr int kHalfBytes = 8 * kBlockBytes;   // 8 blocks: one pipeline's part of a K or V tile
constexpr int kPairBytes = 2 * kHalfBytes;    // a K or V tile: both pipelines' halves
constexpr int kUnitsPerTile = 2;              // K, V
constexpr int kPairs = 3;                     // pair slots: K(n), V(n), K(n + 1) in flight
constexpr int kPipes = 2;
constexpr int kProducers = 4;                 // producer warps, two per pipeline
constexpr int kBlocksPerProducer = kBlocksPerTile / kProducers;   // 4
constexpr int kTabBufs = 4;                   // row tables in flight (the producer runs <= 2 ahead)
constexpr int kMmaWarp = 8;
constexpr int kThreads = 288;
constexpr int kTmemCols = 128;                // S^T buffers at 0 and 96, O^T halves at 32, 64
__device__ __forceinline__ uint32_t s_col(int n) { return (n & 1) ? 96u : 0u; }
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
// key-row codes of the per-tile table
constexpr int8_t kLive = 1;                   // a selected token inside [lo, hi]
constexpr int8_t kDeadLoaded = -1;            // row outside the selection, loaded from memory
constexpr int8_t kDeadZero = 0;               // row the copy fills with zeros (out of range)

struct QsaCtrl {
  uint64_t full[kPipes][kPairs];
  // empty[slot]: the MMAs that read the unit in that slot have completed (one barrier for
  // both pipelines).  For a K unit that is also "S^T of its tile is ready": the softmax waits
  // on it, which is safe because the slot's next phase belongs to V of the same tile, whose
  // PV needs that softmax's P^T first.
  uint64_t empty[kPairs];
  uint64_t tab_full[kTabBufs];
  uint64_t p_full[2];                         // P^T of tiles n with n % 2 = index written
  uint64_t pv_done[2];                        // PV of tiles n with n % 2 = index complete
  uint64_t q_full, q_empty, o_full, o_empty;
  uint32_t tmem_base;
  int abort_flag;
  int8_t tab[kTabBufs][kRows];
  float4 red[4][kN / 4];                      // per-warp column maxima
  float lred[4][kN];
};

constexpr int kQBytes = 4 * kN * 128;         // 4 d-chunks of [32 rows][128 B]
constexpr int kPBytes = 2 * kN * 128;         // one P^T: 2 key-row halves of [32 rows][128 B]
constexpr int kPBufs = 2;
constexpr int kSmemBytes =
    kPairs * kPairBytes + kQBytes + kPBufs * kPBytes + sizeof(QsaCtrl) + 1024;
static_assert(kSmemBytes <= 232448, "qsa_kernel exceeds the per-CTA shared memory limit");

struct QsaLaunch {
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
  int T, Hq, Hkv, G, pairs;
  float scale_log2;
};

__device__ __forceinline__ int f2ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// Position of K(n) and V(n) in the copy order K(0), K(1), V(0), K(2), V(1), ..., V(N - 1).
__device__ __forceinline__ int unit_k(int n) { return n == 0 ? 0 : 2 * n - 1; }
__device__ __forceinline__ int unit_v(int n, int N) { return n == N - 1 ? 2 * N - 1 : 2 * n + 2; }

// Row r of V of tile n (unit u of the pair sequence) is zeroed once its copy has landed: P is
// 0 there, but 0 x (inf or NaN) would not be.
__device__ __noinline__ bool zero_dead_v_row(QsaCtrl* ctl, uint8_t* ring, int u, int r,
                                             uint32_t* status, volatile int* abort_flag) {
  const int j = r >> 3, ps = u % kPairs;
  if (!mbar_wait(&ctl->full[j >> 3][ps], (u / kPairs) & 1, status, abort_flag)) return false;
  for (int c = 0; c < 4; ++c) {
    uint4* row = reinterpret_cast<uint4*>(ring + ps * kPairBytes + j * kBlockBytes + c * 1024 +
                                          (r & 7) * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) row[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  return true;
}

// O^T columns c *= alpha of column c (held by lane c), both d halves of this warp's lanes.
__device__ __noinline__ void rescale_o(uint32_t taddr, float alpha_c) {
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t ov[kN];
    tmem_ld32(taddr + 32 * hh, ov);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < kN; ++c)
      ov[c] = __float_as_uint(__uint_as_float(ov[c]) * __shfl_sync(0xffffffffu, alpha_c, c));
    tmem_st32(taddr + 32 * hh, ov);
  }
  tmem_st_wait();
}

// Normalise and store this thread's d rows (r, r + 128) of every live column; lane c holds
// the running maximum of column c.  Both O^T halves come in with two 32-column TMEM loads
// and one wait; the scalars of the launch are passed by value so that they stay in
// registers (a reference to the kernel parameter would place it in local memory).  Lanes
// 2i and 2i + 1 trade one value per column pair, so that each stores two adjacent d of one
// column (a bf16x2 and a float2 store instead of two of each width).
__device__ __forceinline__ void write_output(__nv_bfloat16* __restrict__ out,
                                             float* __restrict__ out32, float* __restrict__ lse,
                                             int Hq, int G, int T, const QsaCtrl* ctl,
                                             uint32_t taddr, bool have_o, int t, int g0,
                                             bool two, int r, int lane, float m_c) {
  const float L_c = ctl->lred[0][lane] + ctl->lred[1][lane] + ctl->lred[2][lane] +
                    ctl->lred[3][lane];
  const float inv_c = L_c > 0.f ? 1.f / L_c : 0.f;
  uint32_t o0[kN], o1[kN];
  if (have_o) {
    tc_fence_after();
    tmem_ld32(taddr, o0);
    tmem_ld32(taddr + 32, o1);
    tmem_ld_wait();
  } else {
#pragma unroll
    for (int c = 0; c < kN; ++c) o0[c] = o1[c] = 0u;
  }
  const bool odd = lane & 1;
  const long long row0 = static_cast<long long>(t) * Hq * kD + (r & ~1);   // d of the pair
#pragma unroll
  for (int c = 0; c < kN; c += 2) {
    // this lane's d row in both columns, each scaled by its column's 1 / l
    const float inv_a = __shfl_sync(0xffffffffu, inv_c, c);
    const float inv_b = __shfl_sync(0xffffffffu, inv_c, c + 1);
    const float a0 = __uint_as_float(o0[c]) * inv_a, a1 = __uint_as_float(o1[c]) * inv_a;
    const float b0 = __uint_as_float(o0[c + 1]) * inv_b, b1 = __uint_as_float(o1[c + 1]) * inv_b;
    // the even lane keeps column c, the odd lane column c + 1; each sends the other one
    const float x0 = __shfl_xor_sync(0xffffffffu, odd ? a0 : b0, 1);
    const float x1 = __shfl_xor_sync(0xffffffffu, odd ? a1 : b1, 1);
    const int cc = c + (odd ? 1 : 0);
    const int gq = cc / kGroupCols, h = cc % kGroupCols;
    if (h >= G || (gq == 1 && !two)) continue;
    const float lo0 = odd ? x0 : a0, hi0 = odd ? b0 : x0;     // d, d + 1 (rows r & ~1, | 1)
    const float lo1 = odd ? x1 : a1, hi1 = odd ? b1 : x1;     // d + 128, d + 129
    const long long o = row0 + static_cast<long long>((g0 + gq) * G + h) * kD;
    *reinterpret_cast<__nv_bfloat162*>(out + o) = __floats2bfloat162_rn(lo0, hi0);
    *reinterpret_cast<__nv_bfloat162*>(out + o + 128) = __floats2bfloat162_rn(lo1, hi1);
    if (out32) {
      *reinterpret_cast<float2*>(out32 + o) = make_float2(lo0, hi0);
      *reinterpret_cast<float2*>(out32 + o + 128) = make_float2(lo1, hi1);
    }
  }
  // lse of column c from lane c of the first warp
  const int gq = lane / kGroupCols, h = lane % kGroupCols;
  if (r == lane && lse && h < G && (gq == 0 || two))
    lse[static_cast<long long>((g0 + gq) * G + h) * T + t] =
        L_c > 0.f ? (m_c + fast_log2(L_c)) * kLn2 : -INFINITY;
}

__global__ void __launch_bounds__(kThreads, 1)
qsa_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
           const __grid_constant__ CUtensorMap vmap, QsaLaunch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_align<1024>(smem_raw);
  uint8_t* ring = base;
  uint8_t* q_s = ring + kPairs * kPairBytes;
  uint8_t* p_s = q_s + kQBytes;
  QsaCtrl* ctl = reinterpret_cast<QsaCtrl*>(p_s + kPBufs * kPBytes);

  // one decision for the whole CTA: another CTA may set the status word meanwhile
  if (__syncthreads_or(launch_aborted(a.status))) return;
  const int jobs = a.T * a.pairs;                // (query token, KV-head pair) units of work
  const int G = a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The CTA walks jobs blockIdx.x, + gridDim.x, ...; every counter below runs over the whole
  // walk (units, tiles, jobs with tiles), so the rings' phases carry from job to job.
  struct Job {
    int t, g0, beg, nblk, N, lo, hi;
    bool two;
  };
  auto job_of = [&](int jj) -> Job {
    Job jb;
    jb.t = jj / a.pairs;
    jb.g0 = 2 * (jj % a.pairs);
    jb.two = jb.g0 + 1 < a.Hkv;
    jb.beg = __ldg(a.indptr + jb.t);
    jb.nblk = __ldg(a.indptr + jb.t + 1) - jb.beg;
    jb.N = jb.nblk > 0 ? (jb.nblk + kBlocksPerTile - 1) / kBlocksPerTile : 0;
    jb.lo = __ldg(a.lo + jb.t);
    jb.hi = __ldg(a.hi + jb.t);
    return jb;
  };

  // Q rows G..15 of each group and all of P^T start at zero: the copies never write the
  // former, and softmax writes only its own group's half of the latter.
  for (int i = threadIdx.x; i < (kQBytes + kPBufs * kPBytes) / 16; i += kThreads)
    *reinterpret_cast<uint4*>(q_s + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int p = 0; p < kPipes; ++p)
      for (int i = 0; i < kPairs; ++i) mbar_init(&ctl->full[p][i], kProducers / kPipes);
    for (int i = 0; i < kPairs; ++i) mbar_init(&ctl->empty[i], 1);
    for (int i = 0; i < kTabBufs; ++i) mbar_init(&ctl->tab_full[i], 32 * kProducers);
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    mbar_init(&ctl->pv_done[0], 1);
    mbar_init(&ctl->pv_done[1], 1);
    mbar_init(&ctl->p_full[0], 128);
    mbar_init(&ctl->p_full[1], 128);
    mbar_init(&ctl->o_full, 1);
    mbar_init(&ctl->o_empty, 128);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();   // the zeroes (generic proxy) before the copies (async proxy)
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp < kProducers) {
    // ================================ producers ===========================================
    const int pw = warp;
    if (pw == 0 && lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    // lane l < 4 of producer warp pw (pipeline pl = pw / 2) handles block 4 pw + l of each tile
    const int pl = pw / 2;
    const int jb = kBlocksPerProducer * pw + lane;
    int U = 0, gt = 0, jq = 0;                  // units, tiles, jobs with tiles so far
    int issued = 0, q_issued = 0;               // copies issued (units, Q loads)
    int first_t0 = a.T, first_t1 = a.T;  // token coordinate of this lane's block in tiles of parity 0/1
    bool ok = true;
    for (int jj = blockIdx.x; ok && jj < jobs; jj += gridDim.x) {
      const Job J = job_of(jj);
      if (J.N == 0) continue;
      const int S = kUnitsPerTile * J.N;
      if (pw == 0) {
        // Q of this job, once the previous job's last QK has read the buffer
        ok = jq == 0 || mbar_wait_warp(&ctl->q_empty, (jq - 1) & 1, a.status, abort_flag);
        if (!ok) break;
        if (lane == 0)
          mbar_arrive_expect_tx(&ctl->q_full, (J.two ? 8u : 4u) * static_cast<uint32_t>(G) * 128u);
        __syncwarp();
        if (lane < (J.two ? 8 : 4)) {                  // Q: d chunk lane & 3, group lane >> 2
          const int c = lane & 3, gg = lane >> 2;
          tma_load_3d(q_s + c * (kN * 128) + gg * (kGroupCols * 128), &qmap, &ctl->q_full,
                      c * 64, (J.g0 + gg) * G, J.t);
        }
        ++q_issued;
      }
      auto block_of = [&](int n) -> int {
        const int i = n * kBlocksPerTile + jb;
        return (lane < kBlocksPerProducer && n < J.N && i < J.nblk) ? __ldg(a.indices + J.beg + i)
                                                                   : -1;
      };
      // block spans are fetched two tiles ahead of their publication: block ids of tile
      // n + 2 and first/last tokens of tile n + 1 are in flight while tile n is published
      int b_cur = block_of(0), first_cur = 0, last_cur = -1;
      if (b_cur >= 0) {
        first_cur = __ldg(a.bfirst + b_cur);
        last_cur = __ldg(a.blast + b_cur);
      }
      int b_nx = block_of(1);
      for (int s = 0; s < S; ++s) {
        // unit s: K(n) or V(n) in the consumption order
        const bool is_k = s == 0 || (s & 1 && s != S - 1);
        const int n = s == 0 ? 0 : (is_k ? (s + 1) >> 1 : (s == S - 1 ? J.N - 1 : (s - 2) >> 1));
        const int u = U + s, ps = u % kPairs, g = gt + n;
        if (is_k) {                                    // publish tile n's rows
          const int f = b_cur >= 0 ? first_cur : a.T;
          if (g & 1) first_t1 = f; else first_t0 = f;
          if (lane < kBlocksPerProducer) {
            int8_t* tab = ctl->tab[g % kTabBufs] + jb * 8;
#pragma unroll
            for (int o = 0; o < 4; ++o) {
              const int tok = first_cur + o;
#pragma unroll
              for (int gg = 0; gg < 2; ++gg) {
                int8_t code;
                if (b_cur < 0 || tok >= a.T || (gg == 1 && !J.two)) code = kDeadZero;
                else if (tok <= last_cur && tok >= J.lo && tok <= J.hi) code = kLive;
                else code = kDeadLoaded;
                tab[o * 2 + gg] = code;                // row = token offset * 2 + head
              }
            }
          }
          mbar_arrive(&ctl->tab_full[g % kTabBufs]);
          // advance the prefetch: spans of tile n + 1 (ids fetched a tile ago), ids of n + 2
          b_cur = b_nx;
          if (b_cur >= 0) {
            first_cur = __ldg(a.bfirst + b_cur);
            last_cur = __ldg(a.blast + b_cur);
          }
          b_nx = block_of(n + 2);
        }
        if (u >= kPairs &&
            !mbar_wait_warp(&ctl->empty[ps], ((u / kPairs) - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&ctl->full[pl][ps], kBlocksPerProducer * kBlockBytes);
        __syncwarp();
        if (lane < kBlocksPerProducer)
          tma_load_4d(ring + ps * kPairBytes + jb * kBlockBytes, is_k ? &kmap : &vmap,
                      &ctl->full[pl][ps], 0, J.g0, (g & 1) ? first_t1 : first_t0, 0);
        issued = u + 1;
      }
      if (!ok) break;
      U += S;
      gt += J.N;
      ++jq;
    }
    if (*abort_flag && lane == 0) {                    // copies still in flight after an abort
      for (int u = issued > kPairs ? issued - kPairs : 0; u < issued; ++u)
        drain_wait(&ctl->full[pl][u % kPairs], (u / kPairs) & 1);
      if (pw == 0 && q_issued > 0) drain_wait(&ctl->q_full, (q_issued - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ================================ MMA issuer ==========================================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, kN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, kN, true, false);
      const uint32_t ring_addr = smem_u32(ring), q_addr = smem_u32(q_s), p_addr = smem_u32(p_s);
      int U = 0, gt = 0, jq = 0;
      bool ok = true;
      for (int jj = blockIdx.x; ok && jj < jobs; jj += gridDim.x) {
        const int t = jj / a.pairs;
        const int nblk = __ldg(a.indptr + t + 1) - __ldg(a.indptr + t);
        const int N = nblk > 0 ? (nblk + kBlocksPerTile - 1) / kBlocksPerTile : 0;
        if (N == 0) continue;
        // S^T of tile n + 1 is computed while softmax works on tile n (two S^T buffers,
        // indexed by the tile count of the whole walk), so softmax runs tile after tile
        // without waiting for an MMA round trip.
        auto issue_qk = [&](int n) -> bool {
          const int u = U + unit_k(n), sk = u % kPairs;
          if (!mbar_wait(&ctl->full[0][sk], (u / kPairs) & 1, a.status, abort_flag) ||
              !mbar_wait(&ctl->full[1][sk], (u / kPairs) & 1, a.status, abort_flag))
            return false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 16; ++k) {               // chunk k / 4, 16 columns (k % 4)
            const uint32_t ka = ring_addr + sk * kPairBytes + (k >> 2) * 1024 + (k & 3) * 32;
            const uint32_t qa = q_addr + (k >> 2) * (kN * 128) + (k & 3) * 32;
            mma_ss(tmem + s_col(gt + n), sdesc_sw128(ka, 16, kBlockBytes),
                   sdesc_sw128(qa, 16, 1024), idesc_qk, k > 0);
          }
          mma_commit(&ctl->empty[sk]);                 // K(n) read, S^T(n) ready
          if (n == N - 1) mma_commit(&ctl->q_empty);   // the job's Q is no longer read
          return true;
        };
        ok = mbar_wait(&ctl->q_full, jq & 1, a.status, abort_flag) && issue_qk(0);
        for (int n = 0; ok && n < N; ++n) {
          const int g = gt + n;
          // S^T(n + 1) may reuse buffer (g + 1) % 2: softmax(g - 1) finished with it before
          // PV(g - 1) was issued
          if (n + 1 < N && !issue_qk(n + 1)) {
            ok = false;
            break;
          }
          // O^T[d half h] += V^T P^T over both V units (blocks 0-7, 8-15); the first PV of a
          // job overwrites O^T, once the previous job's epilogue has read it
          const int u = U + unit_v(n, N), sv = u % kPairs;
          if (!mbar_wait(&ctl->p_full[g & 1], (g >> 1) & 1, a.status, abort_flag) ||
              !mbar_wait(&ctl->full[0][sv], (u / kPairs) & 1, a.status, abort_flag) ||
              !mbar_wait(&ctl->full[1][sv], (u / kPairs) & 1, a.status, abort_flag) ||
              (n == 0 && jq > 0 &&
               !mbar_wait(&ctl->o_empty, (jq - 1) & 1, a.status, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {           // 16 key rows = 2 blocks per step
              const uint32_t va = ring_addr + sv * kPairBytes + h * 2048 + ks * 2 * kBlockBytes;
              const uint32_t pa = p_addr + (g & 1) * kPBytes + (ks >> 2) * (kN * 128) + (ks & 3) * 32;
              mma_ss(tmem + 32 + 32 * h, sdesc_sw128(va, 1024, kBlockBytes),
                     sdesc_sw128(pa, 16, 1024), idesc_pv, (n > 0 || ks > 0));
            }
          }
          mma_commit(&ctl->empty[sv]);
          mma_commit(&ctl->pv_done[g & 1]);
          if (n == N - 1) mma_commit(&ctl->o_full);
        }
        U += kUnitsPerTile * N;
        gt += N;
        ++jq;
      }
    }
  } else if (warp >= 4) {
    // ================================ softmax =============================================
    const int wq = warp & 3;                           // TMEM lane quadrant of this warp
    const int r = wq * 32 + lane;                      // key row of S^T, d row of O^T
    const int gg = lane & 1;                           // KV head of row r within the pair
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    const int ord_ninf = f2ord(-INFINITY);
    int gt = 0, jq = 0;
    bool alive = true;
    for (int jj = blockIdx.x; alive && jj < jobs; jj += gridDim.x) {
      const int t = jj / a.pairs, g0 = 2 * (jj % a.pairs);
      const bool two = g0 + 1 < a.Hkv;
      const int nblk = __ldg(a.indptr + t + 1) - __ldg(a.indptr + t);
      const int N = nblk > 0 ? (nblk + kBlocksPerTile - 1) / kBlocksPerTile : 0;
      // Column bookkeeping is spread over the lanes: lane c of every warp keeps the running
      // maximum of S^T column c (query head c % 16 of KV head g0 + c / 16); each warp holds
      // an identical copy.  Rows read their 16 columns' values by shuffles, so the per-tile
      // code stays short.
      float m_c = -INFINITY;
      float l[kGroupCols];
#pragma unroll
      for (int h = 0; h < kGroupCols; ++h) l[h] = 0.f;
      // The four softmax warps meet at named barriers every tile, so they must take the same
      // path through the loop: a failed wait does not leave the loop at once but is carried
      // in `ok` to the tile's first barrier, whose reduction tells every warp to leave
      // together.
      for (int n = 0; n < N; ++n) {
        const int g = gt + n;
        const int uk = 2 * gt + unit_k(n);             // S^T(n) ready = K(n)'s slot released
        bool ok = mbar_wait_warp(&ctl->empty[uk % kPairs], (uk / kPairs) & 1, a.status, abort_flag);
        uint32_t sv[kN];
        if (ok) {
          tc_fence_after();
          tmem_ld32(tmem + lane_base + s_col(g), sv);
          tmem_ld_wait();
        }
        ok = ok && mbar_wait_warp(&ctl->tab_full[g % kTabBufs], (g / kTabBufs) & 1, a.status,
                                  abort_flag);
        const int code = ok ? ctl->tab[g % kTabBufs][r] : kDeadZero;
        const bool valid = code == kLive;
        float x[kGroupCols];
#pragma unroll
        for (int h = 0; h < kGroupCols; ++h)
          x[h] = (valid && h < G) ? __uint_as_float(gg ? sv[kGroupCols + h] : sv[h]) * sl2 : -INFINITY;
        if (named_bar_or(1, 128, !ok)) {               // some warp failed: all leave
          alive = false;
          break;
        }
        // The running maxima change only when some score exceeds them by the rescale
        // threshold, which after the first tile is rare: test for that first and compute the
        // exact column maxima of the tile only when it happens.
        bool exceed = false;
#pragma unroll
        for (int h = 0; h < kGroupCols; ++h)
          exceed |= x[h] > __shfl_sync(0xffffffffu, m_c, gg * kGroupCols + h) + kRescaleThreshold;
        float alpha_c = 1.f;
        if (named_bar_or(1, 128, exceed)) {
          float* red = reinterpret_cast<float*>(ctl->red[wq]);
#pragma unroll
          for (int h = 0; h < kGroupCols; ++h) {
            const int v = f2ord(x[h]);
            const int m0 = __reduce_max_sync(0xffffffffu, gg == 0 ? v : ord_ninf);
            const int m1 = __reduce_max_sync(0xffffffffu, gg == 1 ? v : ord_ninf);
            if (lane == 0) {
              red[h] = ord2f(m0);
              red[kGroupCols + h] = ord2f(m1);
            }
          }
          named_bar(1, 128);
          const float* rd = reinterpret_cast<const float*>(ctl->red);
          const float M =
              fmaxf(fmaxf(rd[lane], rd[kN + lane]), fmaxf(rd[2 * kN + lane], rd[3 * kN + lane]));
          if (M > m_c + kRescaleThreshold || (m_c == -INFINITY && M > -INFINITY)) {
            alpha_c = m_c == -INFINITY ? 0.f : fast_exp2(m_c - M);
            m_c = M;
          }
        }
        const bool need = __any_sync(0xffffffffu, alpha_c != 1.f);
        const float mu_c = m_c == -INFINITY ? 0.f : m_c;
        // P^T buffer g % 2 was read by PV(g - 2), which must have completed.  From here on
        // a failure skips the rest of the tile; the next tile's first barrier ends the loop.
        ok = g <= 1 || mbar_wait_warp(&ctl->pv_done[g & 1], ((g - 2) >> 1) & 1, a.status, abort_flag);
        if (ok) {
          // P^T [32 columns][128 rows], two K-major 64-row chunks with the 128-byte swizzle;
          // this thread writes its own group's 16 columns, the other group's stay zero
          uint8_t* prow = p_s + (g & 1) * kPBytes + (r >> 6) * (kN * 128);
          const int rr = r & 63;
#pragma unroll
          for (int h = 0; h < kGroupCols; ++h) {
            const int c = gg * kGroupCols + h;
            const float mu = __shfl_sync(0xffffffffu, mu_c, c);
            const float ac = __shfl_sync(0xffffffffu, alpha_c, c);
            const float pv = fast_exp2(x[h] - mu);
            l[h] = l[h] * ac + pv;
            *reinterpret_cast<__nv_bfloat16*>(prow + c * 128 + ((((rr >> 3) ^ (c & 7)) & 7) << 4) +
                                              (rr & 7) * 2) = __float2bfloat16_rn(pv);
          }
          if (code == kDeadLoaded)
            ok = zero_dead_v_row(ctl, ring, 2 * gt + unit_v(n, N), r, a.status, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && n > 0 && need) {
          // O^T is accumulated by PV(g - 1): it must have completed before the rescale
          ok = mbar_wait_warp(&ctl->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, a.status, abort_flag);
          if (ok) {
            tc_fence_after();
            rescale_o(tmem + lane_base + 32, alpha_c);
          }
        }
        fence_proxy_async_smem();   // P^T and zeroed V rows (generic) -> tensor-core reads
        tc_fence_before();
        mbar_arrive(&ctl->p_full[g & 1]);
      }
      if (!alive) break;
      // ---- epilogue: column sums, normalise, write out / out_fp32 / lse -------------------
      named_bar(1, 128);            // every warp has read the previous job's sums
#pragma unroll
      for (int h = 0; h < kGroupCols; ++h) {
        float v = l[h];
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);   // same group
        if (lane < 2) ctl->lred[wq][lane * kGroupCols + h] = v;
      }
      named_bar(1, 128);
      const bool have_o = N > 0 && mbar_wait_warp(&ctl->o_full, jq & 1, a.status, abort_flag);
      write_output(a.out, a.out32, a.lse, a.Hq, G, a.T, ctl, tmem + lane_base + 32, have_o, t,
                   g0, two, r, lane, m_c);
      if (N > 0) {
        // O^T has been read into registers: the next job's first PV may overwrite it
        tc_fence_before();
        mbar_arrive(&ctl->o_empty);
        gt += N;
        ++jq;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_qsa(const paged_attn_params* p, const paged_attn_meta* m, const void* q, const void* k,
               const void* v, void* out, float* out_fp32, float* lse, const int* indptr,
               const int* indices, uint32_t* status, cudaStream_t st) {
  const int G = p->num_qo_heads / p->num_kv_heads;
  if (G > kGroupCols || p->head_dim != kD) return PAGED_ATTN_ERR_UNSUPPORTED;
  if (!out || !m->lo_dev || !m->hi_dev || !m->block_first_dev || !m->block_last_dev)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(out_fp32)) & 15u)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const int pairs = (p->num_kv_heads + 1) / 2;
  const long long units = static_cast<long long>(p->q_len) * pairs;
  if (units == 0) return PAGED_ATTN_OK;
  if (units >= (1LL << 31)) return PAGED_ATTN_ERR_UNSUPPORTED;
  CUtensorMap qmap, kmap, vmap;
  // Q [T, Hq, D]: box = the G query heads of one KV head, 64 columns; K and V [T, Hkv, D]:
  // box = 4 tokens x 2 KV heads x two 64-column chunks (two swizzle atoms)
  if (!encode_q_map(&qmap, q, p->q_len, p->num_qo_heads, kD, G, 1) ||
      !encode_block_pair_map(&kmap, k, p->q_len, p->num_kv_heads, kD) ||
      !encode_block_pair_map(&vmap, v, p->q_len, p->num_kv_heads, kD))
    return PAGED_ATTN_ERR_CUDA;
  static std::atomic<uint64_t> smem_set{0};
  if (!kernel_smem_ready(qsa_kernel, kSmemBytes, smem_set)) return PAGED_ATTN_ERR_CUDA;
  QsaLaunch a{};
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
  a.pairs = pairs;
  a.scale_log2 = p->sm_scale * 1.4426950408889634f;
  void* tok;
  timer_begin(st, &tok);
  // persistent: one CTA per SM walks the (token, KV-head pair) jobs
  const int sms = current_sm_count();
  if (sms <= 0) return PAGED_ATTN_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  qsa_kernel<<<grid, kThreads, kSmemBytes, st>>>(qmap, kmap, vmap, a);
  timer_end(st, tok);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

}  // namespace pa
