// Paged prefill / block-sparse attention forward on the 5th-generation tensor cores.
//
// Serves the block-sparse form of block_sparse_attention_with_paged_kv_cache (KV blocks
// listed per (request, KV head, query block) in BSR form) and the dense packed-Q form of
// batch_prefill_with_paged_kv_cache (every KV tile that meets the causal / window span).
//
// One CTA owns one planner tile: up to two Q sub-tiles of 128 rows, a row being a (token,
// head-in-group) pair, so the G query heads that share a KV head share every K/V tile.
// Roles (320 threads):
//   warps 0-3  softmax of sub-tile 0 (thread t <-> TMEM lane t <-> row t)
//   warps 4-7  softmax of sub-tile 1
//   warp  8    TMA producer: Q once, then K and V of each 128-key tile, one box per page
//              piece (a page, or the part of a page inside a selected block) and 64-column
//              half, into a 2-stage ring
//   warp  9    TMEM owner and MMA issuer (one thread): S_w = Q_w K^T and O_w += P_w V
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P_w is
// written as packed bf16 over the first 64 columns of S_w and read from TMEM by the PV MMA.
// The online softmax runs in the log2 domain with exp2; the running maximum is only moved
// (and O rescaled) when a tile's maximum exceeds it by more than 8, which leaves the
// normalised result unchanged.
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 320;
constexpr int kQHalf = 128 * 128;              // bytes of a 128-row x 64-col bf16 half
constexpr int kQBytes = 2 * kQHalf;            // one Q sub-tile
constexpr int kKvHalf = kKvTile * 128;         // 128 keys x 64 cols
constexpr int kKvBytes = 2 * kKvHalf;          // one K (or V) tile
constexpr int kStages = 2;
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr float kLn2 = 0.6931471805599453f;

struct Ctrl {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_final[2];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kSmemBytes = 2 * kQBytes + kStages * 2 * kKvBytes + 1024 + 256;

// Geometry of the KV tile sequence of one CTA.
template <int CK>
struct KvWalk {
  int dense;            // 1: tile n covers keys [(kv_begin + n) * 128, +128)
  int kv_begin, kv_end;
  const int* blocks;    // BSR: block ids of the row
  int kvbs, spb;        // keys per block, sub-chunks per block
  int total_sub;        // BSR: sub-chunks in the row
  __device__ int num_tiles() const {
    if (dense) return kv_end - kv_begin;
    return (total_sub + (kKvTile / CK) - 1) / (kKvTile / CK);
  }
  // First key of sub-chunk c of tile n, or -1 when the slot is empty.
  __device__ int key0(int n, int c) const {
    if (dense) return (kv_begin + n) * kKvTile + c * CK;
    const int s = n * (kKvTile / CK) + c;
    if (s >= total_sub) return -1;
    const int blk = __ldg(blocks + s / spb);
    return blk * kvbs + (s % spb) * CK;
  }
};

template <int CK>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, AttnLaunch a) {
  constexpr int NSUB = kKvTile / CK;   // sub-chunks per KV tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = base;                                   // 2 sub-tiles
  uint8_t* kv_s = base + 2 * kQBytes;                    // stages: K then V
  Ctrl* ctl = reinterpret_cast<Ctrl*>(kv_s + kStages * 2 * kKvBytes);

  const int n_live = a.n_tiles ? *a.n_tiles : a.capacity;
  if (static_cast<int>(blockIdx.x) >= n_live || launch_aborted(a.status)) return;
  const TileRec tile = a.tiles[blockIdx.x];
  const int G = a.G;
  const int TM = kMTileRows / G;                         // tokens per sub-tile
  const int ntok0 = min(tile.ntok, TM);
  const int ntok1 = tile.ntok - ntok0;
  const int n_sub_tiles = ntok1 > 0 ? 2 : 1;
  const int L = __ldg(a.seq_lens + tile.b);
  const int nq = a.qo_indptr ? (__ldg(a.qo_indptr + tile.b + 1) - __ldg(a.qo_indptr + tile.b))
                             : a.q_len;

  KvWalk<CK> walk;
  walk.dense = !a.block_sparse;
  walk.kv_begin = tile.kv_begin;
  walk.kv_end = tile.kv_end;
  walk.blocks = a.block_sparse ? a.block_indices + tile.kv_begin : nullptr;
  walk.kvbs = a.kv_block_size;
  walk.spb = a.kv_block_size / CK;
  walk.total_sub = walk.dense ? 0 : (tile.kv_end - tile.kv_begin) * walk.spb;
  const int N = walk.num_tiles();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&ctl->s_full[w], 1);
      mbar_init(&ctl->p_full[w], 128);
      mbar_init(&ctl->o_final[w], 1);
    }
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp == 8) {
    // =============================== producer ==========================================
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      const uint32_t qbox = 128u * G * TM;
      mbar_arrive_expect_tx(&ctl->q_full, qbox * 2 * n_sub_tiles);
      for (int w = 0; w < n_sub_tiles; ++w)
        for (int h = 0; h < 2; ++h)
          tma_load_3d(q_s + w * kQBytes + h * kQHalf, &qmap, &ctl->q_full, h * 64, tile.g * G,
                      tile.q_row0 + w * TM);
      const int ps = a.page_size;
      const int R = CK < ps ? CK : ps;                  // rows per box
      const int* pt = a.pt_indptr ? a.pt + __ldg(a.pt_indptr + tile.b)
                                  : a.pt + static_cast<long long>(tile.b) * a.pt_stride;
      const int max_page_idx = (L + ps - 1) / ps;
      for (int n = 0; n < N; ++n) {
        const int st = n % kStages;
        if (n >= kStages &&
            !mbar_wait(&ctl->kv_empty[st], ((n / kStages) - 1) & 1, a.status, abort_flag))
          break;
        uint8_t* kt = kv_s + st * 2 * kKvBytes;
        uint8_t* vt = kt + kKvBytes;
        int rows[kKvTile / 8];
        uint32_t live = 0;
        int npieces = 0;
#pragma unroll 1
        for (int c = 0; c < NSUB; ++c) {
          const int k0 = walk.key0(n, c);
#pragma unroll 1
          for (int p = 0; p < CK / R; ++p) {
            const int idx = npieces++;
            const int key = k0 + p * R;
            if (k0 < 0 || key >= L) continue;
            const int pidx = key / ps;
            if (pidx >= max_page_idx) continue;
            const int page = __ldg(pt + pidx);
            if (page < 0 || page >= a.num_pages) {
              report_error(a.status, kErrMetadata);
              continue;
            }
            rows[idx] = page * a.page_rows + tile.g * ps + key % ps;
            live |= 1u << idx;
          }
        }
        const uint32_t bytes = static_cast<uint32_t>(__popc(live)) * R * 128u * 2u;
        mbar_arrive_expect_tx(&ctl->k_full[st], bytes);
        for (int i = 0; i < npieces; ++i) {
          if (!((live >> i) & 1u)) continue;
          const uint32_t off = static_cast<uint32_t>(i * R) * 128u;
          tma_load_2d(kt + off, &kmap, &ctl->k_full[st], 0, rows[i] + a.k_head_off);
          tma_load_2d(kt + kKvHalf + off, &kmap, &ctl->k_full[st], 64, rows[i] + a.k_head_off);
        }
        mbar_arrive_expect_tx(&ctl->v_full[st], bytes);
        for (int i = 0; i < npieces; ++i) {
          if (!((live >> i) & 1u)) continue;
          const uint32_t off = static_cast<uint32_t>(i * R) * 128u;
          tma_load_2d(vt + off, &vmap, &ctl->v_full[st], 0, rows[i] + a.v_head_off);
          tma_load_2d(vt + kKvHalf + off, &vmap, &ctl->v_full[st], 64, rows[i] + a.v_head_off);
        }
      }
    }
  } else if (warp == 9) {
    // =============================== MMA issuer ========================================
    if (lane == 0 && N > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, kKvTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, kD, false, true);
      const uint32_t q_addr = smem_u32(q_s);
      const uint32_t kv_addr = smem_u32(kv_s);
      auto issue_qk = [&](int w, int n) {
        const uint32_t qa = q_addr + w * kQBytes;
        const uint32_t ka = kv_addr + (n % kStages) * 2 * kKvBytes;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kQHalf + (ks & 3) * 32;
          const uint32_t koff = (ks >> 2) * kKvHalf + (ks & 3) * 32;
          mma_ss(tmem + w * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + koff, 16, 1024),
                 idesc_qk, ks > 0);
        }
        mma_commit(&ctl->s_full[w]);
      };
      auto issue_pv = [&](int w, int n) {
        const uint32_t va = kv_addr + (n % kStages) * 2 * kKvBytes + kKvBytes;
#pragma unroll
        for (int ks = 0; ks < kKvTile / 16; ++ks) {
          mma_ts(tmem + 256 + w * 128, tmem + w * 128 + ks * 8,
                 sdesc_sw128(va + ks * 16 * 128, kKvHalf, 1024), idesc_pv, (n > 0 || ks > 0));
        }
        if (n == N - 1) mma_commit(&ctl->o_final[w]);
      };
      bool ok = mbar_wait(&ctl->q_full, 0, a.status, abort_flag);
      ok = ok && mbar_wait(&ctl->k_full[0], 0, a.status, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        if (n_sub_tiles > 1) issue_qk(1, 0);
      }
      for (int n = 0; ok && n < N; ++n) {
        const int st = n % kStages;
        if (!mbar_wait(&ctl->v_full[st], (n / kStages) & 1, a.status, abort_flag)) break;
        if (!mbar_wait(&ctl->p_full[0], n & 1, a.status, abort_flag)) break;
        tc_fence_after();
        issue_pv(0, n);
        const bool more = n + 1 < N;
        if (more) {
          if (!mbar_wait(&ctl->k_full[(n + 1) % kStages], ((n + 1) / kStages) & 1, a.status,
                         abort_flag))
            break;
          tc_fence_after();
          issue_qk(0, n + 1);
        }
        if (n_sub_tiles > 1) {
          if (!mbar_wait(&ctl->p_full[1], n & 1, a.status, abort_flag)) break;
          tc_fence_after();
          issue_pv(1, n);
        }
        mma_commit(&ctl->kv_empty[st]);
        if (more && n_sub_tiles > 1) issue_qk(1, n + 1);
      }
    }
  } else {
    // =============================== softmax (one row per thread) =======================
    const int w = warp >> 2;                       // sub-tile
    const int m = threadIdx.x & 127;               // row inside the sub-tile
    const int ntok_w = w == 0 ? ntok0 : ntok1;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + w * 128;
    const uint32_t o_col = tmem + lane_base + 256 + w * 128;
    const int tok = tile.tok0 + w * TM + m / G;    // token index inside the request
    const bool row_valid = (m < G * TM) && (m / G < ntok_w);
    const int pos = L - nq + tok;                  // query position
    const float sl2 = a.scale_log2;
    const bool causal = a.causal != 0;
    const int wl = a.window_left;
    float m_run = -INFINITY, l_run = 0.f;
    if (w < n_sub_tiles) {
      for (int n = 0; n < N; ++n) {
        if (!mbar_wait_warp(&ctl->s_full[w], n & 1, a.status, abort_flag)) break;
        tc_fence_after();
        // ---- per-tile column facts, identical for every row ----------------------------
        int k0[NSUB];
        uint32_t colmask[4];
        bool zero_v = false;
        int kmin = 0x7fffffff, kmax = -1;
#pragma unroll
        for (int c = 0; c < NSUB; ++c) {
          k0[c] = walk.key0(n, c);
          if (k0[c] < 0 || k0[c] + CK > L) zero_v = true;
          if (k0[c] >= 0) {
            kmin = min(kmin, k0[c]);
            kmax = max(kmax, k0[c] + CK - 1);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) colmask[i] = 0u;
#pragma unroll
        for (int c = 0; c < NSUB; ++c) {
          // bits of the CK columns of sub-chunk c (CK = 8, 16, 32, 64 or 128)
#pragma unroll
          for (int part = 0; part < (CK + 31) / 32; ++part) {
            const int col0 = c * CK + part * 32;          // first column of this 32-span
            const int span = CK < 32 ? CK : 32;
            uint32_t bits = 0u;
            if (k0[c] >= 0) {
              const int key = k0[c] + part * 32;
              const int live = L - key;                    // keys < L in this span
              bits = live >= span ? (span == 32 ? 0xffffffffu : ((1u << span) - 1u))
                                  : (live > 0 ? ((1u << live) - 1u) : 0u);
              if (a.valid_bits) {
                const int wi = key >> 5;
                const uint32_t word =
                    wi < a.valid_words
                        ? __ldg(a.valid_bits + static_cast<long long>(tile.b) * a.valid_words + wi)
                        : 0u;
                bits &= (word >> (key & 31));
              }
            }
            colmask[col0 >> 5] |= bits << (col0 & 31);
          }
        }
        // ---- S row -----------------------------------------------------------------------
        uint32_t sraw[kKvTile];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32(s_col + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&sraw[q * 32]));
        tmem_ld_wait();
        float x[kKvTile];
#pragma unroll
        for (int c = 0; c < kKvTile; ++c) x[c] = __uint_as_float(sraw[c]);
        const bool full = !a.valid_bits && !zero_v &&
                          (!causal || kmax <= pos) && (wl < 0 || kmin >= pos - wl);
        float mt = -INFINITY;
        if (full) {
#pragma unroll
          for (int c = 0; c < kKvTile; ++c) {
            x[c] *= sl2;
            mt = fmaxf(mt, x[c]);
          }
        } else {
          int hi_lim[NSUB], lo_lim[NSUB];
#pragma unroll
          for (int c = 0; c < NSUB; ++c) {
            hi_lim[c] = causal ? pos - k0[c] : 0x7fffffff;
            lo_lim[c] = wl >= 0 ? pos - wl - k0[c] : -0x7fffffff;
          }
#pragma unroll
          for (int c = 0; c < kKvTile; ++c) {
            const int sc = c / CK, r = c % CK;
            const bool vis = ((colmask[c >> 5] >> (c & 31)) & 1u) && r <= hi_lim[sc] &&
                             r >= lo_lim[sc];
            x[c] = vis ? x[c] * sl2 : -INFINITY;
            mt = fmaxf(mt, x[c]);
          }
        }
        // ---- online softmax with a lazily moved maximum ----------------------------------
        float alpha = 1.f;
        if (mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY)) {
          alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mt);
          m_run = mt;
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        float rs = 0.f;
        uint32_t pk[kKvTile / 2];
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2) {
          const float p0 = fast_exp2(x[c] - mu);
          const float p1 = fast_exp2(x[c + 1] - mu);
          rs += p0 + p1;
          pk[c >> 1] = pack_bf16(p0, p1);
        }
        l_run = l_run * alpha + rs;
        // O was last written by PV of tile n-1, which completed before S of tile n
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t ov[32];
            tmem_ld32(o_col + q * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(o_col + q * 32, ov);
          }
        }
        tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        tmem_st_wait();
        if (zero_v && w == 0) {
          // Rows of keys that are not live (past the length, or empty slots) may hold
          // stale or non-finite data; P is 0 there, so make V exactly 0 as well.
          const int st = n % kStages;
          if (mbar_wait_warp(&ctl->v_full[st], (n / kStages) & 1, a.status, abort_flag)) {
            const int c = m;                         // this thread clears key slot m
            const int k = k0[c / CK];
            if (k < 0 || k + (c % CK) >= L) {
              uint8_t* vt = kv_s + st * 2 * kKvBytes + kKvBytes;
              uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                *reinterpret_cast<uint4*>(vt + c * 128 + i * 16) = z;
                *reinterpret_cast<uint4*>(vt + kKvHalf + c * 128 + i * 16) = z;
              }
            }
            fence_proxy_async_smem();
          }
        }
        tc_fence_before();
        mbar_arrive(&ctl->p_full[w]);
      }
      // ---- epilogue ------------------------------------------------------------------------
      const bool have_o = N > 0 && mbar_wait_warp(&ctl->o_final[w], 0, a.status, abort_flag);
      if (have_o) tc_fence_after();
      const int head = tile.g * G + (m % G);
      const long long orow = static_cast<long long>(tile.q_row0 + w * TM + m / G) * a.Hq + head;
      const float inv = l_run > 0.f ? a.out_scale / l_run : 0.f;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t ov[32];
        if (have_o) {
          tmem_ld32(o_col + q * 32, ov);
          tmem_ld_wait();
        }
        if (row_valid) {
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[i] = have_o ? pack_bf16(__uint_as_float(ov[2 * i]) * inv,
                                        __uint_as_float(ov[2 * i + 1]) * inv)
                            : 0u;
          uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kD + q * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
        }
      }
      if (row_valid && a.lse)
        a.lse[orow] = l_run > 0.f ? (m_run + fast_log2(l_run)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int CK>
int launch_ck(const AttnLaunch& a, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_tc_kernel<CK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  attn_tc_kernel<CK><<<a.capacity, kThreads, kSmemBytes, st>>>(a.qmap, a.kmap, a.vmap, a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_attn(const AttnLaunch& a, cudaStream_t st) {
  if (a.capacity <= 0) return 0;
  switch (attn_sub_chunk(a.kv_block_size, a.block_sparse != 0)) {
    case 8: return launch_ck<8>(a, st);
    case 16: return launch_ck<16>(a, st);
    case 32: return launch_ck<32>(a, st);
    case 64: return launch_ck<64>(a, st);
    case 128: return launch_ck<128>(a, st);
    default: return -2;
  }
}

}  // namespace pa
