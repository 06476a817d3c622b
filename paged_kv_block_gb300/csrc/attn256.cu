// Dense packed-Q prefill (batch_prefill_with_paged_kv_cache, whose notes allow a head
// dimension of 256) on the 5th-generation tensor cores, for D = 256.
//
// Persistent: one CTA per SM walks the prefill planner's tile list (largest first) with a
// stride of the grid size.  A work tile is one Q sub-tile of 128 rows, a row being a
// (token, head-in-group) pair, so the G query heads that share a KV head share every K/V
// tile.  K and V are walked in 128-key tiles over the keys the tile's rows can see, so that
// the score MMA runs at N = 128 (an M = 128 MMA costs the same for any N up to 128).
// Roles (224 threads):
//   warps 0-3  softmax + epilogue (thread t <-> TMEM lane t <-> row t)
//   warp  4    TMA producer of Q (once per work tile) and K
//   warp  5    TMEM owner and MMA issuer (one thread)
//   warp  6    TMA producer of V
// Tensor memory (512 columns): S_0 [0,128) S_1 [128,256) O [256,512).  The scores of KV tile
// i (counted over the whole launch) land in S_(i%2); P is written over the first 64 columns
// of that buffer as packed bf16 and read from TMEM by the PV MMA.  The MMA issuer queues
// QK(i+2) behind PV(i), so the softmax of tile i+1 runs while PV(i) and QK(i+2) do.
// A whole 128-key K or V tile (64 KB) does not fit twice beside Q, so both stream through
// rings of 16 KB chunks: K in 64-column chunks (128 keys x 64 dims: the score MMA's k-steps
// over those dims need nothing else), V in 32-key chunks (32 keys x 256 dims: two k-steps of
// the PV MMA).  Each chunk is released as soon as its MMAs have read it.
// The online softmax runs in the log2 domain; the running maximum only moves (and O is
// rescaled in TMEM) when a tile's maximum exceeds it by more than 8.
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kD = 256;
constexpr int kKeys = 128;                     // keys per KV tile
constexpr int kChunks = kD / 64;               // 64-column (128-byte) chunks of a row
constexpr int kRows = 128;                     // rows of a Q sub-tile
constexpr int kQChunk = kRows * 128;           // 128 rows x 64 columns of bf16
constexpr int kQBytes = kChunks * kQChunk;     // 64 KB
// K ring slot: 128 keys x 64 columns (one 128-byte-swizzled block, 16 KB)
constexpr int kKSlotBytes = kKeys * 128;
// V ring slot: 32 keys x 256 columns as four 32 x 64 blocks (4 KB each), 16 KB
constexpr int kVKeys = 32;
constexpr int kVBlock = kVKeys * 128;
constexpr int kVSlotBytes = kChunks * kVBlock;
constexpr int kVChunks = kKeys / kVKeys;       // V chunks per KV tile
constexpr int kKSlots = 5;
constexpr int kVSlots = 5;
constexpr int kProdK = 4, kMmaWarp = 5, kProdV = 6;
constexpr int kThreads = 7 * 32;
constexpr int kTmemS = 0;                      // S_0, S_1: 128 columns each
constexpr int kTmemO = 256;                    // O: 256 columns
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr float kLn2 = 0.6931471805599453f;

struct Ctrl {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKSlots], k_empty[kKSlots];
  uint64_t v_full[kVSlots], v_empty[kVSlots];
  uint64_t p_full[2];
  uint64_t o_final, o_empty;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kSmemBytes = kQBytes + kKSlots * kKSlotBytes + kVSlots * kVSlotBytes +
                           static_cast<int>(sizeof(Ctrl)) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// One work tile as every role sees it.
struct Tile {
  int b, g, tok0, ntok, q_row0, L, nq;
  int kt0, N;          // 128-key tiles kt0 .. kt0 + N - 1
};

// The keys the tile's rows can see are [lo, hi): hi = min(L, p(last row) + 1) under the
// causal mask (L otherwise) and lo = max(0, p(first row) - window_left) with a window, where
// p(token i) = L - nq + i.  They are walked in 128-key tiles.
// L and nq are request b's KV length and query count.
__device__ __forceinline__ Tile tile_from_parts(const AttnLaunch& a, const TileRec& r, int L,
                                                int nq) {
  Tile t;
  t.b = r.b;
  t.g = r.g;
  t.tok0 = r.tok0;
  t.ntok = r.ntok;
  t.q_row0 = r.q_row0;
  t.L = L;
  t.nq = nq;
  const long long p0 = static_cast<long long>(t.L) - t.nq + r.tok0;
  const long long p1 = p0 + r.ntok - 1;
  const long long hi = a.causal ? min(static_cast<long long>(t.L), p1 + 1)
                                : static_cast<long long>(t.L);
  const long long lo = (a.causal && a.window_left >= 0) ? max(0LL, p0 - a.window_left) : 0LL;
  if (r.ntok <= 0 || r.kv_end <= r.kv_begin || hi <= lo) {
    t.kt0 = 0;
    t.N = 0;
  } else {
    t.kt0 = static_cast<int>(lo / kKeys);
    t.N = static_cast<int>((hi + kKeys - 1) / kKeys) - t.kt0;
  }
  return t;
}

__device__ __forceinline__ void request_lengths(const AttnLaunch& a, int b, int& L, int& nq) {
  L = __ldg(a.seq_lens + b);
  nq = a.qo_indptr ? __ldg(a.qo_indptr + b + 1) - __ldg(a.qo_indptr + b) : a.q_len;
}

__device__ __forceinline__ Tile make_tile(const AttnLaunch& a, const TileRec& r) {
  int L, nq;
  request_lengths(a, r.b, L, nq);
  return tile_from_parts(a, r, L, nq);
}

__global__ void __launch_bounds__(kThreads, 1)
attn256_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, AttnLaunch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* q_s = smem_align<1024>(smem_raw);
  uint8_t* k_s = q_s + kQBytes;
  uint8_t* v_s = k_s + kKSlots * kKSlotBytes;
  Ctrl* ctl = reinterpret_cast<Ctrl*>(v_s + kVSlots * kVSlotBytes);

  const int n_live = a.n_tiles ? *a.n_tiles : a.capacity;
  if (static_cast<int>(blockIdx.x) >= n_live) return;
  const int G = a.G;
  const int TM = kRows / G;                              // tokens per work tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) mbar_init(&ctl->p_full[w], 4);   // one arrival per softmax warp
    mbar_init(&ctl->o_final, 1);
    mbar_init(&ctl->o_empty, kRows);
    // a launch that an earlier CTA already broke does nothing
    ctl->abort_flag = launch_aborted(a.status) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;

  if (*abort_flag) {
    // nothing to do; fall through to the teardown
  } else if (warp == kProdK || warp == kProdV) {
    // =============================== producers =========================================
    // warp 4 copies Q (lane 0) and K, warp 6 copies V.  A piece is R keys of one page inside
    // a KV tile; its page id is loaded once per tile, while the tile before is copied.  A K
    // chunk is one 64-column block of the tile: every piece, lane p copying piece p.  A V
    // chunk is 32 keys of the tile in all four 64-column blocks: the pieces that fall in it,
    // lane 4 p + c copying column block c of piece p, so that the four copies of a piece
    // leave from four lanes at once.
    const bool is_k = warp == kProdK;
    if (lane == 0) {
      if (is_k) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
      } else {
        tma_prefetch_desc(&vmap);
      }
    }
    const int ps = a.page_size;
    const int R = is_k ? page_piece_rows(ps, kKeys) : page_piece_rows(ps, kVKeys);
    const int pieces = kKeys / R;                // per KV tile: K at most 16, V at most 8
    const int piece = is_k ? lane : lane >> 2;   // V: R >= 16 (page sizes 16 to 128)
    const int vblk = lane & 3;                   // V: the 64-column block this lane copies
    const int my_chunk = (piece * R) / kVKeys;   // V: the chunk this lane's piece falls in
    const int slots = is_k ? kKSlots : kVSlots;
    uint8_t* ring = is_k ? k_s : v_s;
    const int slot_bytes = is_k ? kKSlotBytes : kVSlotBytes;
    uint64_t* full = is_k ? ctl->k_full : ctl->v_full;
    uint64_t* empty = is_k ? ctl->k_empty : ctl->v_empty;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    const int head_off = is_k ? a.k_head_off : a.v_head_off;
    // chunks per KV tile: the four column blocks of K, or the four 32-key parts of V
    constexpr int kPerTile = kChunks;
    static_assert(kVChunks == kChunks, "four K chunks and four V chunks per KV tile");
    int ch = 0, qcount = 0;                      // chunks issued (over the launch), Q loads
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_live; idx += gridDim.x) {
      const Tile t = make_tile(a, a.tiles[idx]);
      if (t.N == 0) continue;
      const int* pt = a.pt_indptr ? a.pt + __ldg(a.pt_indptr + t.b)
                                  : a.pt + static_cast<long long>(t.b) * a.pt_stride;
      // first key of this lane's piece of KV tile n, or -1
      auto key_of = [&](int n) {
        const int key = (t.kt0 + n) * kKeys + piece * R;
        return (piece < pieces && key < t.L) ? key : -1;
      };
      int key = key_of(0);
      int page = key >= 0 ? __ldg(pt + key / ps) : 0;
      if (is_k) {
        if (qcount > 0 &&
            !mbar_wait_warp<true>(&ctl->q_empty, (qcount - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // box: 64 columns x G heads x TM tokens; rows past the tensor read as zero
          mbar_arrive_expect_tx(&ctl->q_full, static_cast<uint32_t>(kChunks * 128 * G * TM));
          for (int c = 0; c < kChunks; ++c)
            tma_load_3d(q_s + c * kQChunk, &qmap, &ctl->q_full, c * 64, t.g * G, t.q_row0);
        }
        ++qcount;
      }
      for (int n = 0; ok && n < t.N; ++n) {
        // the next KV tile's page id, loaded now: it is first used a whole tile later
        const int key_nx = n + 1 < t.N ? key_of(n + 1) : -1;
        const int page_nx = key_nx >= 0 ? __ldg(pt + key_nx / ps) : 0;
        bool live = key >= 0;
        if (live && (page < 0 || page >= a.num_pages)) {
          report_error(a.status, kErrMetadata);
          live = false;
        }
        const int row = page * a.page_rows + t.g * ps + (key >= 0 ? key % ps : 0) + head_off;
        for (int j = 0; j < kPerTile; ++j) {
          const int slot = ch % slots;
          if (ch >= slots &&
              !mbar_wait_warp<true>(&empty[slot], ((ch / slots) - 1) & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          const bool mine = live && (is_k || my_chunk == j);
          const uint32_t nlive = __popc(__ballot_sync(0xffffffffu, mine));
          if (lane == 0)
            mbar_arrive_expect_tx(&full[slot], nlive * R * 128u);   // one R-row box per lane
          __syncwarp();
          if (mine) {
            uint8_t* base = ring + slot * slot_bytes;
            if (is_k) {
              tma_load_2d(base + static_cast<uint32_t>(lane * R) * 128u, map, &full[slot], j * 64,
                          row);
            } else {
              uint8_t* dst = base + static_cast<uint32_t>(piece * R - j * kVKeys) * 128u;
              tma_load_2d(dst + vblk * kVBlock, map, &full[slot], vblk * 64, row);
            }
          }
          ++ch;
        }
        key = key_nx;
        page = page_nx;
      }
    }
    if (!ok && lane == 0) {                      // let copies in flight land before exiting
      for (int c = ch > slots ? ch - slots : 0; c < ch; ++c)
        drain_wait(&full[c % slots], (c / slots) & 1);
      if (is_k && qcount > 0) drain_wait(&ctl->q_full, (qcount - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // =============================== MMA issuer ========================================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kRows, kKeys, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kRows, kD, false, true);
      // Descriptors of the first k-step; later steps add the byte offset / 16 to the start
      // address field, which never carries out of it inside shared memory.
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(q_s), 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(smem_u32(k_s), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(v_s), kVBlock, 1024);
      auto wait = [&](uint64_t* bar, int parity) {
        return mbar_wait_fast(bar, parity, a.status, abort_flag);
      };
      int kc = 0, vc = 0;                        // K and V chunks consumed over the launch
      // S_(it%2) = Q K(it)^T: per 64-column K chunk, the 4 k-steps of 16 columns it holds
      auto issue_qk = [&](int it) -> bool {
        for (int c = 0; c < kChunks; ++c, ++kc) {
          const int slot = kc % kKSlots;
          if (!wait(&ctl->k_full[slot], (kc / kKSlots) & 1)) return false;
          tc_fence_after();
          const uint64_t kd = k_desc0 + static_cast<uint64_t>((slot * kKSlotBytes) >> 4);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            mma_ss(tmem + kTmemS + (it & 1) * kKeys,
                   q_desc0 + static_cast<uint64_t>((c * kQChunk + k4 * 32) >> 4),
                   kd + static_cast<uint64_t>((k4 * 32) >> 4), idesc_qk, c > 0 || k4 > 0);
          mma_commit(&ctl->k_empty[slot]);     // the last one also tells the softmax S is ready
        }
        return true;
      };
      // O += P(it) V(it): per 32-key V chunk, its 2 k-steps of 16 keys
      auto issue_pv = [&](int it, bool acc) -> bool {
        for (int j = 0; j < kVChunks; ++j, ++vc) {
          const int slot = vc % kVSlots;
          if (!wait(&ctl->v_full[slot], (vc / kVSlots) & 1)) return false;
          tc_fence_after();
          const uint64_t vd = v_desc0 + static_cast<uint64_t>((slot * kVSlotBytes) >> 4);
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int ks = 2 * j + k2;
            mma_ts(tmem + kTmemO, tmem + kTmemS + (it & 1) * kKeys + ks * 8,
                   vd + static_cast<uint64_t>((k2 * 16 * 128) >> 4), idesc_pv, acc || ks > 0);
          }
          mma_commit(&ctl->v_empty[slot]);     // the last one also tells the softmax PV is done
        }
        return true;
      };
      int kv_it = 0, qcount = 0, ep = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_live; idx += gridDim.x) {
        const Tile t = make_tile(a, a.tiles[idx]);
        const int N = t.N;
        if (N == 0) continue;
        const int it0 = kv_it;
        if (!wait(&ctl->q_full, qcount & 1)) {
          ok = false;
          break;
        }
        ++qcount;
        for (int n = 0; ok && n < 2 && n < N; ++n) {   // the first two score tiles
          ok = issue_qk(it0 + n);
          if (ok && n == N - 1) mma_commit(&ctl->q_empty);
        }
        for (int n = 0; ok && n < N; ++n) {
          const int it = it0 + n;
          // O is free once the previous work tile's epilogue has read it
          if (!wait(&ctl->p_full[it & 1], (it >> 1) & 1) ||
              (n == 0 && ep > 0 && !wait(&ctl->o_empty, (ep - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!issue_pv(it, n > 0)) {
            ok = false;
            break;
          }
          if (n == N - 1) mma_commit(&ctl->o_final);
          if (n + 2 < N) {                       // QK(it + 2) into the buffer P(it) came from
            if (!issue_qk(it + 2)) {
              ok = false;
              break;
            }
            if (n + 2 == N - 1) mma_commit(&ctl->q_empty);
          }
        }
        kv_it += N;
        ++ep;
      }
    }
  } else if (warp < 4) {
    // =============================== softmax (one row per thread) =======================
    const int m = threadIdx.x;                           // row of the work tile
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t o_col = tmem + lane_base + kTmemO;
    const float sl2 = a.scale_log2;
    const bool causal = a.causal != 0;
    const int wl = a.window_left;
    int kv_it = 0, ep = 0;
    bool ok = true;
    // S(it) lands in buffer it % 2, whose next scores (QK(it + 2)) wait for this softmax's P.
    // PV(j) is complete once it has released V chunk 4 j + 3 (the commit covers every earlier
    // MMA).  The softmax of tile it asks for PV(it - 1) after it has seen S(it); the parity
    // wait is sound there because that slot's previous chunk belongs to PV(it - 2), complete
    // before S(it) (QK(it) was issued after it), and its next one to PV(it) or later, which
    // waits for this softmax's P.
    // S(it) is complete once QK(it) has released K chunk 4 it + 3.  That barrier's previous
    // commit came from QK(it - 1), complete before this softmax saw S(it - 1), and its next
    // from QK(it + 2), which is issued after PV(it) and so after this softmax's P: the parity
    // wait cannot alias (it could with four K slots, where the next commit is QK(it + 1)'s).
    static_assert(kKSlots >= kChunks + 1, "S readiness rides on the K-slot release");
    auto s_ready = [&](int it) {
      const int c = kChunks * it + kChunks - 1;
      return mbar_wait_fast_warp(&ctl->k_empty[c % kKSlots], (c / kKSlots) & 1, a.status,
                                 abort_flag);
    };
    auto pv_done = [&](int it) {
      const int c = kVChunks * it + kVChunks - 1;
      return mbar_wait_warp<true>(&ctl->v_empty[c % kVSlots], (c / kVSlots) & 1, a.status,
                                  abort_flag);
    };
    static_assert(kKSlots >= kChunks && kVSlots >= kVChunks, "ring slots per KV tile");
    // The next work tile's record is read after the current tile's last softmax and its KV
    // length and query count after the wait for O, so a work tile starts without a global
    // round trip.
    TileRec rec_nx = a.tiles[blockIdx.x];
    int L_nx, nq_nx;
    request_lengths(a, rec_nx.b, L_nx, nq_nx);
    for (int idx = blockIdx.x; ok && idx < n_live; idx += gridDim.x) {
      const Tile t = tile_from_parts(a, rec_nx, L_nx, nq_nx);
      const int idx_nx = idx + static_cast<int>(gridDim.x);
      const bool has_nx = idx_nx < n_live;
      const int tok = m / G;                             // token inside the work tile
      const bool row_valid = m < G * TM && tok < t.ntok;
      const int pos = t.L - t.nq + t.tok0 + tok;        // query position
      // keys [klo, khi) of this row
      const int khi = causal ? min(t.L, pos + 1) : t.L;
      const int klo = (causal && wl >= 0) ? max(0, pos - wl) : 0;
      const int kspan = max(khi - klo, 0);
      float m_run = -INFINITY, l_run = 0.f;
      for (int n = 0; n < t.N; ++n) {
        const int it = kv_it + n;
        if (!s_ready(it)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = tmem + lane_base + kTmemS + (it & 1) * kKeys;
        uint32_t r[kKeys];
#pragma unroll
        for (int q = 0; q < kKeys / 32; ++q)
          tmem_ld32(s_col + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[q * 32]));
        tmem_ld_wait();
        const int key0 = (t.kt0 + n) * kKeys;
        if (key0 < klo || key0 + kKeys > khi) {
          // one unsigned range test and a select per column (the limits differ per row)
          const int lo_c = klo - key0;
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const bool out = static_cast<unsigned>(c - lo_c) >= static_cast<unsigned>(kspan);
            r[c] = out ? 0xff800000u : r[c];
          }
        }
        // row maximum: 8 independent chains of 3-input max, then a short tree
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; c += 2)
          mx[(c >> 1) & 7] = max3f(mx[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
        // scores are scaled by sl2 > 0 after the maximum, which commutes with it
        const float mt = fmaxf(max3f(mx[0], mx[1], mx[2]),
                               max3f(mx[3], mx[4], fmaxf(mx[5], fmaxf(mx[6], mx[7])))) * sl2;
        // ---- online softmax with a lazily moved maximum ----------------------------------
        float alpha = 1.f;
        if (mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY)) {
          alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mt);
          m_run = mt;
        }
        const float nmu = m_run == -INFINITY ? 0.f : -m_run;
        // ---- P = exp2(s * sl2 - mu) and the row sum; bf16 pairs packed in place into r[j] ---
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
        for (int j = 0; j < kKeys / 2; ++j) {
          float x0, x1;
          ffma2_bcast(x0, x1, __uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]), sl2, nmu);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          if (j & 1) fadd2(sb0, sb1, p0, p1);
          else fadd2(sa0, sa1, p0, p1);
          r[j] = pack_bf16(p0, p1);
        }
        tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        l_run = l_run * alpha + ((sa0 + sa1) + (sb0 + sb1));
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds PV of the previous KV tile, which may still run: wait for it, then scale
          if (!pv_done(it - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < kD / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(o_col + q * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(o_col + q * 32, ov);
          }
        }
        tmem_st_wait();
        if (key0 + kKeys > t.L && warp == 0) {
          // Rows of keys past the length hold stale or non-finite data (tail slots of the
          // last page, or nothing copied); P is 0 there, so make V exactly 0 as well.  V chunk
          // j of KV tile it is chunk 4 it + j of the launch; lane m clears its key row.
          // The chunk's ring slot last held a chunk of KV tile it - 1, whose copy may not have
          // landed yet, and a parity wait for the phase after the barrier's current one
          // returns at once.  PV(it - 1) waited for every chunk of tile it - 1, so wait for it
          // first.
          if (it > 0 && !pv_done(it - 1)) {
            ok = false;
            break;
          }
          for (int j = 0; j < kVChunks; ++j) {
            if (key0 + (j + 1) * kVKeys <= t.L) continue;
            const int vc = kVChunks * it + j;
            const int slot = vc % kVSlots;
            if (!mbar_wait_warp<true>(&ctl->v_full[slot], (vc / kVSlots) & 1, a.status,
                                      abort_flag)) {
              ok = false;
              break;
            }
            if (key0 + j * kVKeys + m >= t.L) {
              uint8_t* vt = v_s + slot * kVSlotBytes + m * 128;
              const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
              for (int c = 0; c < kChunks; ++c)
#pragma unroll
                for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(vt + c * kVBlock + i * 16) = z;
            }
          }
          fence_proxy_async_smem();
          if (!ok) break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[it & 1]);
      }
      if (!ok) break;
      if (has_nx) rec_nx = a.tiles[idx_nx];
      // ---- epilogue --------------------------------------------------------------------
      bool have_o = false;
      if (t.N > 0) {
        have_o = mbar_wait_warp<true>(&ctl->o_final, ep & 1, a.status, abort_flag);
        ++ep;
        if (!have_o) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (has_nx) request_lengths(a, rec_nx.b, L_nx, nq_nx);
      const long long orow = static_cast<long long>(t.q_row0 + tok) * a.Hq + t.g * G + (m % G);
      const float inv = l_run > 0.f ? a.out_scale / l_run : 0.f;
      // one row per thread in two 128-column halves (four loads in flight each), 32 bytes per
      // store where the output allows it (rows are 512 or 1024 bytes: the base decides)
      const bool wide = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t ov[128];
        if (have_o) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tmem_ld32(o_col + h * 128 + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[q * 32]));
          tmem_ld_wait();
          if (h == 1) {                          // O fully read: the next work tile may write
            tc_fence_before();
            mbar_arrive(&ctl->o_empty);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i) ov[i] = 0u;
        }
        if (row_valid && a.out_dtype == kOutF32) {
          float* dst = static_cast<float*>(a.out) + orow * kD + h * 128;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint32_t v8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v8[e] = __float_as_uint(__uint_as_float(ov[8 * i + e]) * inv);
            if (wide) {
              st_global_v8(dst + 8 * i, v8);
            } else {
              reinterpret_cast<uint4*>(dst + 8 * i)[0] = make_uint4(v8[0], v8[1], v8[2], v8[3]);
              reinterpret_cast<uint4*>(dst + 8 * i)[1] = make_uint4(v8[4], v8[5], v8[6], v8[7]);
            }
          }
        } else if (row_valid) {
          uint16_t* dst = static_cast<uint16_t*>(a.out) + orow * kD + h * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t v8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v8[e] = pack_out2(__uint_as_float(ov[16 * i + 2 * e]) * inv,
                                __uint_as_float(ov[16 * i + 2 * e + 1]) * inv, a.out_dtype);
            if (wide) {
              st_global_v8(dst + 16 * i, v8);
            } else {
              reinterpret_cast<uint4*>(dst + 16 * i)[0] = make_uint4(v8[0], v8[1], v8[2], v8[3]);
              reinterpret_cast<uint4*>(dst + 16 * i)[1] = make_uint4(v8[4], v8[5], v8[6], v8[7]);
            }
          }
        }
      }
      if (row_valid && a.lse)
        a.lse[orow] = l_run > 0.f ? (m_run + fast_log2(l_run)) * kLn2 : -INFINITY;
      kv_it += t.N;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Prefill tiles of D = 256 (one 128-row sub-tile each; the planner's tile_tokens is 128 / G).
int launch_attn256(const AttnLaunch& a, cudaStream_t st) {
  if (a.D != kD || a.G < 1 || a.G > kRows) return -2;
  static std::atomic<uint64_t> smem_set{0};
  if (!kernel_smem_ready(attn256_kernel, kSmemBytes, smem_set)) return -1;
  const int sms = current_sm_count();
  if (sms <= 0) return -1;
  if (a.capacity <= 0) return 0;
  const int grid = a.capacity < sms ? a.capacity : sms;
  attn256_kernel<<<grid, kThreads, kSmemBytes, st>>>(a.qmap, a.kmap, a.vmap, a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace pa
