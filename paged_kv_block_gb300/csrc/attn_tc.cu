// Paged prefill / block-sparse attention forward on the 5th-generation tensor cores.
//
// Serves the block-sparse form of block_sparse_attention_with_paged_kv_cache (KV blocks
// listed per (request, KV head, query block) in BSR form) and the dense packed-Q form of
// batch_prefill_with_paged_kv_cache (every KV tile that meets the causal / window span).
//
// Persistent: one CTA per SM walks the planner's tile list (sorted by cost, largest first).
// CTA c starts with tile c; after that the CTAs claim tiles from a counter in the status area
// (so each takes the largest tile left whenever it needs one: a static stride left the
// slowest CTA ~7% behind the mean on dense prefill).  The claims reach the other roles
// through a small ring in shared memory; the K producer makes them (two tiles ahead) in
// block-sparse launches, warp 11 (otherwise idle) in dense ones.
// A tile holds up to two Q sub-tiles of 128 rows, a row being a (token, head-in-group) pair,
// so the G query heads that share a KV head share every K/V tile.  Roles (384 threads):
//   warps 0-3  softmax + epilogue of sub-tile 0 (thread t <-> TMEM lane t <-> row t)
//   warps 4-7  softmax + epilogue of sub-tile 1
//   warp  8    TMA producer of Q (once per tile) and K (2-stage ring)
//   warp  9    TMEM owner and MMA issuer (one thread): S_w = Q_w K^T and O_w += P_w V
//   warp 10    TMA producer of V (3-stage ring: a V stage is free only after PV of both
//              sub-tiles, later than a K stage after QK, so V gets the deeper ring)
//   warp 11    block-sparse: column facts of each KV tile (first key of each sub-chunk,
//              live-key mask, key range), a few tiles ahead into a small ring, so that the
//              softmax reads them from shared memory instead of issuing block-id and
//              valid-bit loads; dense: work-tile claims
// K and V of a 128-key tile are gathered one TMA box per page piece (a page, or the part of
// a page inside a selected block) and 64-column half.
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
constexpr int kThreads = 384;
constexpr int kQHalf = 128 * 128;              // bytes of a 128-row x 64-col bf16 half
constexpr int kQBytes = 2 * kQHalf;            // one Q sub-tile
constexpr int kKvHalf = kKvTile * 128;         // 128 keys x 64 cols
constexpr int kKvBytes = 2 * kKvHalf;          // one K (or V) tile
constexpr int kKStages = 2;
constexpr int kVStages = 3;
// Register split after set-up (launch: 384 threads x 168): the producer / MMA warpgroup
// gives registers to the two softmax warpgroups; 2 x 128 x 200 + 128 x 104 = 384 x 168.
constexpr int kSoftmaxRegs = 200;
constexpr int kControlRegs = 104;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split");
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kFacts = 4;                      // column-facts ring entries
constexpr int kTileRing = 4;                   // claimed work tiles handed to the roles

// Facts of one KV tile that are the same for every row.
struct TileFacts {
  int k0[kKvTile / 8];     // first key of each sub-chunk (-1: empty slot)
  uint32_t colmask[4];     // live keys: slot used, key < length, valid bit set
  int kmin, kmax;          // key range of the used sub-chunks
  int zero_v;              // some key slot is not live (V rows to zero)
  int pad;
  float cs[kKvTile / 8];   // scaled form: key scale of each sub-chunk's block
};

struct Ctrl {
  TileFacts facts[kFacts];
  uint64_t facts_full[kFacts], facts_empty[kFacts];
  uint64_t q_full, q_empty;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2], o_final[2], o_empty[2];
  uint64_t t_full[kTileRing], t_empty[kTileRing];
  int tidx[kTileRing];      // tile of claim sequence s in slot s % kTileRing
  uint32_t tmem_base;
  int abort_flag;
  int skip;                 // this CTA has no work tile (or the launch was aborted)
};

constexpr int kSmemBytes =
    2 * kQBytes + (kKStages + kVStages) * kKvBytes + static_cast<int>(sizeof(Ctrl)) + 1024;

// Geometry of the KV tile sequence of one planner tile.
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
struct TileInfo {
  TileRec rec;
  int ntok0, ntok1, nsub, L, nq, N;
  KvWalk<CK> walk;
};

// KV length and query count of request b (the two global reads a work tile needs beyond its
// record).
__device__ __forceinline__ void request_lengths(const AttnLaunch& a, int b, int& L, int& nq) {
  L = __ldg(a.seq_lens + b);
  nq = a.qo_indptr ? (__ldg(a.qo_indptr + b + 1) - __ldg(a.qo_indptr + b)) : a.q_len;
}

template <int CK>
__device__ __forceinline__ TileInfo<CK> tile_from_parts(const AttnLaunch& a, const TileRec& rec,
                                                        int L, int nq) {
  TileInfo<CK> t;
  t.rec = rec;
  const int TM = kMTileRows / a.G;
  t.ntok0 = min(t.rec.ntok, TM);
  t.ntok1 = t.rec.ntok - t.ntok0;
  t.nsub = t.ntok1 > 0 ? 2 : 1;
  t.L = L;
  t.nq = nq;
  t.walk.dense = !a.block_sparse;
  t.walk.kv_begin = t.rec.kv_begin;
  t.walk.kv_end = t.rec.kv_end;
  t.walk.blocks = a.block_sparse ? a.block_indices + t.rec.kv_begin : nullptr;
  t.walk.kvbs = a.kv_block_size;
  t.walk.spb = a.kv_block_size / CK;
  t.walk.total_sub = t.walk.dense ? 0 : (t.rec.kv_end - t.rec.kv_begin) * t.walk.spb;
  t.N = t.walk.num_tiles();
  return t;
}

template <int CK>
__device__ __forceinline__ TileInfo<CK> tile_from_rec(const AttnLaunch& a, const TileRec& rec) {
  int L, nq;
  request_lengths(a, rec.b, L, nq);
  return tile_from_parts<CK>(a, rec, L, nq);
}

// Page piece p of KV tile n: keys [key, key + R) of one page (R = page_piece_rows).
// Returns the piece's first key, or -1 (no piece, empty slot, past the length); the page-table
// load it issues is first used by the caller after its next barrier wait, so the loads of
// the whole tile (one per piece) overlap that wait.
template <int CK>
__device__ __forceinline__ int piece_key(const AttnLaunch& a, const TileInfo<CK>& t, int n, int p) {
  const int ps = a.page_size;
  const int R = page_piece_rows(ps, CK);
  if (p >= kKvTile / R) return -1;
  const int k0 = t.walk.key0(n, (p * R) / CK);
  const int key = k0 + (p * R) % CK;
  const int max_page_idx = (t.L + ps - 1) / ps;
  return (k0 >= 0 && key < t.L && key / ps < max_page_idx) ? key : -1;
}

// SCALED: the prequantized form, whose scores carry a scale per query group and per key
// block and whose output carries a scale per channel (all positive).
template <int CK, bool FACTS, bool SCALED>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, AttnLaunch a) {
  constexpr int NSUB = kKvTile / CK;   // sub-chunks per KV tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_align<1024>(smem_raw);
  uint8_t* q_s = base;                                   // 2 sub-tiles
  uint8_t* k_s = q_s + 2 * kQBytes;                      // K ring
  uint8_t* v_s = k_s + kKStages * kKvBytes;              // V ring
  Ctrl* ctl = reinterpret_cast<Ctrl*>(v_s + kVStages * kKvBytes);

  // Block-sparse (FACTS) launches are ordinary: their plan is complete, so CTAs without a
  // tile leave at once.  Dense launches are programmatic and decide after the wait below.
  if constexpr (FACTS) {
    // one decision for the whole CTA: another CTA may set the status word meanwhile
    const int n0 = a.n_tiles ? *a.n_tiles : a.capacity;
    if (__syncthreads_or(static_cast<int>(blockIdx.x) >= n0 || launch_aborted(a.status))) {
      // (no claims, hence no count, when every tile is some CTA's first)
      if (threadIdx.x == 0 && static_cast<int>(gridDim.x) < n0) claims_done(a.status);
      return;
    }
  }
  const int G = a.G;
  const int TM = kMTileRows / G;                         // tokens per sub-tile
  // Column facts need block-id or valid-bit loads only for block-sparse rows or valid bits
  // (FACTS); dense tiles compute them from the tile index in the softmax itself.
  constexpr bool use_facts = FACTS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int f = 0; f < kFacts; ++f) {
      mbar_init(&ctl->facts_full[f], 1);
      mbar_init(&ctl->facts_empty[f], 8);      // one arrival per softmax warp
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&ctl->s_full[w], 1);
      mbar_init(&ctl->p_full[w], 4);           // one arrival per softmax warp
      mbar_init(&ctl->o_final[w], 1);
      mbar_init(&ctl->o_empty[w], 128);
    }
    // readers of every claim: the V producer, the MMA issuer, the eight softmax warps, and
    // the facts warp (block-sparse) or the K producer (dense, where warp 11 claims)
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(&ctl->t_full[i], 1);
      mbar_init(&ctl->t_empty[i], 3 + 8);
    }
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  // Dense launches are programmatic (they start while the planner's last kernel runs, so the
  // prologue above overlaps its tail): the plan (tile list, count) and the status word are
  // read only after the wait, and whether this CTA has work is decided once, by one thread,
  // so that the CTA takes one branch.
  if constexpr (!FACTS) {
    grid_dependency_wait();
    if (threadIdx.x == 0) {
      const int n0 = a.n_tiles ? *a.n_tiles : a.capacity;
      ctl->skip = (static_cast<int>(blockIdx.x) >= n0 || launch_aborted(a.status)) ? 1 : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  if constexpr (!FACTS) {
    if (ctl->skip) {
      if (warp == 9) tmem_dealloc(tmem, 512);
      if (threadIdx.x == 0 && static_cast<int>(gridDim.x) < (a.n_tiles ? *a.n_tiles : a.capacity))
        claims_done(a.status);
      return;
    }
  }
  const int n_live = a.n_tiles ? *a.n_tiles : a.capacity;
  volatile int* abort_flag = &ctl->abort_flag;
  // The tile of claim sequence s >= 1 (sequence 0 is tile blockIdx.x, never in the ring; the
  // ring holds sequence s as entry s - 1), read by one warp (all lanes) or by one thread
  // (single); a failed wait reads as the end of the list.
  auto read_claim = [&](int s, bool single) -> int {
    const int e = s - 1, slot = e % kTileRing;
    const bool got = single ? mbar_wait_fast(&ctl->t_full[slot], (e / kTileRing) & 1, a.status,
                                             abort_flag)
                            : mbar_wait_warp<true>(&ctl->t_full[slot], (e / kTileRing) & 1,
                                                   a.status, abort_flag);
    const int v = got ? *reinterpret_cast<volatile int*>(&ctl->tidx[slot]) : n_live;
    if (!single) __syncwarp();
    if (got && (single || lane == 0)) mbar_arrive(&ctl->t_empty[slot]);
    return v;
  };
  // The claimer (the K producer of block-sparse launches, warp 11 of dense ones) claims
  // sequence s into ring entry s - 1, its slot free once entry s - 5 is read by every
  // reader; a claim past the list is the end marker.
  auto claim = [&](int s) -> int {
    const int e = s - 1, slot = e % kTileRing;
    const bool free = e < kTileRing ||
                      mbar_wait_warp<true>(&ctl->t_empty[slot], ((e / kTileRing) - 1) & 1,
                                           a.status, abort_flag);
    int v = n_live;
    if (lane == 0) {
      // nothing to claim when every tile is some CTA's first (small plans): no round trip
      if (free && static_cast<int>(gridDim.x) < n_live)
        v = min(n_live, static_cast<int>(gridDim.x) +
                            static_cast<int>(atomicAdd(a.status + 2, 1u)));
      ctl->tidx[slot] = v;
      mbar_arrive(&ctl->t_full[slot]);
    }
    return __shfl_sync(0xffffffffu, v, 0);
  };
  if (warp >= 8) {
  regs_decrease<kControlRegs>();
  if (warp == 8 || warp == 10) {
    // =============================== producers =========================================
    // warp 8 copies Q (lane 0) and K, warp 10 copies V; lane i copies page piece i of a tile
    const bool is_k = warp == 8;
    if (lane == 0) {
      if (is_k) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
      } else {
        tma_prefetch_desc(&vmap);
      }
    }
    const int ps = a.page_size;
    const int R = page_piece_rows(ps, CK);
    // lane 2 p + h copies the 64-column half h of page piece p (R >= 8, so at most 16 pieces),
    // so that a piece's two copies leave from two lanes at once
    const int piece = lane >> 1, half = lane & 1;
    const int stages = is_k ? kKStages : kVStages;
    uint8_t* ring = is_k ? k_s : v_s;
    uint64_t* full = is_k ? ctl->k_full : ctl->v_full;
    uint64_t* empty = is_k ? ctl->k_empty : ctl->v_empty;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    const int head_off = is_k ? a.k_head_off : a.v_head_off;
    int kv_it = 0, qcount = 0;
    bool ok = true;
    const bool claimer = is_k && use_facts;
    int claimed = claimer ? claim(1) : 0;       // the newest claim (sequence s + 1)
    TileRec rec_nx = a.tiles[blockIdx.x];       // record of the next work tile, loaded a tile ahead
    for (int idx = blockIdx.x, s = 0; ok && idx < n_live; ++s) {
      const TileInfo<CK> t = tile_from_rec<CK>(a, rec_nx);
      // tile s + 1: claimed by the K producer at the end of tile s - 1 (it claims s + 2 once
      // this tile's copies are issued, keeping the claim's round trip off the tile's start)
      const int nx = claimer ? claimed : read_claim(s + 1, false);
      if (nx < n_live) rec_nx = a.tiles[nx];
      idx = nx;
      if (t.N == 0) {
        if (claimer && claimed < n_live) claimed = claim(s + 2);
        continue;
      }
      // page ids of the first KV tile: loaded before the wait for the Q buffer
      const int* pt = a.pt_indptr ? a.pt + __ldg(a.pt_indptr + t.rec.b)
                                  : a.pt + static_cast<long long>(t.rec.b) * a.pt_stride;
      int key = piece_key<CK>(a, t, 0, piece);
      int page = key >= 0 ? __ldg(pt + key / ps) : 0;
      if (is_k) {
        if (qcount > 0 &&
            !mbar_wait_warp<true>(&ctl->q_empty, (qcount - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t qbox = 128u * G * TM;
          mbar_arrive_expect_tx(&ctl->q_full, qbox * 2 * t.nsub);
          for (int w = 0; w < t.nsub; ++w)
            for (int h = 0; h < 2; ++h)
              tma_load_3d(q_s + w * kQBytes + h * kQHalf, &qmap, &ctl->q_full, h * 64,
                          t.rec.g * G, t.rec.q_row0 + w * TM);
        }
        ++qcount;
      }
      for (int n = 0; n < t.N; ++n) {
        const int it = kv_it + n, slot = it % stages;
        if (it >= stages &&
            !mbar_wait_warp<true>(&empty[slot], ((it / stages) - 1) & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        bool live = key >= 0;
        if (live && (page < 0 || page >= a.num_pages)) {
          report_error(a.status, kErrMetadata);
          live = false;
        }
        const uint32_t nlive = __popc(__ballot_sync(0xffffffffu, live));
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], nlive * R * 128u);   // a box per lane
        __syncwarp();
        if (live) {
          uint8_t* dst = ring + slot * kKvBytes + static_cast<uint32_t>(piece * R) * 128u +
                         half * kKvHalf;
          const int row = page * a.page_rows + t.rec.g * ps + key % ps + head_off;
          tma_load_2d(dst, map, &full[slot], half * 64, row);
        }
        if (n + 1 < t.N) {                       // next tile's page ids, used after the wait
          key = piece_key<CK>(a, t, n + 1, piece);
          page = key >= 0 ? __ldg(pt + key / ps) : 0;
        }
      }
      kv_it += t.N;
      if (claimer && ok && claimed < n_live) claimed = claim(s + 2);
    }
  } else if (warp == 11 && use_facts) {
    // =============================== column facts ======================================
    constexpr int PARTS = (CK + 31) / 32;        // 32-key spans per sub-chunk
    constexpr int SPAN = CK < 32 ? CK : 32;
    int kv_it = 0;
    bool ok = true;
    TileRec rec_nx = a.tiles[blockIdx.x];       // record of the next work tile, loaded a tile ahead
    for (int idx = blockIdx.x, s = 0; ok && idx < n_live; ++s) {
      const TileInfo<CK> t = tile_from_rec<CK>(a, rec_nx);
      idx = read_claim(s + 1, false);
      if (idx < n_live) rec_nx = a.tiles[idx];
      for (int n = 0; n < t.N; ++n) {
        const int it = kv_it + n, slot = it % kFacts;
        if (it >= kFacts &&
            !mbar_wait_warp<true>(&ctl->facts_empty[slot], ((it / kFacts) - 1) & 1, a.status,
                                  abort_flag)) {
          ok = false;
          break;
        }
        TileFacts* f = &ctl->facts[slot];
        const bool has_c = lane < NSUB;          // lane c: sub-chunk c
        const int k0 = has_c ? t.walk.key0(n, lane) : -1;
        if (has_c) f->k0[lane] = k0;
        if (SCALED && has_c)
          f->cs[lane] = k0 >= 0 ? __ldg(a.k_scale + static_cast<long long>(t.rec.b) *
                                                        a.k_scale_stride + k0 / a.kv_block_size)
                                : 0.f;
        // lane s < NSUB * PARTS: span `part` of sub-chunk c
        const int c_of = min(lane / PARTS, NSUB - 1);
        const int kc = __shfl_sync(0xffffffffu, k0, c_of);
        uint32_t bits = 0u;
        int col0 = -32;
        if (lane < NSUB * PARTS) {
          const int part = lane % PARTS;
          col0 = c_of * CK + part * 32;
          if (kc >= 0) {
            const int key = kc + part * 32;
            const int live = t.L - key;          // keys < L in this span
            bits = live >= SPAN ? (SPAN == 32 ? 0xffffffffu : ((1u << SPAN) - 1u))
                                : (live > 0 ? ((1u << live) - 1u) : 0u);
            if (a.valid_bits) {
              const int wi = key >> 5;
              const uint32_t word =
                  wi < a.valid_words
                      ? __ldg(a.valid_bits + static_cast<long long>(t.rec.b) * a.valid_words + wi)
                      : 0u;
              bits &= (word >> (key & 31));
            }
          }
        }
        uint32_t words[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          words[i] = __reduce_or_sync(0xffffffffu, (col0 >> 5) == i ? bits << (col0 & 31) : 0u);
        const bool zero = __any_sync(0xffffffffu, has_c && (k0 < 0 || k0 + CK > t.L));
        const int kmin = __reduce_min_sync(0xffffffffu, (has_c && k0 >= 0) ? k0 : 0x7fffffff);
        const int kmax = __reduce_max_sync(0xffffffffu, (has_c && k0 >= 0) ? k0 + CK - 1 : -1);
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) f->colmask[i] = words[i];
          f->kmin = kmin;
          f->kmax = kmax;
          f->zero_v = zero;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->facts_full[slot]);
      }
      kv_it += t.N;
    }
  } else if (warp == 11) {
    // =============================== work-tile claims (dense) ==========================
    // up to four claims ahead of the slowest reader, off every other role's path
    for (int s = 1; claim(s) < n_live; ++s) {
    }
  } else if (warp == 9) {
    // =============================== MMA issuer ========================================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, kKvTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, kD, false, true);
      const uint32_t q_addr = smem_u32(q_s);
      const uint32_t k_addr = smem_u32(k_s), v_addr = smem_u32(v_s);
      // Descriptors of the first k-step; later steps add the byte offset / 16 to the start
      // address field (bits 0-13), which never carries out of it inside shared memory.
      const uint64_t q_desc0 = sdesc_sw128(q_addr, 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(k_addr, 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(v_addr, kKvHalf, 1024);
      auto issue_qk = [&](int w, int kslot) {
        const uint64_t qd = q_desc0 + static_cast<uint64_t>((w * kQBytes) >> 4);
        const uint64_t kd = k_desc0 + static_cast<uint64_t>((kslot * kKvBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kQHalf + (ks & 3) * 32) >> 4;
          const uint32_t koff = ((ks >> 2) * kKvHalf + (ks & 3) * 32) >> 4;
          mma_ss(tmem + w * 128, qd + off, kd + koff, idesc_qk, ks > 0);
        }
        mma_commit(&ctl->s_full[w]);
      };
      auto issue_pv = [&](int w, int vslot, bool acc) {
        const uint64_t vd = v_desc0 + static_cast<uint64_t>((vslot * kKvBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kKvTile / 16; ++ks)
          mma_ts(tmem + 256 + w * 128, tmem + w * 128 + ks * 8, vd + ((ks * 16 * 128) >> 4),
                 idesc_pv, (acc || ks > 0));
      };
      int kv_it = 0, qcount = 0, pc1 = 0;
      int ep[2] = {0, 0};                        // epilogues that read O_w so far
      bool ok = true;
      TileRec rec_nx = a.tiles[blockIdx.x];     // record of the next work tile, a tile ahead
      for (int idx = blockIdx.x, s = 0; ok && idx < n_live; ++s) {
        const TileInfo<CK> t = tile_from_rec<CK>(a, rec_nx);
        idx = read_claim(s + 1, true);
        if (idx < n_live) rec_nx = a.tiles[idx];
        const int N = t.N;
        if (N == 0) continue;
        const bool two = t.nsub > 1;
        const int it0 = kv_it;
        ok = mbar_wait_fast(&ctl->q_full, qcount & 1, a.status, abort_flag) &&
             mbar_wait_fast(&ctl->k_full[it0 % kKStages], (it0 / kKStages) & 1, a.status, abort_flag);
        ++qcount;
        if (!ok) break;
        tc_fence_after();
        issue_qk(0, it0 % kKStages);
        if (two) issue_qk(1, it0 % kKStages);
        mma_commit(&ctl->k_empty[it0 % kKStages]);
        if (N == 1) mma_commit(&ctl->q_empty);
        for (int n = 0; n < N; ++n) {
          const int it = it0 + n, vs = it % kVStages;
          const bool more = n + 1 < N;
          const int ks_next = (it + 1) % kKStages;
          // Every input of PV_0(n) and QK_0(n + 1) first (the next K stage has normally landed
          // long before), so that the two groups issue back to back: the issuing thread
          // blocks while the pipe accepts each MMA, and a wait between them would leave the
          // pipe idle on this sub-tile's critical chain P -> PV -> QK -> S.
          if (!mbar_wait_fast(&ctl->v_full[vs], (it / kVStages) & 1, a.status, abort_flag) ||
              (more && !mbar_wait_fast(&ctl->k_full[ks_next], ((it + 1) / kKStages) & 1,
                                        a.status, abort_flag)) ||
              (n == 0 && ep[0] > 0 &&
               !mbar_wait_fast(&ctl->o_empty[0], (ep[0] - 1) & 1, a.status, abort_flag)) ||
              !mbar_wait_fast(&ctl->p_full[0], it & 1, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, vs, n > 0);
          if (more) issue_qk(0, ks_next);
          if (n == N - 1) mma_commit(&ctl->o_final[0]);
          if (two) {
            if (!mbar_wait_fast(&ctl->p_full[1], pc1 & 1, a.status, abort_flag) ||
                (n == 0 && ep[1] > 0 &&
                 !mbar_wait_fast(&ctl->o_empty[1], (ep[1] - 1) & 1, a.status, abort_flag))) {
              ok = false;
              break;
            }
            ++pc1;
            tc_fence_after();
            issue_pv(1, vs, n > 0);
            if (more) issue_qk(1, ks_next);
            if (n == N - 1) mma_commit(&ctl->o_final[1]);
          }
          if (more) {
            mma_commit(&ctl->k_empty[ks_next]);
            if (n + 1 == N - 1) mma_commit(&ctl->q_empty);
          }
          mma_commit(&ctl->v_empty[vs]);
        }
        kv_it += N;
        ++ep[0];
        if (two) ++ep[1];
      }
    }
  }
  } else {
    regs_increase<kSoftmaxRegs>();
    // =============================== softmax (one row per thread) =======================
    const int w = warp >> 2;                       // sub-tile
    const int m = threadIdx.x & 127;               // row inside the sub-tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + w * 128;
    const uint32_t o_col = tmem + lane_base + 256 + w * 128;
    const float sl2 = a.scale_log2;
    const bool causal = a.causal != 0;
    const int wl = a.window_left;
    int kv_it = 0, sc = 0, oc = 0;
    bool ok = true;
    // The next work tile's record is read after the current tile's last softmax and its KV
    // length and query count after the wait for O, so both reads overlap the end of the tile
    // and a work tile starts without a global round trip.
    TileRec rec_nx = a.tiles[blockIdx.x];
    int L_nx, nq_nx;
    request_lengths(a, rec_nx.b, L_nx, nq_nx);
    int idx_nx = 0;                                // the next claim, read at the tile's end
    for (int idx = blockIdx.x, s = 0; ok && idx < n_live; idx = idx_nx, ++s) {
      const TileInfo<CK> t = tile_from_parts<CK>(a, rec_nx, L_nx, nq_nx);
      const int N = t.N;
      const int ntok_w = w == 0 ? t.ntok0 : t.ntok1;
      if (w >= t.nsub) {                           // this sub-tile is empty
        for (int n = 0; ok && use_facts && n < N; ++n) {   // release the tiles' column facts
          const int it = kv_it + n;
          ok = mbar_wait_warp<true>(&ctl->facts_full[it % kFacts], (it / kFacts) & 1, a.status,
                                    abort_flag);
          if (ok && lane == 0) mbar_arrive(&ctl->facts_empty[it % kFacts]);
        }
        idx_nx = read_claim(s + 1, false);
        if (idx_nx < n_live) {
          rec_nx = a.tiles[idx_nx];
          request_lengths(a, rec_nx.b, L_nx, nq_nx);
        }
        kv_it += N;
        continue;
      }
      const int L = t.L;
      const int tok = t.rec.tok0 + w * TM + m / G;   // token index inside the request
      const bool row_valid = (m < G * TM) && (m / G < ntok_w);
      const int pos = L - t.nq + tok;                // query position
      // scaled form: the row's query scale joins the softmax scale (scales are positive)
      float sl2r = sl2;
      if constexpr (SCALED)
        if (row_valid)
          sl2r = sl2 * __ldg(a.q_scale + static_cast<long long>(t.rec.b) * a.q_scale_stride +
                             tok / a.q_scale_group);
      float m_run = -INFINITY, l_run = 0.f;
      for (int n = 0; n < N; ++n) {
        const int it = kv_it + n;
        if (!mbar_wait_fast_warp(&ctl->s_full[w], sc & 1, a.status, abort_flag)) {
          ok = false;
          break;
        }
        ++sc;
        tc_fence_after();
        // ---- per-tile column facts, identical for every row ----------------------------
        int k0[NSUB];
        float cs[NSUB];                            // scaled form: key scale per sub-chunk
        uint32_t colmask[4];
        int kmin, kmax;
        bool zero_v, full;
        if constexpr (FACTS) {                     // from the facts warp
          if (!mbar_wait_warp<true>(&ctl->facts_full[it % kFacts], (it / kFacts) & 1, a.status,
                                    abort_flag)) {
            ok = false;
            break;
          }
          const TileFacts* fc = &ctl->facts[it % kFacts];
#pragma unroll
          for (int c = 0; c < NSUB; ++c) k0[c] = fc->k0[c];
#pragma unroll
          for (int i = 0; i < 4; ++i) colmask[i] = fc->colmask[i];
          kmin = fc->kmin;
          kmax = fc->kmax;
          zero_v = fc->zero_v != 0;
          if constexpr (SCALED) {
#pragma unroll
            for (int c = 0; c < NSUB; ++c) cs[c] = fc->cs[c];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->facts_empty[it % kFacts]);
          full = !a.valid_bits && !zero_v && (!causal || kmax <= pos) && (wl < 0 || kmin >= pos - wl);
        } else {                                   // dense rows: facts from the tile index
          zero_v = false;
          kmin = 0x7fffffff;
          kmax = -1;
  #pragma unroll
          for (int c = 0; c < NSUB; ++c) {
            k0[c] = t.walk.key0(n, c);
            if (k0[c] < 0 || k0[c] + CK > L) zero_v = true;
            if (k0[c] >= 0) {
              kmin = min(kmin, k0[c]);
              kmax = max(kmax, k0[c] + CK - 1);
            }
          }
          full = !a.valid_bits && !zero_v &&
                            (!causal || kmax <= pos) && (wl < 0 || kmin >= pos - wl);
          if (!full) {
  #pragma unroll
            for (int i = 0; i < 4; ++i) colmask[i] = 0u;
  #pragma unroll
            for (int c = 0; c < NSUB; ++c) {
              // live-key bits of the CK columns of sub-chunk c
  #pragma unroll
              for (int part = 0; part < (CK + 31) / 32; ++part) {
                const int col0 = c * CK + part * 32;        // first column of this 32-span
                const int span = CK < 32 ? CK : 32;
                uint32_t bits = 0u;
                if (k0[c] >= 0) {
                  const int key = k0[c] + part * 32;
                  const int live = L - key;                  // keys < L in this span
                  bits = live >= span ? (span == 32 ? 0xffffffffu : ((1u << span) - 1u))
                                      : (live > 0 ? ((1u << live) - 1u) : 0u);
                  if (a.valid_bits) {
                    const int wi = key >> 5;
                    const uint32_t word =
                        wi < a.valid_words
                            ? __ldg(a.valid_bits + static_cast<long long>(t.rec.b) * a.valid_words +
                                    wi)
                            : 0u;
                    bits &= (word >> (key & 31));
                  }
                }
                colmask[col0 >> 5] |= bits << (col0 & 31);
              }
            }
          }
        }
        // ---- S row: four 32-column loads in flight, one wait ----------------------------
        uint32_t r[kKvTile];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32(s_col + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[q * 32]));
        tmem_ld_wait();
        if constexpr (SCALED) {
#pragma unroll
          for (int c = 0; c < kKvTile; ++c)
            r[c] = __float_as_uint(__uint_as_float(r[c]) * cs[c / CK]);
        }
        if (!full) {
          // Invisible scores become -inf in place.  Column facts (slot live, j < len, valid
          // bit) are the same for every row: only 32-column words with a dead key are touched.
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t wbits = colmask[q];
            if (wbits != 0xffffffffu) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (!(wbits & (1u << i))) r[q * 32 + i] = 0xff800000u;
            }
          }
          // causal / window limits only where this row's position cuts the tile
          if ((causal && kmax > pos) || (wl >= 0 && kmin < pos - wl)) {
            int hi_lim[NSUB], lo_lim[NSUB];          // per sub-chunk, relative to its first key
#pragma unroll
            for (int c = 0; c < NSUB; ++c) {
              hi_lim[c] = causal ? pos - k0[c] : 0x7fffffff;
              lo_lim[c] = wl >= 0 ? pos - wl - k0[c] : -0x7fffffff;
            }
            if constexpr (!FACTS) {
              // one unsigned range test and a select per column (the limits differ per row, so
              // a data-dependent branch here would diverge across the warp)
              int span[NSUB];
#pragma unroll
              for (int c = 0; c < NSUB; ++c) {
                // limits clamped into the sub-chunk; an empty range masks every column
                int lo_c = max(lo_lim[c], 0), hi_c = min(hi_lim[c], CK - 1);
                if (hi_c < lo_c) lo_c = hi_c = CK;
                lo_lim[c] = lo_c;
                span[c] = hi_c - lo_c;
              }
#pragma unroll
              for (int c = 0; c < kKvTile; ++c) {
                const bool out = static_cast<unsigned>(c % CK - lo_lim[c / CK]) >
                                 static_cast<unsigned>(span[c / CK]);
                r[c] = out ? 0xff800000u : r[c];
              }
            } else {
              // (block-sparse tiles keep the plain per-column test, which compiles better there)
#pragma unroll
              for (int c = 0; c < kKvTile; ++c)
                if (c % CK > hi_lim[c / CK] || c % CK < lo_lim[c / CK]) r[c] = 0xff800000u;
            }
          }
        }
        // row maximum: 8 independent chains of 3-input max, then a short tree
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2)
          mx[(c >> 1) & 7] = max3f(mx[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
        // scores are scaled by sl2 > 0 after the maximum, which commutes with it
        const float mt =
            fmaxf(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], fmaxf(mx[5], fmaxf(mx[6], mx[7])))) *
            sl2r;
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
        for (int j = 0; j < kKvTile / 2; ++j) {
          float x0, x1;
          ffma2_bcast(x0, x1, __uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]), sl2r, nmu);
          // two f32 ex2 per pair outrun the f16x2 form, whose three conversions cost more
          // than the second ex2
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          if (j & 1) fadd2(sb0, sb1, p0, p1);
          else fadd2(sa0, sa1, p0, p1);
          r[j] = pack_bf16(p0, p1);
        }
        tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        l_run = l_run * alpha + ((sa0 + sa1) + (sb0 + sb1));
        // O was last written by PV of the previous KV tile, which completed before this S
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
        tmem_st_wait();
        if (zero_v && w == 0) {
          // Rows of keys that are not live (past the length, or empty slots) may hold
          // stale or non-finite data; P is 0 there, so make V exactly 0 as well.
          const int vs = it % kVStages;
          if (mbar_wait_warp<true>(&ctl->v_full[vs], (it / kVStages) & 1, a.status, abort_flag)) {
            const int c = m;                         // this thread clears key slot m
            const int k = k0[c / CK];
            if (k < 0 || k + (c % CK) >= L) {
              uint8_t* vt = v_s + vs * kKvBytes;
              const uint4 z = make_uint4(0u, 0u, 0u, 0u);
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[w]);
      }
      idx_nx = read_claim(s + 1, false);
      const bool has_nx = idx_nx < n_live;
      if (has_nx) rec_nx = a.tiles[idx_nx];
      // ---- epilogue ------------------------------------------------------------------------
      bool have_o = false;
      if (ok && N > 0) {
        have_o = mbar_wait_warp<true>(&ctl->o_final[w], oc & 1, a.status, abort_flag);
        ++oc;
        if (have_o) tc_fence_after();
      }
      if (has_nx) request_lengths(a, rec_nx.b, L_nx, nq_nx);
      const int head = t.rec.g * G + (m % G);
      const long long orow = static_cast<long long>(t.rec.q_row0 + w * TM + m / G) * a.Hq + head;
      const float inv = l_run > 0.f ? a.out_scale / l_run : 0.f;
      // the whole O row in flight at once; O_w is then free for the next tile's PV
      uint32_t ov[kD];
      if (have_o) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32(o_col + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[q * 32]));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&ctl->o_empty[w]);
      } else {
#pragma unroll
        for (int i = 0; i < kD; ++i) ov[i] = 0u;
      }
      if constexpr (SCALED) {                 // per-channel value scales
        const float* vsc = a.v_scale + static_cast<long long>(t.rec.b) * a.v_scale_stride;
#pragma unroll
        for (int i = 0; i < kD; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * __ldg(vsc + i));
      }
      // one row per thread, 32 bytes per store where the output allows it (rows are 256 or
      // 512 bytes, so only the base address decides)
      const bool wide = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
      if (row_valid && a.out_dtype == kOutF32) {
        float* dst = static_cast<float*>(a.out) + orow * kD;
#pragma unroll
        for (int i = 0; i < kD / 8; ++i) {
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
        uint16_t* dst = static_cast<uint16_t*>(a.out) + orow * kD;
#pragma unroll
        for (int i = 0; i < kD / 16; ++i) {
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
      if (row_valid && a.lse)
        a.lse[orow] = l_run > 0.f ? (m_run + fast_log2(l_run)) * kLn2 : -INFINITY;
      kv_it += N;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && static_cast<int>(gridDim.x) < n_live) claims_done(a.status);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int CK, bool FACTS, bool SCALED = false>
int launch_ck(const AttnLaunch& a, cudaStream_t st) {
  static std::atomic<uint64_t> smem_set{0};
  if (!kernel_smem_ready(attn_tc_kernel<CK, FACTS, SCALED>, kSmemBytes, smem_set)) return -1;
  const int sms = current_sm_count();
  if (sms <= 0) return -1;
  const int grid = a.capacity < sms ? a.capacity : sms;
  // Dense tiles: programmatic, so the prologue overlaps the planner's last kernel (one
  // GB300: dense prefill step 0.483 -> 0.455 ms).  Block-sparse tiles: an ordinary launch;
  // programmatic, the long block-sparse step got 3.6% slower.
  cudaError_t e;
  if constexpr (!FACTS) {
    e = launch_after_previous(attn_tc_kernel<CK, FACTS, SCALED>, dim3(grid), dim3(kThreads),
                              kSmemBytes, st, a.qmap, a.kmap, a.vmap, a);
  } else {
    attn_tc_kernel<CK, FACTS, SCALED><<<grid, kThreads, kSmemBytes, st>>>(a.qmap, a.kmap, a.vmap, a);
    e = cudaSuccess;
  }
  count_launches(1);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_attn(const AttnLaunch& a, cudaStream_t st) {
  if (a.capacity <= 0) return 0;
  if (a.k_scale) {                               // the prequantized form: 64-key blocks only
    if (!a.block_sparse || attn_sub_chunk(a.kv_block_size, true) != 64 || !a.q_scale ||
        !a.v_scale || a.q_scale_group <= 0)
      return -2;
    return launch_ck<64, true, true>(a, st);
  }
  switch (attn_sub_chunk(a.kv_block_size, a.block_sparse != 0)) {
    case 8: return launch_ck<8, true>(a, st);
    case 16: return launch_ck<16, true>(a, st);
    case 32: return launch_ck<32, true>(a, st);
    case 64: return launch_ck<64, true>(a, st);
    case 128:
      return (a.block_sparse || a.valid_bits) ? launch_ck<128, true>(a, st)
                                              : launch_ck<128, false>(a, st);
    default: return -2;
  }
}

}  // namespace pa
