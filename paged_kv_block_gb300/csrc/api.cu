// C ABI of libpagedattn: argument checks, workspace layouts, tensor-map encoding and the
// launch sequence of each entry point (include/paged_attn.h documents the contract).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/paged_attn.h"
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr size_t kAlign = 256;
constexpr float kLog2e = 1.4426950408889634f;

// ---- tensor-map encoding through the driver entry point -----------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bump allocator over the caller's workspace (offsets only).
struct Layout {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  }
};

// ---- sparse (BSR / bitmap) layouts -------------------------------------------------------
struct SparseLayout {
  size_t status, n_tiles, tmp, sorted, hist, offs, indptr, indices, total;
  int capacity, max_cost, tile_tokens;
  long long bitmap_capacity;
};

bool sparse_params_ok(const paged_attn_params* p) {
  if (!p) return false;
  if (p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->num_qo_heads % p->num_kv_heads) return false;
  if (p->q_len < 0) return false;
  if (p->form == PAGED_ATTN_FORM_BSR) {
    const int G = p->num_qo_heads / p->num_kv_heads;
    if (p->batch < 0 || p->head_dim != 128 || G > 128) return false;
    if (p->page_size < 8 || p->page_size > 128 || p->page_size % 8) return false;
    if (p->num_pages <= 0 || p->q_block_size <= 0) return false;
    const int kvbs = p->kv_block_size;
    if (!(kvbs == 8 || kvbs == 16 || kvbs == 32 || (kvbs > 0 && kvbs % 64 == 0))) return false;
    if ((static_cast<long long>(p->q_block_size) * G) % 8) return false;
    if (p->max_seq_len_kv < 0) return false;
    if (p->mask_type != PAGED_ATTN_MASK_DENSE && p->mask_type != PAGED_ATTN_MASK_CAUSAL) return false;
    const long long rows = static_cast<long long>(p->num_pages) * (p->combined_cache ? 2 : 1) *
                           p->num_kv_heads * p->page_size;
    if (rows >= (1LL << 31)) return false;
    if (static_cast<long long>(p->batch) * p->q_len >= (1LL << 31)) return false;
    return true;
  }
  if (p->form == PAGED_ATTN_FORM_BITMAP || p->form == PAGED_ATTN_FORM_INDEXED) {
    if (p->head_dim != 256 || p->block_size != 4 || p->num_blocks < 0) return false;
    if (p->form == PAGED_ATTN_FORM_INDEXED && p->index_width <= 0) return false;
    return true;
  }
  return false;
}

SparseLayout sparse_layout(const paged_attn_params* p) {
  SparseLayout s{};
  Layout l;
  s.status = l.take(sizeof(uint32_t) * 4);
  s.n_tiles = s.status + sizeof(uint32_t);
  if (p->form == PAGED_ATTN_FORM_BSR) {
    const int G = p->num_qo_heads / p->num_kv_heads;
    s.tile_tokens = cta_tile_tokens(G);
    const int Sq = p->q_len, qbs = p->q_block_size;
    const int nqb = Sq > 0 ? ceil_div(Sq, qbs) : 0;
    long long per_bg = 0;
    if (nqb > 0) {
      const int full = ceil_div(qbs, s.tile_tokens);
      const int last_n = Sq - (nqb - 1) * qbs;
      per_bg = static_cast<long long>(nqb - 1) * full + ceil_div(last_n, s.tile_tokens);
    }
    s.capacity = static_cast<int>(static_cast<long long>(p->batch) * p->num_kv_heads * per_bg);
    const int max_blocks = p->max_seq_len_kv > 0 ? ceil_div(p->max_seq_len_kv, p->kv_block_size) : 1;
    s.max_cost = max_blocks < kMaxSortCost ? max_blocks : kMaxSortCost;
    s.tmp = l.take(sizeof(TileRec) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
    s.sorted = l.take(sizeof(TileRec) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
    const size_t ints = tile_sort_scratch_ints(s.capacity, s.max_cost);
    s.hist = l.take(ints * sizeof(int));
    s.offs = l.take(ints * sizeof(int));
  } else {
    const long long T = p->q_len;
    const long long mb = p->max_blocks_per_query > 0 ? p->max_blocks_per_query
                         : (p->form == PAGED_ATTN_FORM_INDEXED ? p->index_width : p->num_blocks);
    s.bitmap_capacity = T * (mb > 0 ? mb : 1);
    s.indptr = l.take(sizeof(int) * static_cast<size_t>(T + 1));
    s.indices = l.take(sizeof(int) * static_cast<size_t>(s.bitmap_capacity));
  }
  s.total = l.off;
  return s;
}

// ---- prefill layout ----------------------------------------------------------------------
struct PrefillLayout {
  size_t status, n_tiles, tile_off, tmp, sorted, hist, offs, total;
  int capacity, max_cost, tile_tokens;
};

bool prefill_params_ok(const paged_prefill_params* p) {
  if (!p) return false;
  if (p->batch < 0 || p->total_q < 0) return false;
  if (p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->num_qo_heads % p->num_kv_heads) return false;
  const int G = p->num_qo_heads / p->num_kv_heads;
  if (G > 128 || (p->head_dim != 128 && p->head_dim != 256)) return false;
  if (!(p->page_size == 16 || p->page_size == 32 || p->page_size == 64 || p->page_size == 128))
    return false;
  if (p->num_pages <= 0 || p->max_pages_per_request <= 0) return false;
  if (p->mask_type != PAGED_ATTN_MASK_DENSE && p->mask_type != PAGED_ATTN_MASK_CAUSAL) return false;
  if (p->window_left < -1) return false;
  if (p->window_left >= 0 && p->mask_type != PAGED_ATTN_MASK_CAUSAL) return false;
  if (p->out_dtype < PAGED_ATTN_DTYPE_BF16 || p->out_dtype > PAGED_ATTN_DTYPE_FP32) return false;
  if (static_cast<long long>(p->num_pages) * p->num_kv_heads * p->page_size >= (1LL << 31))
    return false;
  return true;
}

PrefillLayout prefill_layout(const paged_prefill_params* p) {
  PrefillLayout s{};
  Layout l;
  s.status = l.take(sizeof(uint32_t) * 4);
  s.n_tiles = s.status + sizeof(uint32_t);
  const int G = p->num_qo_heads / p->num_kv_heads;
  // D = 128: two 128-row sub-tiles per tile; D = 256: one
  s.tile_tokens = p->head_dim == 256 ? sub_tile_tokens(G) : cta_tile_tokens(G);
  s.capacity = static_cast<int>(static_cast<long long>(p->num_kv_heads) *
                                (ceil_div(p->total_q, s.tile_tokens) + p->batch));
  const long long max_keys = static_cast<long long>(p->max_pages_per_request) * p->page_size;
  const long long mc = ceil_div_ll(max_keys, kKvTile);
  s.max_cost = static_cast<int>(mc < kMaxSortCost ? mc : kMaxSortCost);
  s.tile_off = l.take(sizeof(int) * static_cast<size_t>(p->batch + 1));
  s.tmp = l.take(sizeof(TileRec) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
  s.sorted = l.take(sizeof(TileRec) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
  const size_t ints = tile_sort_scratch_ints(s.capacity, s.max_cost);
  s.hist = l.take(ints * sizeof(int));
  s.offs = l.take(ints * sizeof(int));
  s.total = l.off;
  return s;
}

// ---- decode layout ------------------------------------------------------------------------
// Rows of one (request, KV head) unit: G x (queries per request).  Up to kDecodeMaxRows the
// split-KV decode kernel runs; beyond, the work is prefill-shaped and runs as dense tiles of
// the tensor-core kernel over the CSR page table.
constexpr int kDecodeMaxRows = 64;

struct DecodeLayout {
  size_t status, split_off, counters, items, order, part_lse, part_o;   // split-KV route
  size_t n_tiles, tile_off, tmp, sorted, hist, offs;             // tile route
  size_t total;
  int capacity, chunk, max_splits;
  int q_per_item, q_rows, rows, tiled, max_cost, tile_tokens;
};

bool decode_packed(const paged_decode_params* p) { return p->max_seq_len_q > 0; }
int decode_q_per_item(const paged_decode_params* p) {
  return decode_packed(p) ? p->max_seq_len_q : (p->seq_len_q > 1 ? p->seq_len_q : 1);
}

bool decode_params_ok(const paged_decode_params* p) {
  if (!p) return false;
  if (p->batch < 0 || p->num_qo_heads <= 0 || p->num_kv_heads <= 0) return false;
  if (p->num_qo_heads % p->num_kv_heads) return false;
  const int G = p->num_qo_heads / p->num_kv_heads;
  if (G > 16 || p->head_dim != 128) return false;
  if (p->page_size < 8 || p->page_size > 128 || p->page_size % 8) return false;
  if (p->num_pages <= 0) return false;
  if (p->max_seq_len <= 0 || p->max_seq_len > 2147483520) return false;
  if (p->mask_type != PAGED_ATTN_MASK_DENSE && p->mask_type != PAGED_ATTN_MASK_CAUSAL) return false;
  if (p->window_left < -1) return false;
  if (p->window_left >= 0 && p->mask_type != PAGED_ATTN_MASK_CAUSAL) return false;
  if (p->split_chunk < 0 || p->split_chunk % 128) return false;
  if (p->seq_len_q < 0 || p->max_seq_len_q < 0 || p->total_q < 0) return false;
  if (p->out_dtype < PAGED_ATTN_DTYPE_BF16 || p->out_dtype > PAGED_ATTN_DTYPE_FP32) return false;
  if (decode_packed(p)) {
    if (p->seq_len_q > 1) return false;                    // one form at a time
    if (p->total_q < p->batch) return false;               // every request owns >= 1 row
    if (static_cast<long long>(p->batch) * p->max_seq_len_q < p->total_q) return false;
  } else if (static_cast<long long>(p->batch) * decode_q_per_item(p) >= (1LL << 31)) {
    return false;
  }
  const long long rows = static_cast<long long>(p->num_pages) * (p->combined_cache ? 2 : 1) *
                         p->num_kv_heads * p->page_size;
  if (rows >= (1LL << 31)) return false;
  if (static_cast<long long>(G) * decode_q_per_item(p) > kDecodeMaxRows && G * 2 > kMTileRows)
    return false;
  return true;
}

int decode_chunk(const paged_decode_params* p) {
  if (p->split_chunk > 0) return p->split_chunk;
  const long long tiles = ceil_div_ll(p->max_seq_len, 128);
  long long ct = static_cast<long long>(p->batch) * p->num_kv_heads * tiles / (16LL * num_sms());
  if (ct < 1) ct = 1;
  if (ct > tiles) ct = tiles;
  return static_cast<int>(128 * ct);
}

DecodeLayout decode_layout(const paged_decode_params* p) {
  DecodeLayout s{};
  Layout l;
  const int G = p->num_qo_heads / p->num_kv_heads;
  s.q_per_item = decode_q_per_item(p);
  s.q_rows = decode_packed(p) ? p->total_q : p->batch * s.q_per_item;
  const long long rows = static_cast<long long>(G) * s.q_per_item;
  s.tiled = rows > kDecodeMaxRows;
  s.rows = s.tiled ? 0 : static_cast<int>(rows);
  s.chunk = decode_chunk(p);
  s.status = l.take(sizeof(uint32_t) * 4);
  if (!s.tiled) {
    s.max_splits = static_cast<int>(ceil_div_ll(p->max_seq_len, s.chunk));
    if (s.max_splits < 1) s.max_splits = 1;
    s.capacity = static_cast<int>(static_cast<long long>(p->batch) * p->num_kv_heads * s.max_splits);
    s.split_off = l.take(sizeof(int) * static_cast<size_t>(p->batch + 1));
    s.counters = l.take(sizeof(int) * (static_cast<size_t>(p->batch) * p->num_kv_heads + 1));
    s.items = l.take(sizeof(SplitItem) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
    s.order = l.take(sizeof(int) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
    s.part_lse = l.take(sizeof(float) * static_cast<size_t>(s.capacity) * s.rows + 4);
    s.part_o = l.take(sizeof(float) * static_cast<size_t>(s.capacity) * s.rows * p->head_dim + 4);
  } else {
    s.n_tiles = s.status + sizeof(uint32_t);
    s.tile_tokens = cta_tile_tokens(G);
    s.capacity = static_cast<int>(static_cast<long long>(p->num_kv_heads) *
                                  (ceil_div(s.q_rows, s.tile_tokens) + p->batch));
    const long long mc = ceil_div_ll(p->max_seq_len, kKvTile);
    s.max_cost = static_cast<int>(mc < kMaxSortCost ? mc : kMaxSortCost);
    s.tile_off = l.take(sizeof(int) * static_cast<size_t>(p->batch + 1));
    s.tmp = l.take(sizeof(TileRec) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
    s.sorted = l.take(sizeof(TileRec) * static_cast<size_t>(s.capacity > 0 ? s.capacity : 1));
    const size_t ints = tile_sort_scratch_ints(s.capacity, s.max_cost);
    s.hist = l.take(ints * sizeof(int));
    s.offs = l.take(ints * sizeof(int));
  }
  s.total = l.off;
  return s;
}

// ---- prequantized block-sparse layout ------------------------------------------------------
struct SageLayout {
  paged_attn_params bsr;       // the block-sparse form the inputs are turned into
  SparseLayout s;              // its plan, at offset 0 (so the status word is the usual one)
  size_t q_bf16, k_bf16, v_bf16, counts, block_indptr, block_indices, kv_indptr, kv_indices,
      seq_lens, valid_bits, total;
  int NB, QB, QG, BH;
};

bool sage_params_ok(const paged_sage_params* p) {
  if (!p) return false;
  if (p->batch < 0 || p->num_heads <= 0 || p->q_len < 0 || p->kv_len < 0) return false;
  if (p->head_dim != 128 || p->capacity < 0) return false;
  if (p->block_sparse_num < 0 || p->block_sparse_num > p->capacity) return false;
  if (p->block_sizes_rank < 0 || p->block_sizes_rank > 3) return false;
  const long long BH = static_cast<long long>(p->batch) * p->num_heads;
  if (BH > 65535) return false;
  const long long NB = (p->kv_len + 63) / 64;
  if (BH * NB * 64 * 128 >= (1LL << 31) || BH * p->q_len >= (1LL << 31)) return false;
  return true;
}

SageLayout sage_layout(const paged_sage_params* p) {
  SageLayout g{};
  g.BH = p->batch * p->num_heads;
  g.NB = (p->kv_len + 63) / 64;
  g.QB = (p->q_len + 63) / 64;
  g.QG = (p->q_len + 127) / 128 * 4;
  paged_attn_params& b = g.bsr;
  b.form = PAGED_ATTN_FORM_BSR;
  b.batch = g.BH;
  b.q_len = p->q_len;
  b.num_qo_heads = 1;
  b.num_kv_heads = 1;
  b.head_dim = 128;
  b.page_size = 64;
  b.num_pages = g.BH * g.NB > 0 ? g.BH * g.NB : 1;
  b.combined_cache = 0;
  b.q_block_size = 64;
  b.kv_block_size = 64;
  b.max_seq_len_kv = g.NB * 64;
  b.mask_type = PAGED_ATTN_MASK_DENSE;
  b.has_valid_bits = 1;
  b.sm_scale = p->softmax_scale;
  g.s = sparse_layout(&b);
  Layout l;
  l.off = g.s.total;
  const size_t BH = static_cast<size_t>(g.BH), NB = static_cast<size_t>(g.NB);
  const size_t QB = static_cast<size_t>(g.QB);
  g.q_bf16 = l.take(BH * p->q_len * 128 * 2 + 16);
  g.k_bf16 = l.take(BH * NB * 64 * 128 * 2 + 16);
  g.v_bf16 = l.take(BH * NB * 64 * 128 * 2 + 16);
  g.counts = l.take(sizeof(int) * (BH * QB + 1));
  g.block_indptr = l.take(sizeof(int) * (BH * (QB + 1) + 1));
  g.block_indices = l.take(sizeof(int) * (BH * QB * static_cast<size_t>(p->capacity) + 1));
  g.kv_indptr = l.take(sizeof(int) * (BH + 1));
  g.kv_indices = l.take(sizeof(int) * (BH * NB + 1));
  g.seq_lens = l.take(sizeof(int) * (BH + 1));
  g.valid_bits = l.take(sizeof(uint32_t) * (BH * 2 * NB + 1));
  g.total = l.off;
  return g;
}

// Scales of the prequantized form (see AttnLaunch).
struct ScaleSet {
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int q_group, q_stride, k_stride, v_stride;
};

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

bool encode_rows_map(CUtensorMap* map, const void* base, long long rows, int D, int box_rows) {
  auto fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap* map, const void* base, long long rows, int Hq, int D,
                  int box_heads, int box_tokens) {
  auto fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_tokens)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_block_pair_map(CUtensorMap* map, const void* base, long long tokens, int Hkv, int D) {
  auto fn = encode_fn();
  if (!fn || tokens <= 0 || D % 64 || D > 256) return false;
  // [tokens, Hkv, D] viewed as (64 columns, head, token, 64-column chunk); the chunk stride
  // (128 B) is smaller than the others, which the copy engine allows.
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(tokens),
                        static_cast<cuuint64_t>(D / 64)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hkv) * D * 2,
                           128};
  cuuint32_t box[4] = {64, 2, 4, static_cast<cuuint32_t>(D / 64)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- kernel timer and launch counter -------------------------------------------------------
namespace {
std::atomic<long long> g_launches{0};
struct Timer {
  std::mutex mu;
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pairs;
  size_t used = 0;
} g_timer;
}  // namespace

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

void timer_begin(cudaStream_t st, void** token) {
  *token = nullptr;
  std::lock_guard<std::mutex> lk(g_timer.mu);
  if (!g_timer.on) return;
  if (g_timer.used == g_timer.pairs.size()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return; }
    g_timer.pairs.emplace_back(a, b);
  }
  auto& pr = g_timer.pairs[g_timer.used++];
  cudaEventRecord(pr.first, st);
  *token = pr.second;
}

void timer_end(cudaStream_t st, void* token) {
  if (token) cudaEventRecord(static_cast<cudaEvent_t>(token), st);
}

int launch_qsa(const paged_attn_params* p, const paged_attn_meta* m, const void* q,
               const void* k, const void* v, void* out, float* out_fp32, float* lse,
               const int* indptr, const int* indices, uint32_t* status, cudaStream_t st);

namespace {

// Decode whose (request, KV head) units exceed kDecodeMaxRows rows: the dense tile planner
// and the tensor-core kernel, with the decode page table (CSR) and query layout.
int decode_run_tiled(const paged_decode_params* p, const DecodeLayout& s, const void* query,
                     const void* k, const void* v, const int32_t* kv_indptr,
                     const int32_t* kv_indices, const int32_t* seq_lens,
                     const int32_t* qo_indptr, void* out, float* lse, void* ws,
                     cudaStream_t st) {
  const int Hq = p->num_qo_heads, Hkv = p->num_kv_heads, G = Hq / Hkv, D = p->head_dim;
  const int ps = p->page_size;
  const int causal = p->mask_type == PAGED_ATTN_MASK_CAUSAL;
  const int q_len = qo_indptr ? 0 : s.q_per_item;
  uint32_t* status = at<uint32_t>(ws, s.status);
  int* n_tiles = at<int>(ws, s.n_tiles);
  TileRec* tmp = at<TileRec>(ws, s.tmp);
  TileRec* sorted = at<TileRec>(ws, s.sorted);
  launch_prefill_tiles(qo_indptr, q_len, seq_lens, p->batch, Hkv, s.tile_tokens, causal,
                       p->window_left, s.capacity, at<int>(ws, s.tile_off), n_tiles, tmp, status,
                       st);
  launch_tile_sort(tmp, sorted, n_tiles, 0, s.capacity, s.max_cost, at<int>(ws, s.hist),
                   at<int>(ws, s.offs), st);
  const float scale =
      p->bmm1_scale > 0.f ? p->bmm1_scale : 1.0f / std::sqrt(static_cast<float>(D));
  AttnLaunch a{};
  const int R = page_piece_rows(ps, kKvTile);
  const long long pool_rows = static_cast<long long>(p->num_pages) * (p->combined_cache ? 2 : 1) *
                              Hkv * ps;
  if (!encode_q_map(&a.qmap, query, s.q_rows, Hq, D, G, sub_tile_tokens(G)) ||
      !encode_rows_map(&a.kmap, k, pool_rows, D, R) ||
      !encode_rows_map(&a.vmap, p->combined_cache ? k : v, pool_rows, D, R))
    return PAGED_ATTN_ERR_CUDA;
  a.tiles = sorted;
  a.n_tiles = n_tiles;
  a.capacity = s.capacity;
  a.pt = kv_indices;
  a.pt_indptr = kv_indptr;
  a.pt_stride = 0;
  a.seq_lens = seq_lens;
  a.qo_indptr = qo_indptr;
  a.q_len = q_len;
  a.valid_bits = nullptr;
  a.valid_words = 0;
  a.block_sparse = 0;
  a.block_indices = nullptr;
  a.kv_block_size = kKvTile;
  a.out = out;
  a.out_dtype = p->out_dtype;
  a.lse = lse;
  a.status = status;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.D = D;
  a.page_size = ps;
  a.page_rows = (p->combined_cache ? 2 : 1) * Hkv * ps;
  a.k_head_off = 0;
  a.v_head_off = p->combined_cache ? Hkv * ps : 0;
  a.num_pages = p->num_pages;
  a.causal = causal;
  a.window_left = p->window_left;
  a.scale_log2 = scale * kLog2e;
  a.out_scale = p->bmm2_scale;
  void* tok;
  timer_begin(st, &tok);
  const int rc = launch_attn(a, st);
  timer_end(st, tok);
  if (rc == -2) return PAGED_ATTN_ERR_UNSUPPORTED;
  return rc == 0 ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

}  // namespace

// Block-sparse launch of a planned BSR form (the workspace holds the plan at `s`); `sc`
// carries the scales of the prequantized form, nullptr otherwise.
int bsr_launch(const paged_attn_params* p, const paged_attn_meta* m, const SparseLayout& s,
               const void* q, const void* k, const void* v, void* out, float* lse, void* ws,
               uint32_t* status, float scale, const ScaleSet* sc, cudaStream_t st) {
  const int D = p->head_dim;
  if (s.capacity == 0) return PAGED_ATTN_OK;
  const int Hq = p->num_qo_heads, Hkv = p->num_kv_heads, G = Hq / Hkv, ps = p->page_size;
  AttnLaunch a{};
  const int ck = attn_sub_chunk(p->kv_block_size, true);
  const int R = page_piece_rows(ps, ck);
  const long long pool_rows = static_cast<long long>(p->num_pages) * (p->combined_cache ? 2 : 1) *
                              Hkv * ps;
  if (!encode_q_map(&a.qmap, q, static_cast<long long>(p->batch) * p->q_len, Hq, D, G,
                    sub_tile_tokens(G)) ||
      !encode_rows_map(&a.kmap, k, pool_rows, D, R) ||
      !encode_rows_map(&a.vmap, p->combined_cache ? k : v, pool_rows, D, R))
    return PAGED_ATTN_ERR_CUDA;
  a.tiles = at<TileRec>(ws, s.sorted);
  a.n_tiles = nullptr;
  a.capacity = s.capacity;
  a.pt = m->kv_indices_dev;
  a.pt_indptr = m->kv_indptr_dev;
  a.pt_stride = 0;
  a.seq_lens = m->seq_lens_kv_dev;
  a.qo_indptr = nullptr;
  a.q_len = p->q_len;
  a.valid_bits = p->has_valid_bits ? m->kv_valid_bits_dev : nullptr;
  a.valid_words = ceil_div(p->max_seq_len_kv > 0 ? p->max_seq_len_kv : 1, 32);
  a.block_sparse = 1;
  a.block_indices = m->block_indices_dev;
  a.kv_block_size = p->kv_block_size;
  a.out = out;
  a.out_dtype = PAGED_ATTN_DTYPE_BF16;
  a.lse = lse;
  a.status = status;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.D = D;
  a.page_size = ps;
  a.page_rows = (p->combined_cache ? 2 : 1) * Hkv * ps;
  a.k_head_off = 0;
  a.v_head_off = p->combined_cache ? Hkv * ps : 0;
  a.num_pages = p->num_pages;
  a.causal = p->mask_type == PAGED_ATTN_MASK_CAUSAL;
  a.window_left = -1;
  a.scale_log2 = scale * kLog2e;
  a.out_scale = 1.0f;
  if (sc) {
    a.q_scale = sc->q_scale;
    a.k_scale = sc->k_scale;
    a.v_scale = sc->v_scale;
    a.q_scale_group = sc->q_group;
    a.q_scale_stride = sc->q_stride;
    a.k_scale_stride = sc->k_stride;
    a.v_scale_stride = sc->v_stride;
  }
  void* tok;
  timer_begin(st, &tok);
  const int rc = launch_attn(a, st);
  timer_end(st, tok);
  if (rc == -2) return PAGED_ATTN_ERR_UNSUPPORTED;
  return rc == 0 ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* paged_attn_strerror(int s) {
  switch (s) {
    case PAGED_ATTN_OK: return "ok";
    case PAGED_ATTN_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PAGED_ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case PAGED_ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case PAGED_ATTN_ERR_CUDA: return "CUDA error";
    case PAGED_ATTN_ERR_TIMEOUT: return "a device-side wait timed out";
    case PAGED_ATTN_ERR_METADATA: return "metadata outside its contract";
    case PAGED_ATTN_ERR_CAPACITY: return "plan exceeded its workspace capacity";
    default: return "unknown status";
  }
}

size_t paged_attn_workspace_size(const paged_attn_params* p) {
  if (!sparse_params_ok(p)) return 0;
  return sparse_layout(p).total;
}

int paged_attn_validate_bsr(const paged_attn_params* p, const int32_t* kv_indptr,
                            const int32_t* kv_indices, int64_t n_kv_indices,
                            const int32_t* block_indptr, const int32_t* block_indices,
                            int64_t n_block_indices, const int32_t* seq_lens, int64_t* bad) {
  auto fail = [&](int64_t i) {
    if (bad) *bad = i;
    return PAGED_ATTN_ERR_METADATA;
  };
  if (!sparse_params_ok(p) || p->form != PAGED_ATTN_FORM_BSR) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (!kv_indptr || !seq_lens || !block_indptr) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (n_kv_indices > 0 && !kv_indices) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (n_block_indices > 0 && !block_indices) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const int B = p->batch, Hkv = p->num_kv_heads, ps = p->page_size;
  if (kv_indptr[0] != 0) return fail(0);
  for (int b = 0; b < B; ++b) {
    if (kv_indptr[b + 1] < kv_indptr[b]) return fail(b + 1);
    const int L = seq_lens[b];
    if (L < 0 || L > p->max_seq_len_kv) return fail(b);
    const int need = ceil_div(L, ps);
    if (kv_indptr[b + 1] - kv_indptr[b] < need) return fail(b);
    for (int i = 0; i < need; ++i) {
      const int64_t j = static_cast<int64_t>(kv_indptr[b]) + i;
      if (j >= n_kv_indices) return fail(j);
      if (kv_indices[j] < 0 || kv_indices[j] >= p->num_pages) return fail(j);
    }
  }
  if (kv_indptr[B] != n_kv_indices) return fail(B);
  const int nqb = p->q_len > 0 ? ceil_div(p->q_len, p->q_block_size) : 0;
  const int max_blk = ceil_div(p->max_seq_len_kv, p->kv_block_size);
  std::vector<uint8_t> seen(static_cast<size_t>(max_blk > 0 ? max_blk : 1), 0);
  for (int b = 0; b < B; ++b)
    for (int g = 0; g < Hkv; ++g)
      for (int r = 0; r < nqb; ++r) {
        const int64_t row = (static_cast<int64_t>(b) * Hkv + g) * (nqb + 1) + r;
        const int s = block_indptr[row], e = block_indptr[row + 1];
        if (s < 0 || e < s || e > n_block_indices) return fail(row);
        for (int i = s; i < e; ++i) {
          const int c = block_indices[i];
          if (c < 0 || c >= max_blk || seen[c]) {
            for (int k = s; k < i; ++k)
              if (block_indices[k] >= 0 && block_indices[k] < max_blk) seen[block_indices[k]] = 0;
            return fail(i);
          }
          seen[c] = 1;
        }
        for (int i = s; i < e; ++i) seen[block_indices[i]] = 0;
      }
  return PAGED_ATTN_OK;
}

int paged_attn_plan(const paged_attn_params* p, const paged_attn_meta* m, void* ws,
                    size_t ws_bytes, void* stream) {
  if (!sparse_params_ok(p) || !m) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const SparseLayout s = sparse_layout(p);
  if (!ws || ws_bytes < s.total) return PAGED_ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, s.status);
  if (p->form == PAGED_ATTN_FORM_BSR && m->block_indptr_dev &&
      bsr_plan_is_small(p->batch, p->num_kv_heads, p->q_len, p->q_block_size, s.capacity,
                        s.max_cost)) {
    // one launch: tiles, their order and the status clear
    launch_bsr_plan_small(m->block_indptr_dev, p->batch, p->num_kv_heads, p->q_len,
                          p->q_block_size, s.tile_tokens, s.capacity, s.max_cost,
                          at<TileRec>(ws, s.sorted), status, st);
    return cudaGetLastError() == cudaSuccess ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
  }
  if (cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), st) != cudaSuccess) return PAGED_ATTN_ERR_CUDA;
  if (p->form == PAGED_ATTN_FORM_BSR) {
    if (!m->block_indptr_dev) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
    TileRec* tmp = at<TileRec>(ws, s.tmp);
    launch_bsr_tiles(m->block_indptr_dev, p->batch, p->num_kv_heads, p->q_len, p->q_block_size,
                     s.tile_tokens, tmp, st);
    launch_tile_sort(tmp, at<TileRec>(ws, s.sorted), nullptr, s.capacity, s.capacity, s.max_cost,
                     at<int>(ws, s.hist), at<int>(ws, s.offs), st);
  } else if (p->form == PAGED_ATTN_FORM_INDEXED) {
    if (!m->sel_indices_dev || !m->lo_dev || !m->hi_dev || !m->block_first_dev ||
        !m->block_last_dev)
      return PAGED_ATTN_ERR_INVALID_ARGUMENT;
    launch_indexed_plan(m->sel_indices_dev, p->index_width, m->lo_dev, m->hi_dev,
                        m->block_first_dev, m->block_last_dev, p->q_len, p->num_blocks,
                        s.bitmap_capacity, at<int>(ws, s.indptr), at<int>(ws, s.indices), status,
                        st);
  } else {
    if (!m->sel_blocks_dev || !m->lo_dev || !m->hi_dev || !m->block_first_dev || !m->block_last_dev)
      return PAGED_ATTN_ERR_INVALID_ARGUMENT;
    launch_bitmap_plan(m->sel_blocks_dev, m->lo_dev, m->hi_dev, m->block_first_dev,
                       m->block_last_dev, p->q_len, p->num_blocks, s.bitmap_capacity,
                       at<int>(ws, s.indptr), at<int>(ws, s.indices), status, st);
  }
  return cudaGetLastError() == cudaSuccess ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

int paged_attn_run(const paged_attn_params* p, const paged_attn_meta* m, const void* q,
                   const void* k, const void* v, void* out, float* out_fp32, float* lse,
                   void* ws, size_t ws_bytes, void* stream) {
  if (!sparse_params_ok(p) || !m || !q || !k || !out) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const SparseLayout s = sparse_layout(p);
  if (!ws || ws_bytes < s.total) return PAGED_ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, s.status);
  const int D = p->head_dim;
  const float scale = p->sm_scale > 0.f ? p->sm_scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (p->form == PAGED_ATTN_FORM_BITMAP || p->form == PAGED_ATTN_FORM_INDEXED) {
    if (!v) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
    paged_attn_params pp = *p;
    pp.sm_scale = scale;
    const int rc = launch_qsa(&pp, m, q, k, v, out, out_fp32, lse, at<int>(ws, s.indptr),
                              at<int>(ws, s.indices), status, st);
    return rc;
  }
  if (!m->kv_indptr_dev || !m->block_indptr_dev || !m->seq_lens_kv_dev)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (!p->combined_cache && !v) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (p->has_valid_bits && !m->kv_valid_bits_dev) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || (v && !aligned16(v)) || !aligned16(out))
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  return bsr_launch(p, m, s, q, k, v, out, lse, ws, status, scale, nullptr, st);
}

size_t paged_prefill_workspace_size(const paged_prefill_params* p) {
  if (!prefill_params_ok(p)) return 0;
  return prefill_layout(p).total;
}

int paged_prefill_run(const paged_prefill_params* p, const void* q, const void* kc,
                      const void* vc, const int32_t* qo_indptr, const int32_t* block_tables,
                      const int32_t* seq_lens, void* out, float* lse, void* ws, size_t ws_bytes,
                      void* stream) {
  if (!prefill_params_ok(p) || !q || !kc || !vc || !qo_indptr || !block_tables || !seq_lens ||
      !out)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(out))
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const PrefillLayout s = prefill_layout(p);
  if (!ws || ws_bytes < s.total) return PAGED_ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, s.status);
  if (cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), st) != cudaSuccess) return PAGED_ATTN_ERR_CUDA;
  if (p->batch == 0 || p->total_q == 0) return PAGED_ATTN_OK;
  const int Hq = p->num_qo_heads, Hkv = p->num_kv_heads, G = Hq / Hkv, D = p->head_dim;
  const int ps = p->page_size;
  const int causal = p->mask_type == PAGED_ATTN_MASK_CAUSAL;
  int* n_tiles = at<int>(ws, s.n_tiles);
  TileRec* tmp = at<TileRec>(ws, s.tmp);
  TileRec* sorted = at<TileRec>(ws, s.sorted);
  launch_prefill_tiles(qo_indptr, 0, seq_lens, p->batch, Hkv, s.tile_tokens, causal,
                       p->window_left, s.capacity, at<int>(ws, s.tile_off), n_tiles, tmp, status,
                       st);
  launch_tile_sort(tmp, sorted, n_tiles, 0, s.capacity, s.max_cost, at<int>(ws, s.hist),
                   at<int>(ws, s.offs), st);
  const float scale = p->sm_scale > 0.f ? p->sm_scale : 1.0f / std::sqrt(static_cast<float>(D));
  AttnLaunch a{};
  // keys per page piece of a copy: 128-key tiles; the D = 256 kernel copies V 32 keys at a time
  const int RK = page_piece_rows(ps, kKvTile);
  const int RV = page_piece_rows(ps, D == 256 ? 32 : kKvTile);
  const long long pool_rows = static_cast<long long>(p->num_pages) * Hkv * ps;
  if (!encode_q_map(&a.qmap, q, p->total_q, Hq, D, G, sub_tile_tokens(G)) ||
      !encode_rows_map(&a.kmap, kc, pool_rows, D, RK) ||
      !encode_rows_map(&a.vmap, vc, pool_rows, D, RV))
    return PAGED_ATTN_ERR_CUDA;
  a.tiles = sorted;
  a.n_tiles = n_tiles;
  a.capacity = s.capacity;
  a.pt = block_tables;
  a.pt_indptr = nullptr;
  a.pt_stride = p->max_pages_per_request;
  a.seq_lens = seq_lens;
  a.qo_indptr = qo_indptr;
  a.q_len = 0;
  a.valid_bits = nullptr;
  a.valid_words = 0;
  a.block_sparse = 0;
  a.block_indices = nullptr;
  a.kv_block_size = kKvTile;
  a.out = out;
  a.out_dtype = p->out_dtype;
  a.lse = lse;
  a.status = status;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.D = D;
  a.page_size = ps;
  a.page_rows = Hkv * ps;
  a.k_head_off = 0;
  a.v_head_off = 0;
  a.num_pages = p->num_pages;
  a.causal = causal;
  a.window_left = p->window_left;
  a.scale_log2 = scale * kLog2e;
  a.out_scale = p->output_scale;
  void* tok;
  timer_begin(st, &tok);
  const int rc = D == 256 ? launch_attn256(a, st) : launch_attn(a, st);
  timer_end(st, tok);
  if (rc == -2) return PAGED_ATTN_ERR_UNSUPPORTED;
  return rc == 0 ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

size_t paged_decode_workspace_size(const paged_decode_params* p) {
  if (!decode_params_ok(p)) return 0;
  return decode_layout(p).total;
}

int paged_decode_split_chunk(const paged_decode_params* p) {
  if (!decode_params_ok(p)) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  return decode_chunk(p);
}

int paged_decode_run(const paged_decode_params* p, const void* query, const void* k,
                     const void* v, const int32_t* kv_indptr, const int32_t* kv_indices,
                     const int32_t* seq_lens, const int32_t* qo_indptr, void* out, float* lse,
                     void* ws, size_t ws_bytes, void* stream) {
  if (!decode_params_ok(p) || !query || !k || !kv_indptr || !kv_indices || !seq_lens || !out)
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (!p->combined_cache && !v) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (decode_packed(p) != (qo_indptr != nullptr)) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  if (!aligned16(query) || !aligned16(k) || (v && !aligned16(v)) || !aligned16(out))
    return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const DecodeLayout s = decode_layout(p);
  if (!ws || ws_bytes < s.total) return PAGED_ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, s.status);
  // the split route's planner clears the status word itself
  if ((s.tiled || p->batch == 0 || s.q_rows == 0) &&
      cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), st) != cudaSuccess)
    return PAGED_ATTN_ERR_CUDA;
  if (p->batch == 0 || s.q_rows == 0) return PAGED_ATTN_OK;
  if (s.tiled)
    return decode_run_tiled(p, s, query, k, v, kv_indptr, kv_indices, seq_lens, qo_indptr, out,
                            lse, ws, st);
  const int Hkv = p->num_kv_heads, ps = p->page_size, D = p->head_dim;
  const int G = p->num_qo_heads / Hkv;
  int* split_off = at<int>(ws, s.split_off);
  SplitItem* items = at<SplitItem>(ws, s.items);
  int* counters = at<int>(ws, s.counters);
  const int q_len = qo_indptr ? 0 : s.q_per_item;
  int* order = at<int>(ws, s.order);
  launch_decode_plan(seq_lens, qo_indptr, q_len, s.q_per_item, s.q_rows, p->batch, Hkv, s.chunk,
                     p->window_left, s.max_splits, split_off, items, order, counters, status, st);
  const int R = page_piece_rows(ps, 64);
  const long long pool_rows = static_cast<long long>(p->num_pages) * (p->combined_cache ? 2 : 1) *
                              Hkv * ps;
  CUtensorMap kmap, vmap, qmap;
  if (!encode_rows_map(&kmap, k, pool_rows, D, R) ||
      !encode_rows_map(&vmap, p->combined_cache ? k : v, pool_rows, D, R) ||
      !encode_q_map(&qmap, query, s.q_rows, p->num_qo_heads, D, G, s.q_per_item))
    return PAGED_ATTN_ERR_CUDA;
  const float scale =
      p->bmm1_scale > 0.f ? p->bmm1_scale : 1.0f / std::sqrt(static_cast<float>(D));
  DecodeLaunch a{};
  a.kmap = &kmap;
  a.vmap = &vmap;
  a.qmap = &qmap;
  a.counters = counters;
  a.work_counter = counters + static_cast<long long>(p->batch) * Hkv;
  a.qo_indptr = qo_indptr;
  a.q_len = q_len;
  a.q_rows = s.q_rows;
  a.rows = s.rows;
  a.nrb = s.rows <= 16 ? 1 : (s.rows <= 32 ? 2 : 4);
  a.causal = p->mask_type == PAGED_ATTN_MASK_CAUSAL;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.seq_lens = seq_lens;
  a.split_offset = split_off;
  a.items = items;
  a.order = order;
  a.part_o = at<float>(ws, s.part_o);
  a.part_lse = at<float>(ws, s.part_lse);
  a.out = out;
  a.out_dtype = p->out_dtype;
  a.lse = lse;
  a.status = status;
  a.B = p->batch;
  a.Hq = p->num_qo_heads;
  a.Hkv = Hkv;
  a.D = D;
  a.page_size = ps;
  a.page_rows = (p->combined_cache ? 2 : 1) * Hkv * ps;
  a.k_head_off = 0;
  a.v_head_off = p->combined_cache ? Hkv * ps : 0;
  a.num_pages = p->num_pages;
  a.capacity = s.capacity;
  a.scale_log2 = scale * kLog2e;
  a.out_scale = p->bmm2_scale;
  a.window_left = p->window_left;
  a.timer_token = nullptr;
  return launch_decode(a, st) == 0 ? PAGED_ATTN_OK : PAGED_ATTN_ERR_CUDA;
}

int paged_attn_plan_layout_of(const paged_attn_params* p, paged_attn_plan_layout* o) {
  if (!sparse_params_ok(p) || !o) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const SparseLayout s = sparse_layout(p);
  *o = paged_attn_plan_layout{};
  o->status_offset = s.status;
  if (p->form == PAGED_ATTN_FORM_BSR) {
    o->tiles_offset = s.sorted;
    o->tiles_capacity = s.capacity;
    o->tile_tokens = s.tile_tokens;
  } else {
    o->indptr_offset = s.indptr;
    o->indices_offset = s.indices;
    o->indices_capacity = s.bitmap_capacity;
  }
  return PAGED_ATTN_OK;
}

int paged_prefill_plan_layout_of(const paged_prefill_params* p, paged_attn_plan_layout* o) {
  if (!prefill_params_ok(p) || !o) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const PrefillLayout s = prefill_layout(p);
  *o = paged_attn_plan_layout{};
  o->status_offset = s.status;
  o->tiles_offset = s.sorted;
  o->tiles_capacity = s.capacity;
  o->count_offset = s.n_tiles;
  o->tile_tokens = s.tile_tokens;
  return PAGED_ATTN_OK;
}

int paged_decode_plan_layout_of(const paged_decode_params* p, paged_attn_plan_layout* o) {
  if (!decode_params_ok(p) || !o) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const DecodeLayout s = decode_layout(p);
  *o = paged_attn_plan_layout{};
  o->status_offset = s.status;
  if (s.tiled) {
    o->tiles_offset = s.sorted;
    o->tiles_capacity = s.capacity;
    o->count_offset = s.n_tiles;
    o->tile_tokens = s.tile_tokens;
  } else {
    o->split_offset_offset = s.split_off;
    o->items_offset = s.items;
    o->items_capacity = s.capacity;
    o->order_offset = s.order;
    o->split_chunk = s.chunk;
  }
  return PAGED_ATTN_OK;
}

int paged_attn_kernel_timer(int enable) {
  std::lock_guard<std::mutex> lk(g_timer.mu);
  g_timer.on = enable != 0;
  if (enable) g_timer.used = 0;
  return PAGED_ATTN_OK;
}

int paged_attn_kernel_timer_read(double* total_ms, int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_timer.mu);
  double tot = 0.0;
  for (size_t i = 0; i < g_timer.used; ++i) {
    auto& pr = g_timer.pairs[i];
    if (cudaEventSynchronize(pr.second) != cudaSuccess) return PAGED_ATTN_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, pr.first, pr.second) != cudaSuccess) return PAGED_ATTN_ERR_CUDA;
    tot += ms;
  }
  if (total_ms) *total_ms = tot;
  if (launches) *launches = static_cast<int64_t>(g_timer.used);
  return PAGED_ATTN_OK;
}

int64_t paged_attn_launch_count(void) { return g_launches.load(); }

int paged_attn_workspace_status(const void* ws, void* stream, uint32_t* raw) {
  if (!ws) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return PAGED_ATTN_ERR_CUDA;
  if (raw) *raw = word;
  if (word & kErrTimeout) return PAGED_ATTN_ERR_TIMEOUT;
  if (word & kErrCapacity) return PAGED_ATTN_ERR_CAPACITY;
  if (word & kErrMetadata) return PAGED_ATTN_ERR_METADATA;
  return PAGED_ATTN_OK;
}


size_t paged_sage_workspace_size(const paged_sage_params* p) {
  if (!sage_params_ok(p)) return 0;
  return sage_layout(p).total;
}

int paged_sage_run(const paged_sage_params* p, const int8_t* q_int8, const int8_t* k_int8,
                   const uint8_t* v_fp8, const float* q_scale, const float* k_scale,
                   const float* v_scale, const int32_t* idx, const int32_t* nums,
                   const int32_t* block_sizes, void* out, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!sage_params_ok(p) || !out || !aligned16(out)) return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  const SageLayout g = sage_layout(p);
  // every argument is checked before anything is enqueued; the inputs only matter when there
  // are rows and keys
  if (g.BH > 0 && p->q_len > 0 && g.NB > 0) {
    if (!q_int8 || !k_int8 || !v_fp8 || !q_scale || !k_scale || !v_scale ||
        (p->capacity > 0 && !idx) || (p->block_sizes_rank > 0 && !block_sizes))
      return PAGED_ATTN_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_int8) || !aligned16(k_int8) || (reinterpret_cast<uintptr_t>(v_fp8) & 3u))
      return PAGED_ATTN_ERR_INVALID_ARGUMENT;
  }
  if (!ws || ws_bytes < g.total) return PAGED_ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, g.s.status);
  if (cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), st) != cudaSuccess) return PAGED_ATTN_ERR_CUDA;
  if (g.BH == 0 || p->q_len == 0) return PAGED_ATTN_OK;
  if (g.NB == 0) {                               // no keys: every row is empty, O = 0
    return cudaMemsetAsync(out, 0, static_cast<size_t>(g.BH) * p->q_len * 128 * 2, st) ==
                   cudaSuccess
               ? PAGED_ATTN_OK
               : PAGED_ATTN_ERR_CUDA;
  }
  SagePrepare sp{};
  sp.q_int8 = q_int8;
  sp.k_int8 = k_int8;
  sp.v_fp8 = v_fp8;
  sp.q_bf16 = at<__nv_bfloat16>(ws, g.q_bf16);
  sp.k_bf16 = at<__nv_bfloat16>(ws, g.k_bf16);
  sp.v_bf16 = at<__nv_bfloat16>(ws, g.v_bf16);
  sp.idx = idx;
  sp.nums = p->uniform_block_count ? nullptr : nums;
  sp.uniform = p->block_sparse_num;
  sp.cap = p->capacity;
  sp.block_sizes = block_sizes;
  sp.bs_rank = p->block_sizes_rank;
  sp.B = p->batch;
  sp.H = p->num_heads;
  sp.Sq = p->q_len;
  sp.Sk = p->kv_len;
  sp.NB = g.NB;
  sp.QB = g.QB;
  sp.counts = at<int>(ws, g.counts);
  sp.block_indptr = at<int>(ws, g.block_indptr);
  sp.block_indices = at<int>(ws, g.block_indices);
  sp.kv_indptr = at<int>(ws, g.kv_indptr);
  sp.kv_indices = at<int>(ws, g.kv_indices);
  sp.seq_lens = at<int>(ws, g.seq_lens);
  sp.valid_bits = at<uint32_t>(ws, g.valid_bits);
  sp.status = status;
  launch_sage_prepare(sp, st);
  // the block-sparse plan of the (b, h) requests
  const SparseLayout& s = g.s;
  launch_bsr_tiles(sp.block_indptr, g.BH, 1, p->q_len, 64, s.tile_tokens, at<TileRec>(ws, s.tmp), st);
  launch_tile_sort(at<TileRec>(ws, s.tmp), at<TileRec>(ws, s.sorted), nullptr, s.capacity,
                   s.capacity, s.max_cost, at<int>(ws, s.hist), at<int>(ws, s.offs), st);
  paged_attn_meta m{};
  m.kv_indptr_dev = sp.kv_indptr;
  m.kv_indices_dev = sp.kv_indices;
  m.block_indptr_dev = sp.block_indptr;
  m.block_indices_dev = sp.block_indices;
  m.seq_lens_kv_dev = sp.seq_lens;
  m.kv_valid_bits_dev = sp.valid_bits;
  ScaleSet sc{q_scale, k_scale, v_scale, 32, g.QG, g.NB, 128};
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt(128.0f);
  return bsr_launch(&g.bsr, &m, s, sp.q_bf16, sp.k_bf16, sp.v_bf16, out, nullptr, ws, status,
                    scale, &sc, st);
}

}  // extern "C"
