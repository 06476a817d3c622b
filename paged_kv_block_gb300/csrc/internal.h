// Declarations shared by the translation units of libpagedattn (not part of the ABI).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pa {

// Launch `kernel` with programmatic stream serialization: it may start while the previous
// kernel of the stream still runs (once every CTA of that kernel has called
// grid_launch_dependents() or exited), so its launch and prologue overlap that kernel's
// tail.  The kernel must call grid_dependency_wait() before it reads anything the previous
// kernels wrote.  After a copy or a memset the launch is an ordinary one.
template <typename... Params, typename... Args>
inline cudaError_t launch_after_previous(void (*kernel)(Params...), dim3 grid, dim3 block,
                                         size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// A kernel's dynamic shared memory limit is set per device, so it is set once on every device
// the library launches it on: `done` holds one bit per device index below 64 (devices past
// that are set on every launch).
template <typename Kernel>
inline bool kernel_smem_ready(Kernel* kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  if (bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

// SM count of the current device, looked up once per device index below 64; 0 on failure.
inline int current_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool cacheable = dev >= 0 && dev < 64;
  if (cacheable && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cacheable) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Tile record written by the planner and read by the prefill / block-sparse kernel:
// b, g, tok0, ntok, kv_begin, kv_end, q_row0, 0.
struct TileRec {
  int b, g, tok0, ntok, kv_begin, kv_end, q_row0, pad;
};

// Split-KV work item of the decode kernel.
struct SplitItem {
  int b, g, kv_begin, kv_end;
};

constexpr int kSortChunk = 1024;     // records per counting-sort chunk
constexpr int kMaxSortCost = 4095;   // costs are capped at this value for ordering
constexpr int kKvTile = 128;         // keys per KV tile of the prefill kernel
constexpr int kMTileRows = 128;      // rows per Q sub-tile (one TMEM lane per row)

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// Keys per TMA page piece.  A piece is a run of consecutive keys inside one page, and the
// pieces of a `span`-key stage or sub-chunk tile it in order (span is a power of two).  A
// power-of-two page size gives min(page_size, span); any other multiple of 8 gives 8-key
// pieces, which never straddle a page boundary because page boundaries are multiples of 8.
__host__ __device__ inline int page_piece_rows(int page_size, int span) {
  if ((page_size & (page_size - 1)) != 0) return 8;
  return page_size < span ? page_size : span;
}

#ifdef __CUDACC__
// Work-tile claims of the persistent tensor-core kernels: status[2] counts the tiles claimed
// beyond the first one of every CTA, status[3] the CTAs that have finished; the last CTA of a
// launch to finish sets both back to zero, so every launch (and every graph replay) starts
// from zero.  Called once per CTA, by one thread, on every exit path.
__device__ __forceinline__ void claims_done(uint32_t* status) {
  __threadfence();
  if (atomicAdd(status + 3, 1u) == gridDim.x - 1) {
    atomicExch(status + 2, 0u);
    atomicExch(status + 3, 0u);
  }
}
#endif

// Tokens per Q sub-tile: floor(128 / G); a CTA holds two sub-tiles.
inline int sub_tile_tokens(int G) { return kMTileRows / G; }
inline int cta_tile_tokens(int G) { return 2 * sub_tile_tokens(G); }

// ---- planner launchers (planner.cu) ----------------------------------------------------
// All write the status word on capacity problems; none synchronises the host.
void launch_bsr_tiles(const int* block_indptr, int B, int Hkv, int Sq, int qbs, int tile_tokens,
                      TileRec* tmp, cudaStream_t st);
// A block-sparse plan small enough for one CTA (capacity and rows within one sort chunk):
// launch_bsr_plan_small then writes the sorted records directly and clears the 4 status
// words, in place of launch_bsr_tiles + launch_tile_sort.
bool bsr_plan_is_small(int B, int Hkv, int Sq, int qbs, int capacity, int max_cost);
void launch_bsr_plan_small(const int* block_indptr, int B, int Hkv, int Sq, int qbs,
                           int tile_tokens, int capacity, int max_cost, TileRec* out,
                           uint32_t* status, cudaStream_t st);
// Request b has qo_indptr[b + 1] - qo_indptr[b] queries at rows from qo_indptr[b], or
// (qo_indptr == nullptr) q_len queries at rows from b * q_len.
void launch_prefill_tiles(const int* qo_indptr, int q_len, const int* seq_lens, int B, int Hkv,
                          int tile_tokens, int causal, int window_left, int capacity,
                          int* tile_offsets, int* n_tiles, TileRec* tmp, uint32_t* status,
                          cudaStream_t st);
// Stable sort of n records (n_dev: device count, or nullptr to use n_static) by
// min(kv_end - kv_begin, max_cost) descending.
void launch_tile_sort(const TileRec* in, TileRec* out, const int* n_dev, int n_static,
                      int capacity, int max_cost, int* hist, int* offs, cudaStream_t st);
size_t tile_sort_scratch_ints(int capacity, int max_cost);

void launch_bitmap_plan(const uint8_t* sel, const int* lo, const int* hi, const int* bfirst,
                        const int* blast, int T, int NB, long long capacity, int* indptr,
                        int* indices, uint32_t* status, cudaStream_t st);

// Indexed form: per-query CSR from index rows [T, K] (caller order; negative entries unused;
// ids >= NB dropped and reported as kErrMetadata; ids whose span misses [lo, hi] dropped).
void launch_indexed_plan(const int* idx, int K, const int* lo, const int* hi, const int* bfirst,
                         const int* blast, int T, int NB, long long capacity, int* indptr,
                         int* indices, uint32_t* status, cudaStream_t st);

// Split-KV work list, its claim order (items by size class, largest first; stable), and
// zeroed work / merge counters (B * Hkv + 1 ints).  Request b has
// qo_indptr[b + 1] - qo_indptr[b] queries (qo_indptr != nullptr) or q_len; packed offsets
// that break their contract (start 0, steps in [1, max_q], end total_q) set kErrMetadata.
void launch_decode_plan(const int* seq_lens, const int* qo_indptr, int q_len, int max_q,
                        int total_q, int B, int Hkv, int chunk, int window_left, int max_splits,
                        int* split_offset, SplitItem* items, int* order, int* counters,
                        uint32_t* status, cudaStream_t st);

// Keys per sub-chunk of a 128-key KV tile: the largest of 128, 64 or kv_block_size that
// divides kv_block_size (dense tiles use 128).
inline int attn_sub_chunk(int kv_block_size, bool block_sparse) {
  if (!block_sparse) return kKvTile;
  if (kv_block_size % kKvTile == 0) return kKvTile;
  if (kv_block_size % 64 == 0) return 64;
  return kv_block_size;
}

// ---- kernels launchers ------------------------------------------------------------------
struct DecodeLaunch {
  const CUtensorMap* kmap;   // host copies, passed by value to the kernel
  const CUtensorMap* vmap;
  const CUtensorMap* qmap;   // query [q_rows, Hq, D], box 64 x G heads x rows / G queries
  int* work_counter;         // next work item (zeroed by the planner)
  int* counters;             // finished splits per (request, KV head) (zeroed by the planner)
  const int* qo_indptr;      // packed queries: request b owns query rows qo_indptr[b]..;
                             // nullptr: q_len queries per request at rows b * q_len..
  int q_len;
  int q_rows;                // rows of query / out: writes outside [0, q_rows) are skipped
  int rows;                  // M = G x queries per item (<= 64): rows of one work item
  int nrb;                   // 16-row blocks of an item: 1 (M <= 16), 2 (<= 32) or 4
  int causal;                // keys after a query's position are masked
  const int* kv_indptr;
  const int* kv_indices;
  const int* seq_lens;
  const int* split_offset;
  const SplitItem* items;
  const int* order;          // claim order: the k-th claimed item is items[order[k]]
  float* part_o;             // [items, M, D]
  float* part_lse;           // [items, M]
  void* out;                 // [q_rows, Hq, D] of out_dtype
  int out_dtype;             // kOutBf16, kOutF16 or kOutF32
  float* lse;                // [q_rows, Hq] or nullptr
  uint32_t* status;
  int B, Hq, Hkv, D, page_size, page_rows, k_head_off, v_head_off, num_pages;
  int capacity;              // launched work items
  float scale_log2, out_scale;
  int window_left;
  void* timer_token;
};
int launch_decode(const DecodeLaunch& a, cudaStream_t st);

// Benchmark hooks (api.cu): count kernel launches; bracket the main kernel with events.
void count_launches(int n);
void timer_begin(cudaStream_t st, void** token);
void timer_end(cudaStream_t st, void* token);

struct AttnLaunch {
  CUtensorMap qmap, kmap, vmap;
  const TileRec* tiles;
  const int* n_tiles;        // device count (nullptr: all `capacity` tiles are live)
  int capacity;
  // page table: CSR (pt_indptr != nullptr) or row-strided (pt_stride)
  const int* pt;
  const int* pt_indptr;
  int pt_stride;
  const int* seq_lens;
  const int* qo_indptr;      // packed-Q form: nq of request b; nullptr -> fixed q_len
  int q_len;
  const uint32_t* valid_bits;
  int valid_words;
  int block_sparse;          // 1: KV tiles walk block_indices; 0: dense KV tile ranges
  const int* block_indices;  // BSR form (may be null when no row lists a block)
  int kv_block_size;
  void* out;                 // rows of out_dtype
  int out_dtype;             // kOutBf16, kOutF16 or kOutF32
  float* lse;
  uint32_t* status;
  int Hq, Hkv, G, D, page_size, page_rows, k_head_off, v_head_off, num_pages;
  int causal, window_left;
  float scale_log2, out_scale;
  // Prequantized form (all nullptr otherwise): score scale q_scale[b * q_scale_stride +
  // token / q_scale_group] * k_scale[b * k_scale_stride + key / kv_block_size], output column
  // d scaled by v_scale[b * v_scale_stride + d]; every scale positive.
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int q_scale_group, q_scale_stride, k_scale_stride, v_scale_stride;
};
int launch_attn(const AttnLaunch& a, cudaStream_t st);
// Dense prefill tiles of head dimension 256 (one 128-row sub-tile per planner tile).
int launch_attn256(const AttnLaunch& a, cudaStream_t st);

// ---- prequantized block-sparse form (sage.cu) ------------------------------------------------
// Exact bf16 copies of the int8 Q/K and FP8 V, and the block-sparse metadata of the (b, h)
// requests: identity pages of 64 keys, lengths, validity bits from the block sizes, BSR rows
// from the index rows (ids outside [0, NB) dropped and reported).
struct SagePrepare {
  const int8_t* q_int8;          // [B, H, Sq, 128]
  const int8_t* k_int8;          // [B, H, Sk, 128]
  const uint8_t* v_fp8;          // [B, H, 128, NB * 64]
  __nv_bfloat16* q_bf16;         // [B * H, Sq, 128]
  __nv_bfloat16* k_bf16;         // [B * H * NB pages, 64, 128]
  __nv_bfloat16* v_bf16;         // [B * H * NB pages, 64, 128]
  const int* idx;                // [B, H, QB, cap]
  const int* nums;               // [B, H, QB] or nullptr (uniform)
  int uniform, cap;
  const int* block_sizes;        // rank bs_rank: 0 none, 1 [NB], 2 [B, NB], 3 [B, H, NB]
  int bs_rank;
  int B, H, Sq, Sk, NB, QB;
  int* counts;                   // [B * H * QB] scratch
  int* block_indptr;             // [B * H, QB + 1]
  int* block_indices;            // [B * H * QB * cap]
  int* kv_indptr;                // [B * H + 1]
  int* kv_indices;               // [B * H * NB]
  int* seq_lens;                 // [B * H]
  uint32_t* valid_bits;          // [B * H, 2 * NB]
  uint32_t* status;
};
void launch_sage_prepare(const SagePrepare& s, cudaStream_t st);

// ---- tensor maps (api.cu) -----------------------------------------------------------------
bool encode_rows_map(CUtensorMap* map, const void* base, long long rows, int D, int box_rows);
bool encode_q_map(CUtensorMap* map, const void* base, long long rows, int Hq, int D,
                  int box_heads, int box_tokens);
// [tokens, Hkv, D] bf16 with box = 4 tokens x 2 KV heads x all D / 64 column chunks: one
// 4-token block of a KV-head pair lands as D / 64 8-row, 128-byte-swizzled atoms.
bool encode_block_pair_map(CUtensorMap* map, const void* base, long long tokens, int Hkv, int D);

}  // namespace pa
