/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged-KV attention forward library.
 *
 * One shared library (libpagedattn.so) exposes the forward attention hot path over a
 * paged KV cache:
 *   - block-sparse (BSR) attention over a CSR-paged cache, and per-query block-bitmap
 *     attention over packed K/V   -> paged_attn_plan / paged_attn_run
 *   - packed-Q dense / causal / sliding-window prefill over separate HND page pools with
 *     a row-strided page table   -> paged_prefill_run
 *   - decode over a CSR-paged cache (one, SQ fixed or packed queries per request) with
 *     split-KV partials and a merge -> paged_decode_run
 *   - block-sparse attention on prequantized inputs (int8 Q/K, FP8 E4M3 V, fp32 scales)
 *     -> paged_sage_run
 * The bitmap form also takes its selection as index rows (PAGED_ATTN_FORM_INDEXED).  The
 * operations are those of the FlashInfer API pages
 *   [BSA]  flashinfer.attention.prims_ts.block_sparse_attention_with_paged_kv_cache
 *   [PRE]  flashinfer.attention.prims_ts.batch_prefill_with_paged_kv_cache
 *   [QSA]  flashinfer.qsa.qsa_forward
 *   [DEC]  flashinfer.attention.prims_ts.prims_ts_batch_decode_with_kv_cache
 *   [SAGE] flashinfer.cute_dsl.sparse.bsa_attn_sm120.bsa_attn_sm120_blk64_sage_fwd
 * cited below by tag and by the section of the page (signature, a named parameter, or the
 * notes).
 *
 * Conventions for every entry point
 *   - Pointers named *_dev are device pointers; pointers named *_host are host pointers.
 *     All memory is owned by the caller; the run path allocates nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *     device work is enqueued on it; no entry point of the run path synchronises the host
 *     or copies device metadata back to the host, so a planned run can be captured in a
 *     CUDA graph ([BSA] summary; [DEC] notes, which rule out any read-back of device
 *     metadata to the host during a launch).
 *   - Element types: Q, K and V are bf16 (int8 and FP8 E4M3 bytes in the prequantized
 *     form); outputs are bf16, or fp16 / fp32 where out_dtype selects them (prefill and
 *     decode); page tables, lengths and offsets are int32; kv_valid_bits is uint32; LSE and
 *     fp32 outputs are float.
 *   - Q, K, V and output base pointers must be 16-byte aligned (PAGED_ATTN_ERR_INVALID_ARGUMENT
 *     otherwise; the FP8 V of the prequantized form needs 4 bytes).
 *   - Return value: PAGED_ATTN_OK or a negative PAGED_ATTN_ERR_* code.  Argument checks
 *     happen on the host before anything is enqueued.  Device-side faults of the contract
 *     that the kernels detect (a wait that timed out, a plan that outgrew its capacity) are
 *     OR-ed into a status word inside the workspace; read it with
 *     paged_attn_workspace_status().
 *   - The GQA group is G = num_qo_heads / num_kv_heads; query head h reads KV head h / G.
 *   - Query position: query i of a request with nq queries and L keys is at position
 *     L - nq + i (queries are the last nq positions).  The causal mask keeps keys j <= that
 *     position; window_left = w >= 0 also drops keys j < position - w.
 *   - A query row that sees no key gets an output of exactly 0 and an LSE of -inf
 *     ([QSA] notes state this for the bitmap form; the library applies it to every form).
 *   - LSE is the natural logarithm of sum_j exp(sm_scale * q.k_j) over the visible keys.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------ */
#define PAGED_ATTN_OK 0
#define PAGED_ATTN_ERR_INVALID_ARGUMENT (-1) /* null pointer, bad size or value          */
#define PAGED_ATTN_ERR_UNSUPPORTED (-2)      /* valid per the pages but not built here   */
#define PAGED_ATTN_ERR_WORKSPACE (-3)        /* workspace missing or too small           */
#define PAGED_ATTN_ERR_CUDA (-4)             /* a CUDA runtime/driver call failed        */
#define PAGED_ATTN_ERR_TIMEOUT (-5)          /* status word: a device wait timed out      */
#define PAGED_ATTN_ERR_METADATA (-6)         /* validation found metadata off-contract   */
#define PAGED_ATTN_ERR_CAPACITY (-7)         /* status word: plan exceeded its capacity   */

#define PAGED_ATTN_MASK_DENSE 0
#define PAGED_ATTN_MASK_CAUSAL 1

/* Output element types ([PRE] and [DEC] out_dtype).  Inputs are bf16; the normalised
 * fp32 result is rounded to nearest-even into the output type. */
#define PAGED_ATTN_DTYPE_BF16 0
#define PAGED_ATTN_DTYPE_FP16 1
#define PAGED_ATTN_DTYPE_FP32 2

#define PAGED_ATTN_FORM_BSR 0    /* [BSA]: BSR rows per (request, KV head, query block) */
#define PAGED_ATTN_FORM_BITMAP 1 /* [QSA]: uint8 block bitmap per packed query token    */
#define PAGED_ATTN_FORM_INDEXED 2 /* [QSA] notes (qsa_indexed_forward): each packed query
                                    token's selected global block ids as an index row  */

/* Static description of a sparse launch (everything the plan's size depends on).
 * [BSA] signature and parameters; [QSA] signature and parameters. */
typedef struct paged_attn_params {
  int form;              /* PAGED_ATTN_FORM_*                                            */
  int batch;             /* BSR: B requests                                              */
  int q_len;             /* BSR: Sq queries per request; BITMAP: T packed tokens          */
  int num_qo_heads;      /* Hq                                                           */
  int num_kv_heads;      /* Hkv; Hq % Hkv == 0                                           */
  int head_dim;          /* D: 128 (BSR); 256 (BITMAP)                                   */
  /* BSR only */
  int page_size;         /* tokens per page: a multiple of 8, at most 128                */
  int num_pages;         /* P: pages in the pool                                         */
  int combined_cache;    /* 1: one cache [P, 2, Hkv, page_size, D] (axis 1: 0 = K, 1 = V);
                            0: separate K and V pools [P, Hkv, page_size, D]             */
  int q_block_size;      /* queries per BSR row; q_block_size * G % 8 == 0 ([BSA])      */
  int kv_block_size;     /* keys per BSR block id: 8, 16, 32 or a multiple of 64 ([BSA])*/
  int max_seq_len_kv;    /* static bound on seq_lens_kv, used for planning ([BSA])        */
  int mask_type;         /* PAGED_ATTN_MASK_DENSE or _CAUSAL, inside each block          */
  int has_valid_bits;    /* 1: kv_valid_bits_dev is given                                */
  /* BITMAP and INDEXED */
  int num_blocks;        /* NB: columns of sel_blocks; blocks in block_first/last        */
  int block_size;        /* tokens per block: must be 4 ([QSA] block_size)               */
  int max_blocks_per_query; /* plan capacity: selected blocks per query on average over
                               the launch (0 = NB for BITMAP, index_width for INDEXED)   */
  float sm_scale;        /* softmax scale; <= 0 selects 1/sqrt(D) ([BSA] sm_scale)        */
  /* INDEXED only */
  int index_width;       /* K: entries per index row of sel_indices                      */
} paged_attn_params;

/* Device metadata of a sparse launch.  Unused pointers may be NULL.  Layouts follow the
 * pages' tensor contracts exactly; every array is contiguous. */
typedef struct paged_attn_meta {
  /* BSR ([BSA] parameters) */
  const int32_t* kv_indptr_dev;      /* [B + 1] offsets into kv_indices                   */
  const int32_t* kv_indices_dev;     /* physical page ids; request b owns
                                        kv_indices[kv_indptr[b] : kv_indptr[b + 1]]       */
  const int32_t* block_indptr_dev;   /* [B, Hkv, ceil(Sq / q_block_size) + 1]             */
  const int32_t* block_indices_dev;  /* logical KV-block ids of each BSR row (distinct)    */
  const int32_t* seq_lens_kv_dev;    /* [B] live keys per request                         */
  const uint32_t* kv_valid_bits_dev; /* [B, ceil(max_seq_len_kv / 32)]: bit (j & 31) of
                                        word (j >> 5) is 1 for a live token (NULL = all)  */
  /* BITMAP ([QSA] parameters) */
  const uint8_t* sel_blocks_dev;     /* [T, NB]; nonzero selects global block g           */
  const int32_t* lo_dev;             /* [T] inclusive first visible key token             */
  const int32_t* hi_dev;             /* [T] inclusive last visible key token              */
  const int32_t* blk_base_dev;       /* [T] first global block of the query's sequence    */
  const int32_t* tok_base_dev;       /* [T] first token of the query's sequence           */
  const int32_t* block_first_dev;    /* [NB] inclusive token span of each block, in       */
  const int32_t* block_last_dev;     /* [NB] increasing order                              */
  /* INDEXED (the [QSA] notes' indexed entry point; the pages give no signature): lo, hi,
   * block_first and block_last as above, plus */
  const int32_t* sel_indices_dev;    /* [T, K]: row t lists the global block ids query t
                                        selects, distinct, in any order; negative entries
                                        are unused; ids >= NB break the contract (dropped,
                                        metadata status bit)                              */
} paged_attn_meta;

/* Workspace bytes needed by paged_attn_plan + paged_attn_run for these static params
 * (0 on invalid params).  The workspace holds the status word and the plan. */
size_t paged_attn_workspace_size(const paged_attn_params* params);

/* Host-side validation of BSR metadata, the analogue of the synchronous checks that the
 * [BSA] convenience entry point makes on the page table and the block lists before it runs
 * ([BSA] summary).
 * All pointers are HOST copies.  Checks: kv_indptr starts at 0, is non-decreasing and
 * ends at num_kv_indices; every request owns ceil(len / page_size) pages; every live page
 * id is in [0, num_pages); 0 <= len <= max_seq_len_kv; block_indptr rows are
 * non-decreasing and stay inside [0, num_block_indices]; block ids are distinct within a
 * row and below ceil(max_seq_len_kv / kv_block_size).  Returns PAGED_ATTN_OK or
 * PAGED_ATTN_ERR_METADATA (first offending item written to *bad_index when non-NULL). */
int paged_attn_validate_bsr(const paged_attn_params* params, const int32_t* kv_indptr_host,
                            const int32_t* kv_indices_host, int64_t num_kv_indices,
                            const int32_t* block_indptr_host,
                            const int32_t* block_indices_host, int64_t num_block_indices,
                            const int32_t* seq_lens_kv_host, int64_t* bad_index);

/* Build the work plan on the device ([BSA] summary: plan, then run).
 *   BSR:    a list of M-tiles (<= 256 rows of (token, head-in-group)), each with the
 *           block_indices slice of its BSR row, sorted by block count (largest first).
 *   BITMAP: a per-query CSR of selected global block ids meeting [lo, hi] (ascending).
 *   INDEXED: the same CSR from the index rows: each row's ids in [0, NB) whose span meets
 *           [lo, hi], in the row's order (no [T, NB] scan).
 * Reads only the metadata; writes only the workspace.  Clears the status word. */
int paged_attn_plan(const paged_attn_params* params, const paged_attn_meta* meta,
                    void* workspace_dev, size_t workspace_bytes, void* stream);

/* Run the planned launch.
 *   q_dev:   BSR [B, Sq, Hq, D]; BITMAP and INDEXED [T, Hq, D]                    ([BSA] q)
 *   k_dev:   BSR: K pool [P, Hkv, ps, D] or the combined cache [P, 2, Hkv, ps, D];
 *            BITMAP: k [T, Hkv, D]
 *   v_dev:   BSR: V pool [P, Hkv, ps, D] (NULL with a combined cache); BITMAP: v [T, Hkv, D]
 *   out_dev: bf16, same shape as q                                            ([BSA] out)
 *   out_fp32_dev: BITMAP only, optional fp32 copy of the output before the bf16 cast
 *   lse_dev: optional fp32 LSE; BSR [B, Sq, Hq]; BITMAP [Hq, T]             ([QSA] lse)
 * The metadata must be the one given to paged_attn_plan. */
int paged_attn_run(const paged_attn_params* params, const paged_attn_meta* meta,
                   const void* q_dev, const void* k_dev, const void* v_dev, void* out_dev,
                   float* out_fp32_dev, float* lse_dev, void* workspace_dev,
                   size_t workspace_bytes, void* stream);

/* ---- [PRE] packed-Q prefill ---------------------------------------------------------- */
typedef struct paged_prefill_params {
  int batch;            /* B                                                              */
  int total_q;          /* rows of q / out ([PRE] q: [total_q, Hq, D])                    */
  int num_qo_heads, num_kv_heads, head_dim; /* D = 128 or 256 ([PRE] notes)             */
  int page_size;        /* 16, 32, 64 or 128 ([PRE] summary)                              */
  int num_pages;        /* P                                                              */
  int max_pages_per_request; /* C: columns of block_tables ([PRE] block_tables [B, C])     */
  int mask_type;        /* PAGED_ATTN_MASK_*                                              */
  int window_left;      /* -1 = no window; >= 0 needs the causal mask ([DEC] notes)       */
  float sm_scale;       /* <= 0 selects 1/sqrt(D) ([PRE] sm_scale)                         */
  float output_scale;   /* multiplies the normalised output ([PRE] output_scale)           */
  int out_dtype;        /* PAGED_ATTN_DTYPE_* of out ([PRE] out_dtype; 0 = bf16)          */
} paged_prefill_params;

size_t paged_prefill_workspace_size(const paged_prefill_params* params);

/* Plan and run one packed-Q prefill launch.
 *   q_dev [total_q, Hq, D]; k_cache_dev, v_cache_dev [P, Hkv, page_size, D] (HND);
 *   qo_indptr_dev [B + 1] (request b owns rows qo_indptr[b] : qo_indptr[b + 1]);
 *   block_tables_dev [B, C] row-strided physical page ids; seq_lens_kv_dev [B];
 *   out_dev [total_q, Hq, D] of out_dtype; lse_dev [total_q, Hq] fp32 (optional).
 * Every request needs len_q <= len_kv under the causal mask and ceil(len_kv / page_size)
 * <= C.  Table entries past a request's live pages are never read. */
int paged_prefill_run(const paged_prefill_params* params, const void* q_dev,
                      const void* k_cache_dev, const void* v_cache_dev,
                      const int32_t* qo_indptr_dev, const int32_t* block_tables_dev,
                      const int32_t* seq_lens_kv_dev, void* out_dev, float* lse_dev,
                      void* workspace_dev, size_t workspace_bytes, void* stream);

/* ---- [DEC] decode with split-KV --------------------------------------------------------- */
typedef struct paged_decode_params {
  int batch;            /* B                                                              */
  int num_qo_heads, num_kv_heads, head_dim; /* D = 128; G = Hq / Hkv <= 16                */
  int page_size;        /* a multiple of 8, at most 128                                   */
  int num_pages;        /* P                                                              */
  int combined_cache;   /* 1: [P, 2, Hkv, ps, D]; 0: separate K and V pools                */
  int max_seq_len;      /* static bound on seq_lens, <= 2147483520 ([DEC] max_seq_len)   */
  int mask_type;        /* PAGED_ATTN_MASK_*; with one query both keep every live key     */
  int window_left;      /* -1 = no window; w >= 0 (causal) keeps keys j >= p - w for the
                           query at position p = len - nq + i                            */
  float bmm1_scale;     /* softmax scale; <= 0 selects 1/sqrt(D)                          */
  float bmm2_scale;     /* multiplies the normalised output ([DEC] bmm2_scale)             */
  int split_chunk;      /* keys per split-KV partition, a multiple of 128; 0 = automatic:
                           128 * max(1, B * Hkv * ceil(max_seq_len / 128) / (16 * SMs))     */
  /* Query layout ([DEC] seq_len_q, qo_indptr, max_seq_len_q).  Zero-initialised fields give
   * one query per request, query [B, Hq, D]. */
  int seq_len_q;        /* fixed form: SQ queries per request; SQ > 1 gives token-major
                           query / out [B, SQ, Hq, D] and LSE [B, SQ, Hq]                 */
  int max_seq_len_q;    /* > 0 selects the packed form: paged_decode_run takes qo_indptr,
                           query / out are [total_q, Hq, D], and every request has between
                           1 and max_seq_len_q queries (the static bound of [DEC])         */
  int total_q;          /* packed form: rows of query and out, = qo_indptr[B]              */
  int out_dtype;        /* PAGED_ATTN_DTYPE_* of out ([DEC] out_dtype; 0 = bf16)          */
} paged_decode_params;

/* Workspace bytes for the decode plan and the fp32 split partials. */
size_t paged_decode_workspace_size(const paged_decode_params* params);

/* The split chunk (keys) that paged_decode_run will use for these params on the current
 * device; a pure function of the static params and the SM count. */
int paged_decode_split_chunk(const paged_decode_params* params);

/* Plan (split-KV work list), run the partial kernel and merge ([DEC] signature).
 *   query_dev: [B, Hq, D] (one query per request), [B, SQ, Hq, D] (seq_len_q = SQ > 1) or
 *   [total_q, Hq, D] (packed form); k_dev: combined cache or K pool; v_dev: V pool or NULL;
 *   kv_indptr_dev [B + 1], kv_indices_dev: CSR page ids ([DEC] notes: indptr starts at 0,
 *   ends at the number of indices, and each request owns ceil(len / page_size) entries);
 *   seq_lens_dev [B] (1 <= len <= max_seq_len);
 *   qo_indptr_dev [B + 1]: packed form only (NULL otherwise); request b owns query rows
 *   qo_indptr[b] .. qo_indptr[b + 1]; the offsets start at 0, each step is between 1 and
 *   max_seq_len_q, and they end at total_q ([DEC] notes; a plan that sees them break
 *   this sets the metadata status bit and rows outside [0, total_q) are never written);
 *   out_dev: out_dtype in the query's layout; lse_dev: fp32, one per output row and head
 *   (optional).
 * Under the causal mask every request needs nq <= len ([DEC] notes); a query before the
 * first key sees nothing and gets 0 / -inf.  A (request, KV head) unit of at most 64 rows
 * (G x queries) runs on the split-KV decode kernel; larger units run as dense tiles on the
 * tensor-core kernel (the prefill kernel over the CSR table), no split-KV workspace used.
 * The workspace is exclusive to one launch in flight ([DEC] notes on workspace_buffer). */
int paged_decode_run(const paged_decode_params* params, const void* query_dev,
                     const void* k_dev, const void* v_dev, const int32_t* kv_indptr_dev,
                     const int32_t* kv_indices_dev, const int32_t* seq_lens_dev,
                     const int32_t* qo_indptr_dev, void* out_dev, float* lse_dev,
                     void* workspace_dev, size_t workspace_bytes, void* stream);

/* ---- [SAGE] prequantized block-sparse attention ---------------------------------------
 * bsa_attn_sm120_blk64_sage_fwd computes block-sparse attention on dequantized inputs:
 * q = q_int8 * q_scale[b, h, i / 32] (four scales per 128 queries, [SAGE] q_scale shape
 * [B, H, ceil(Sq / 128) * 4]), k = k_int8 * k_scale[b, h, j / 64], v[j, d] = e4m3(v_fp8[b, h,
 * d, j]) * v_scale[b, h, d]; query block r = i / 64 of (b, h) sees the keys of the first n
 * entries of q2k_block_index[b, h, r] (n = q2k_block_nums[b, h, r], or block_sparse_num
 * when the counts are NULL or uniform_block_count is set), a key j of block c only when
 * j < Sk and j - 64 c < block_sizes[..c]; no causal mask; a query block selecting nothing
 * gets exactly 0 ([SAGE] notes).  The library computes the integer scores exactly (bf16
 * tensor-core MMAs on the int8 values) and applies the scales in fp32.  The
 * contiguous_block_indices hint of the page changes nothing here and has no field. */
typedef struct paged_sage_params {
  int batch;                 /* B                                                        */
  int num_heads;             /* H: the same heads for Q, K and V (MHA)                   */
  int q_len, kv_len;         /* Sq, Sk                                                   */
  int head_dim;              /* 128                                                      */
  int capacity;              /* last dimension of q2k_block_index                        */
  int block_sparse_num;      /* blocks per query block without per-row counts            */
  int uniform_block_count;   /* 1: every query block uses block_sparse_num               */
  int block_sizes_rank;      /* 0: no block_sizes (64 keys each); 1: [NB]; 2: [B, NB];
                                3: [B, H, NB]; NB = ceil(Sk / 64)                        */
  float softmax_scale;       /* > 0; <= 0 selects 1/sqrt(128)                              */
} paged_sage_params;

/* Workspace bytes of paged_sage_run (bf16 copies of Q, K and V, and the block-sparse plan);
 * 0 on invalid params. */
size_t paged_sage_workspace_size(const paged_sage_params* params);

/* Run the prequantized form.  Device pointers: q_int8_dev [B, H, Sq, 128] int8 (16-byte
 * aligned); k_int8_dev [B, H, Sk, 128] int8 (16-byte aligned); v_fp8_dev [B, H, 128, NB * 64]
 * FP8 E4M3 bytes (4-byte aligned); q_scale_dev [B, H, ceil(Sq / 128) * 4], k_scale_dev
 * [B, H, NB], v_scale_dev [B, H, 128] fp32, all positive; q2k_block_index_dev
 * [B, H, ceil(Sq / 64), capacity] int32; q2k_block_nums_dev [B, H, ceil(Sq / 64)] int32 or
 * NULL; block_sizes_dev of rank block_sizes_rank (NULL for rank 0); out_dev [B, H, Sq, 128]
 * bf16.  Counts outside [0, capacity] and block ids outside [0, NB) break the contract: they
 * are clamped or dropped and the metadata bit is set in the status word. */
int paged_sage_run(const paged_sage_params* params, const int8_t* q_int8_dev,
                   const int8_t* k_int8_dev, const uint8_t* v_fp8_dev, const float* q_scale_dev,
                   const float* k_scale_dev, const float* v_scale_dev,
                   const int32_t* q2k_block_index_dev, const int32_t* q2k_block_nums_dev,
                   const int32_t* block_sizes_dev, void* out_dev, void* workspace_dev,
                   size_t workspace_bytes, void* stream);

/* Decode without a workspace argument.  The pages describe no counterpart of this entry
 * point; it exists for callers that cannot allocate device memory at call time (code inside
 * an allocator or out-of-memory handler, plugins whose host owns every device allocation,
 * runtimes that forbid allocations after start-up).  Same arguments and results as
 * paged_decode_run, minus the workspace: the scratch lives in a fixed array inside the
 * library of PAGED_DECODE_STATIC_SCRATCH_BYTES bytes, reserved on every GPU that loads the
 * library until the process exits.  No cudaMalloc, cudaFree or other allocating call is
 * made.
 *   - Returns PAGED_ATTN_ERR_WORKSPACE without enqueuing anything when the problem needs
 *     more scratch than that (paged_decode_workspace_size tells how much it needs).
 *   - The first call on a device looks up the array's address on that device (the device
 *     current at the call); make that first call before any stream capture.
 *   - Every call on a device uses the same array, so calls whose work may overlap on the
 *     GPU (other streams, other threads) race and must be serialised by the caller.
 *   - The device status word (timeouts, page ids outside the pool, broken query offsets)
 *     lives inside the array; read it with paged_decode_static_status. */
#define PAGED_DECODE_STATIC_SCRATCH_BYTES (32u << 20)
int paged_decode_run_static(const paged_decode_params* params, const void* query_dev,
                            const void* k_dev, const void* v_dev, const int32_t* kv_indptr_dev,
                            const int32_t* kv_indices_dev, const int32_t* seq_lens_dev,
                            const int32_t* qo_indptr_dev, void* out_dev, float* lse_dev,
                            void* stream);

/* Status of the last paged_decode_run_static call on the current device: synchronises
 * `stream` (the one that call used), reads the status word from the fixed array and maps it
 * like paged_attn_workspace_status (PAGED_ATTN_OK, _ERR_TIMEOUT, _ERR_CAPACITY or
 * _ERR_METADATA; the raw word to *raw_word when non-NULL).  Allocates nothing.  A call of
 * paged_decode_run_static on this device that is enqueued in between overwrites the word. */
int paged_decode_static_status(void* stream, uint32_t* raw_word);

/* ---- plan inspection -------------------------------------------------------------------- */

/* Where a plan lives inside the workspace (byte offsets from its start), so that callers
 * and tests can read it back.  Fields that do not apply to a form are 0.
 *   tiles:   TileRec {b, g, tok0, ntok, kv_begin, kv_end, q_row0, 0} (8 x int32) in launch
 *            order; BSR: tiles_capacity records; prefill: int32 count at count_offset
 *   bitmap:  int32 indptr [T + 1] and int32 block ids
 *   decode:  int32 split_offset [B + 1], items {b, g, kv_begin, kv_end} (4 x int32) and
 *            the int32 claim order of the items (by size class min(7, 8 x keys / split_chunk),
 *            largest first, list order within a class); the live item count is
 *            num_kv_heads * split_offset[B] */
typedef struct paged_attn_plan_layout {
  size_t status_offset;
  size_t tiles_offset;
  int64_t tiles_capacity;
  size_t count_offset;
  size_t indptr_offset;
  size_t indices_offset;
  int64_t indices_capacity;
  size_t split_offset_offset;
  size_t items_offset;
  int64_t items_capacity;
  int split_chunk;
  int tile_tokens;
  size_t order_offset;   /* decode: int32 claim order of the split items */
} paged_attn_plan_layout;

int paged_attn_plan_layout_of(const paged_attn_params* params, paged_attn_plan_layout* out);
int paged_prefill_plan_layout_of(const paged_prefill_params* params, paged_attn_plan_layout* out);
int paged_decode_plan_layout_of(const paged_decode_params* params, paged_attn_plan_layout* out);

/* ---- benchmark hooks ------------------------------------------------------------------ */

/* Kernel timer.  While enabled, every run brackets its main attention kernel (the
 * block-sparse / prefill tensor-core kernel, the bitmap kernel, or the split-KV decode
 * kernel) with a pair of CUDA events recorded on the launch stream.  enable = 1 clears the
 * record and starts collecting; 0 stops.  Not for use inside CUDA graph capture. */
int paged_attn_kernel_timer(int enable);

/* Sum of the bracketed kernel times in milliseconds and the number of bracketed launches
 * since the timer was last enabled; waits for the recorded events. */
int paged_attn_kernel_timer_read(double* total_ms, int64_t* launches);

/* L2 read rate probe.  Enqueues on `stream` one kernel that reads the `bytes` bytes at
 * buf_dev (16-byte aligned, a multiple of 16) `reps` times with 16-byte loads that bypass L1,
 * spread over every SM; a buffer well inside L2 then measures the rate at which the SMs read
 * L2, the second roofline of the bitmap form (its K/V rows are gathered from L2 once per
 * selecting query).  Time it with events on the same stream: bytes * reps / time.  sink_dev
 * (4 bytes) is written at most once, so that the loads are not optimised away.  Not part of
 * the attention path ([QSA] names no such call). */
int paged_attn_l2_read_probe(const void* buf_dev, size_t bytes, int reps, uint32_t* sink_dev,
                             void* stream);

/* Number of kernels this library has enqueued since it was loaded. */
int64_t paged_attn_launch_count(void);

/* ---- status -------------------------------------------------------------------------- */

/* Synchronise `stream`, read the workspace status word and map it to a status code:
 * PAGED_ATTN_OK, PAGED_ATTN_ERR_TIMEOUT, PAGED_ATTN_ERR_CAPACITY or
 * PAGED_ATTN_ERR_METADATA.  The raw word is stored to *raw_word when non-NULL. */
int paged_attn_workspace_status(const void* workspace_dev, void* stream, uint32_t* raw_word);

/* Static text for a status code. */
const char* paged_attn_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H */
