// Device-side work planner: expands BSR rows, packed-Q prefill requests, per-query block
// bitmaps and decode requests into the work lists the attention kernels consume.  All
// outputs are integers with one correct value each (deterministic ordering, no atomics
// whose order matters), so they can be compared bit for bit with a reference planner.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

// Exclusive scan of one int per thread over a CTA of blockDim.x (a multiple of 32, <=1024)
// threads.  `total` receives the sum over the CTA.
__device__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int before = w > 0 ? warp_sums[w - 1] : 0;
  total = warp_sums[nw - 1];
  __syncthreads();
  return before + x - v;
}

// Exclusive block scan of N values per thread at once (N independent sums); total[k] is the
// block total of value k.  ws: N * 32 ints of shared memory.
template <int N>
__device__ void block_exclusive_scan_n(const int (&v)[N], int (&ex)[N], int (&total)[N], int* ws) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    x[k] = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < N; ++k) ws[k * 32 + w] = x[k];
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      int t = lane < nw ? ws[k * 32 + lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      ws[k * 32 + lane] = t;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    ex[k] = (w > 0 ? ws[k * 32 + w - 1] : 0) + x[k] - v[k];
    total[k] = ws[k * 32 + nw - 1];
  }
}

// ---- block-sparse tiles ----------------------------------------------------------------
// One thread per BSR row (b, g, r).  Tile (b, g, r, m) goes to natural index
// (b * Hkv + g) * tiles_per_bg + r * ceil(qbs / tt) + m.
__global__ void bsr_tiles_kernel(const int* __restrict__ block_indptr, int B, int Hkv, int Sq,
                                 int qbs, int tt, TileRec* __restrict__ tmp) {
  grid_launch_dependents();   // the tile sort may launch now; it waits for these records
  const int nqb = (Sq + qbs - 1) / qbs;
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= B * Hkv * nqb) return;
  const int r = row % nqb, bg = row / nqb, g = bg % Hkv, b = bg / Hkv;
  const int full_tiles = (qbs + tt - 1) / tt;
  const int last_n = Sq - (nqb - 1) * qbs;
  const int tiles_per_bg = (nqb - 1) * full_tiles + (last_n + tt - 1) / tt;
  const int n_r = min(qbs, Sq - r * qbs);
  const int base = bg * tiles_per_bg + r * full_tiles;
  const int kb = block_indptr[bg * (nqb + 1) + r];
  const int ke = block_indptr[bg * (nqb + 1) + r + 1];
  for (int m = 0; m * tt < n_r; ++m) {
    TileRec t;
    t.b = b;
    t.g = g;
    t.tok0 = r * qbs + m * tt;
    t.ntok = min(tt, n_r - m * tt);
    t.kv_begin = kb;
    t.kv_end = ke;
    t.q_row0 = b * Sq + t.tok0;
    t.pad = 0;
    tmp[base + m] = t;
  }
}

// ---- packed-Q prefill tiles --------------------------------------------------------------
__global__ void prefill_count_kernel(const int* __restrict__ qo, int q_len, int B, int Hkv,
                                     int tt, int capacity, int* __restrict__ off, int* n_tiles,
                                     uint32_t* status) {
  grid_launch_dependents();
  __shared__ int warp_sums[32];
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int c = 0;
    if (b < B) {
      const int nq = qo ? qo[b + 1] - qo[b] : q_len;
      c = nq > 0 ? (nq + tt - 1) / tt : 0;
    }
    int total;
    const int ex = block_exclusive_scan(c, warp_sums, total);
    if (b < B) off[b] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) {
    off[B] = carry;
    long long n = static_cast<long long>(Hkv) * carry;
    if (n > capacity) {
      report_error(status, kErrCapacity);
      n = capacity;
    }
    *n_tiles = static_cast<int>(n);
  }
}

__global__ void prefill_fill_kernel(const int* __restrict__ qo, int q_len,
                                    const int* __restrict__ lens, int Hkv, int tt, int causal,
                                    int window_left, int capacity, const int* __restrict__ off,
                                    TileRec* __restrict__ tmp) {
  grid_launch_dependents();
  grid_dependency_wait();     // the tile offsets of the count kernel
  const int b = blockIdx.x;
  const int nq = qo ? qo[b + 1] - qo[b] : q_len;
  const int row0 = qo ? qo[b] : b * q_len;
  const int L = lens[b];
  const int nt = off[b + 1] - off[b];
  for (int idx = threadIdx.x; idx < Hkv * nt; idx += blockDim.x) {
    const int g = idx / nt, m = idx % nt;
    const long long pos = static_cast<long long>(Hkv) * off[b] + idx;
    if (pos >= capacity) continue;
    const int tok0 = m * tt;
    const int ntok = min(tt, nq - tok0);
    const long long p0 = static_cast<long long>(L) - nq + tok0;
    const long long p1 = p0 + ntok - 1;
    const long long hi = causal ? min(static_cast<long long>(L), p1 + 1) : L;
    const long long lo = (causal && window_left >= 0) ? max(0LL, p0 - window_left) : 0LL;
    TileRec t;
    t.b = b;
    t.g = g;
    t.tok0 = tok0;
    t.ntok = ntok;
    if (hi <= lo) {
      t.kv_begin = t.kv_end = 0;
    } else {
      t.kv_begin = static_cast<int>(lo / kKvTile);
      t.kv_end = static_cast<int>((hi + kKvTile - 1) / kKvTile);
    }
    t.q_row0 = row0 + tok0;
    t.pad = 0;
    tmp[pos] = t;
  }
}

// ---- stable counting sort of tiles by capped cost, descending ------------------------------
__device__ __forceinline__ int rec_cost(const TileRec& r, int maxc) {
  const int c = r.kv_end - r.kv_begin;
  return c < 0 ? 0 : (c > maxc ? maxc : c);
}

__global__ void sort_hist_kernel(const TileRec* __restrict__ in, const int* n_dev, int n_static,
                                 int maxc, int* __restrict__ hist) {
  grid_launch_dependents();
  grid_dependency_wait();     // the records and their count
  extern __shared__ int h[];
  const int n = n_dev ? *n_dev : n_static;
  for (int k = threadIdx.x; k <= maxc; k += blockDim.x) h[k] = 0;
  __syncthreads();
  const int i = blockIdx.x * kSortChunk + threadIdx.x;
  if (i < n) atomicAdd(&h[rec_cost(in[i], maxc)], 1);
  __syncthreads();
  for (int k = threadIdx.x; k <= maxc; k += blockDim.x)
    hist[static_cast<long long>(blockIdx.x) * (maxc + 1) + k] = h[k];
}

__global__ void sort_offsets_kernel(int nchunks, int maxc, const int* __restrict__ hist,
                                    int* __restrict__ offs) {
  grid_launch_dependents();
  grid_dependency_wait();     // the histograms
  extern __shared__ int tot[];
  __shared__ int warp_sums[32];
  const long long W = maxc + 1;
  for (int k = threadIdx.x; k <= maxc; k += blockDim.x) {
    int run = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int v = hist[c * W + k];
      offs[c * W + k] = run;
      run += v;
    }
    tot[k] = run;
  }
  __syncthreads();
  // base[k] = number of records with a larger cost: scan the bins from the top.
  int carry = 0;
  for (int d0 = 0; d0 <= maxc; d0 += blockDim.x) {
    const int d = d0 + threadIdx.x;
    const int v = d <= maxc ? tot[maxc - d] : 0;
    int total;
    const int ex = block_exclusive_scan(v, warp_sums, total);
    if (d <= maxc) tot[maxc - d] = carry + ex;
    carry += total;
  }
  __syncthreads();
  for (int k = threadIdx.x; k <= maxc; k += blockDim.x)
    for (int c = 0; c < nchunks; ++c) offs[c * W + k] += tot[k];
}

__global__ void sort_scatter_kernel(const TileRec* __restrict__ in, TileRec* __restrict__ out,
                                    const int* n_dev, int n_static, int maxc,
                                    const int* __restrict__ offs) {
  grid_launch_dependents();   // the attention kernel may start its prologue
  grid_dependency_wait();     // the offsets (and, through the chain, the records)
  extern __shared__ int cnt[];
  const int n = n_dev ? *n_dev : n_static;
  for (int k = threadIdx.x; k <= maxc; k += blockDim.x) cnt[k] = 0;
  __syncthreads();
  const int i = blockIdx.x * kSortChunk + threadIdx.x;
  const bool live = i < n;
  const int k = live ? rec_cost(in[i], maxc) : -1;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned peers = __match_any_sync(0xffffffffu, k);
  const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
  const int leader = __ffs(peers) - 1;
  int my_base = 0;
  // Warps take their turn in index order, so equal costs keep their input order.
  for (int step = 0; step < (kSortChunk >> 5); ++step) {
    if (w == step) {
      if (live) my_base = cnt[k];
      __syncwarp();
      if (live && lane == leader) cnt[k] = my_base + __popc(peers);
    }
    __syncthreads();
  }
  if (live) {
    const long long pos =
        offs[static_cast<long long>(blockIdx.x) * (maxc + 1) + k] + my_base + rank_in_warp;
    out[pos] = in[i];
  }
}

// ---- block-sparse plan of at most one sort chunk, in one CTA ------------------------------
// The records of bsr_tiles_kernel and the stable counting sort of the three sort kernels
// (same records, same order), built in shared memory by one CTA of kSortChunk threads: a
// small plan costs one launch instead of four.  Also clears the workspace status words.
__global__ void __launch_bounds__(kSortChunk)
bsr_plan_small_kernel(const int* __restrict__ block_indptr, int B, int Hkv, int Sq, int qbs,
                      int tt, int maxc, int n, TileRec* __restrict__ out,
                      uint32_t* __restrict__ status) {
  extern __shared__ int4 sm_small[];
  TileRec* recs = reinterpret_cast<TileRec*>(sm_small);          // n records
  int* cnt = reinterpret_cast<int*>(recs + n);                   // maxc + 1 bins
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid < 4) status[tid] = 0u;
  // tiles in their natural order (the indexing of bsr_tiles_kernel)
  const int nqb = (Sq + qbs - 1) / qbs;
  if (tid < B * Hkv * nqb) {
    const int r = tid % nqb, bg = tid / nqb, g = bg % Hkv, b = bg / Hkv;
    const int full_tiles = (qbs + tt - 1) / tt;
    const int last_n = Sq - (nqb - 1) * qbs;
    const int tiles_per_bg = (nqb - 1) * full_tiles + (last_n + tt - 1) / tt;
    const int n_r = min(qbs, Sq - r * qbs);
    const int base = bg * tiles_per_bg + r * full_tiles;
    const int kb = block_indptr[bg * (nqb + 1) + r];
    const int ke = block_indptr[bg * (nqb + 1) + r + 1];
    for (int m = 0; m * tt < n_r; ++m) {
      TileRec t;
      t.b = b;
      t.g = g;
      t.tok0 = r * qbs + m * tt;
      t.ntok = min(tt, n_r - m * tt);
      t.kv_begin = kb;
      t.kv_end = ke;
      t.q_row0 = b * Sq + t.tok0;
      t.pad = 0;
      recs[base + m] = t;
    }
  }
  for (int k = tid; k <= maxc; k += blockDim.x) cnt[k] = 0;
  __syncthreads();
  const bool live = tid < n;
  const int k = live ? rec_cost(recs[tid], maxc) : -1;
  if (live) atomicAdd(&cnt[k], 1);
  __syncthreads();
  // cnt[k] := number of records with a larger cost (scan of the bins from the top)
  int carry = 0;
  for (int d0 = 0; d0 <= maxc; d0 += blockDim.x) {
    const int d = d0 + tid;
    const int v = d <= maxc ? cnt[maxc - d] : 0;
    int total;
    const int ex = block_exclusive_scan(v, warp_sums, total);
    if (d <= maxc) cnt[maxc - d] = carry + ex;
    carry += total;
  }
  __syncthreads();
  // stable scatter: warps take their turn in index order, lanes by rank among equal costs
  const unsigned peers = __match_any_sync(0xffffffffu, k);
  const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
  const int leader = __ffs(peers) - 1;
  int my_base = 0;
  for (int step = 0; step < (kSortChunk >> 5); ++step) {
    if (w == step) {
      if (live) my_base = cnt[k];
      __syncwarp();
      if (live && lane == leader) cnt[k] = my_base + __popc(peers);
    }
    __syncthreads();
  }
  if (live) out[my_base + rank_in_warp] = recs[tid];
}

// ---- bitmap planner ------------------------------------------------------------------------
__device__ __forceinline__ int first_block_ending_at_or_after(const int* __restrict__ blast,
                                                              int NB, int lo) {
  int a = 0, b = NB;
  while (a < b) {
    const int m = (a + b) >> 1;
    if (blast[m] < lo) a = m + 1;
    else b = m;
  }
  return a;
}

// One warp per query token; lane l looks at blocks base + 4l .. base + 4l + 3.
template <bool kFill>
__global__ void bitmap_scan_kernel(const uint8_t* __restrict__ sel, const int* __restrict__ lo,
                                   const int* __restrict__ hi, const int* __restrict__ bfirst,
                                   const int* __restrict__ blast, int T, int NB,
                                   int* __restrict__ counts, const int* __restrict__ indptr,
                                   int* __restrict__ indices, long long capacity) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int l = lo[t], h = hi[t];
  long long written = kFill ? indptr[t] : 0;
  int cnt = 0;
  if (h >= l) {
    const int g0 = first_block_ending_at_or_after(blast, NB, l);
    const long long rowbase = static_cast<long long>(t) * NB;
    for (int base = g0; base < NB; base += 128) {
      bool stop = false;
      int mine[4];
      int c = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int g = base + lane * 4 + e;
        if (g < NB) {
          const int f = bfirst[g];
          if (f > h) {
            stop = true;
          } else if (sel[rowbase + g] != 0 && max(f, l) <= min(blast[g], h)) {
            mine[c++] = g;
          }
        }
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (kFill) {
        const long long at = written + incl - c;
        for (int e = 0; e < c; ++e)
          if (at + e < capacity) indices[at + e] = mine[e];
      }
      written += total;
      cnt += total;
      if (__any_sync(0xffffffffu, stop)) break;
    }
  }
  if (!kFill && lane == 0) counts[t] = cnt;
}

__global__ void counts_to_indptr_kernel(const int* __restrict__ counts, int T, long long capacity,
                                        int* __restrict__ indptr, uint32_t* status) {
  __shared__ int warp_sums[32];
  long long carry = 0;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    const int c = t < T ? counts[t] : 0;
    int total;
    const int ex = block_exclusive_scan(c, warp_sums, total);
    if (t < T) indptr[t] = static_cast<int>(carry + ex);
    carry += total;
  }
  if (threadIdx.x == 0) {
    indptr[T] = static_cast<int>(carry);
    if (carry > capacity) report_error(status, kErrCapacity);
  }
}

// ---- indexed per-query block plan --------------------------------------------------------
// One warp per query token t: the K entries of row t are read 32 at a time (coalesced); an
// entry g is kept when 0 <= g < NB and its span meets [lo[t], hi[t]], in the caller's order
// (ballot compaction).  Entries >= NB break the contract: they are dropped and reported.
// kFill = false writes the count of row t; kFill = true writes the ids from indptr[t] on.
template <bool kFill>
__global__ void indexed_scan_kernel(const int* __restrict__ idx, int K,
                                    const int* __restrict__ lo, const int* __restrict__ hi,
                                    const int* __restrict__ bfirst,
                                    const int* __restrict__ blast, int T, int NB,
                                    int* __restrict__ counts, const int* __restrict__ indptr,
                                    int* __restrict__ indices, long long capacity,
                                    uint32_t* status) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int l = lo[t], h = hi[t];
  long long written = kFill ? indptr[t] : 0;
  const long long rowbase = static_cast<long long>(t) * K;
  bool bad = false;
  for (int base = 0; base < K; base += 32) {
    const int e = base + lane;
    bool keep = false;
    int g = -1;
    if (e < K) {
      g = idx[rowbase + e];
      if (g >= NB) bad = true;
      else if (g >= 0) keep = max(bfirst[g], l) <= min(blast[g], h);
    }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (kFill && keep) {
      const long long at = written + __popc(m & ((1u << lane) - 1u));
      if (at < capacity) indices[at] = g;
    }
    written += __popc(m);
  }
  if (!kFill) {
    if (__any_sync(0xffffffffu, bad) && lane == 0) report_error(status, kErrMetadata);
    if (lane == 0) counts[t] = static_cast<int>(written);
  }
}

// ---- decode split planner -----------------------------------------------------------------
__device__ __forceinline__ void decode_split_range(int L, int nq, int chunk, int window_left,
                                                   int& lo, int& s0, int& n) {
  if (L < 0) L = 0;
  // the earliest query sits at L - nq and keeps keys from L - nq - window_left on
  const long long first = static_cast<long long>(L) - nq - window_left;
  lo = window_left >= 0 ? static_cast<int>(first > 0 ? first : 0) : 0;
  s0 = lo / chunk;
  const int s1 = max((L + chunk - 1) / chunk, s0 + 1);
  n = s1 - s0;
}

constexpr int kOrderClasses = 8;   // size classes of the claim order

// One CTA: split counts, their exclusive scan, the work items, their claim order and zeroed
// counters.
__global__ void decode_plan_kernel(const int* __restrict__ lens, const int* __restrict__ qo,
                                   int q_len, int max_q, int total_q, int B, int Hkv, int chunk,
                                   int window_left, int max_splits, int* __restrict__ off,
                                   SplitItem* __restrict__ items, int* __restrict__ order,
                                   int* __restrict__ counters, uint32_t* status) {
  __shared__ int warp_sums[32];
  // the split kernel that follows may start its prologue now; it reads nothing of the plan
  // before this kernel has completed
  grid_launch_dependents();
  if (threadIdx.x < 4) status[threadIdx.x] = 0;   // the status word of this run
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int n = 0;
    if (b < B) {
      const int nq = qo ? qo[b + 1] - qo[b] : q_len;
      if (qo && (nq < 1 || nq > max_q || (b == 0 && qo[0] != 0) || (b == B - 1 && qo[B] != total_q)))
        report_error(status, kErrMetadata);
      int lo, s0;
      decode_split_range(lens[b], nq, chunk, window_left, lo, s0, n);
      n = min(n, max_splits);
    }
    int total;
    const int ex = block_exclusive_scan(n, warp_sums, total);
    if (b < B) off[b] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) off[B] = carry;
  for (int i = threadIdx.x; i <= B * Hkv; i += blockDim.x) counters[i] = 0;
  __syncthreads();
  // items of request b: one warp per request
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int b = threadIdx.x >> 5; b < B; b += nw) {
    int L = lens[b];
    const int nq = qo ? qo[b + 1] - qo[b] : q_len;
    int lo, s0, n_all;
    decode_split_range(L, nq, chunk, window_left, lo, s0, n_all);
    if (L < 0) L = 0;
    const int n = off[b + 1] - off[b];
    for (int idx = lane; idx < Hkv * n; idx += 32) {
      const int g = idx / n, k = idx % n;
      const long long s = static_cast<long long>(s0) + k;
      SplitItem it;
      it.b = b;
      it.g = g;
      it.kv_begin = static_cast<int>(max(s * chunk, static_cast<long long>(lo)));
      it.kv_end = static_cast<int>(min((s + 1) * chunk, static_cast<long long>(L)));
      items[static_cast<long long>(Hkv) * off[b] + idx] = it;
    }
  }
  __syncthreads();
  // Claim order: items by size class min(7, 8 * size / chunk), largest first, list order
  // within a class.  Thread t ranks a contiguous run of items: class counts in registers,
  // one block scan per class, then the positions.  The class of a size is the number of
  // thresholds ceil(c * chunk / 8), c = 1..7, it reaches.
  const int n_items = Hkv * off[B];
  const int per = (n_items + blockDim.x - 1) / blockDim.x;
  const int i0 = min(n_items, static_cast<int>(threadIdx.x) * per);
  const int i1 = min(n_items, i0 + per);
  int thr[kOrderClasses];
#pragma unroll
  for (int c = 1; c < kOrderClasses; ++c)
    thr[c] = static_cast<int>((static_cast<long long>(c) * chunk + kOrderClasses - 1) / kOrderClasses);
  auto cls = [&](int i) {
    const int z = items[i].kv_end - items[i].kv_begin;
    int c = 0;
#pragma unroll
    for (int k = 1; k < kOrderClasses; ++k) c += z >= thr[k];
    return c;
  };
  int cnt[kOrderClasses];
#pragma unroll
  for (int c = 0; c < kOrderClasses; ++c) cnt[c] = 0;
  for (int i = i0; i < i1; ++i) {
    const int ci = cls(i);
#pragma unroll
    for (int c = 0; c < kOrderClasses; ++c) cnt[c] += ci == c;
  }
  __shared__ int class_sums[kOrderClasses * 32];
  int pos[kOrderClasses], tot[kOrderClasses];
  block_exclusive_scan_n<kOrderClasses>(cnt, pos, tot, class_sums);
  int base = 0;
#pragma unroll
  for (int c = kOrderClasses - 1; c >= 0; --c) {
    pos[c] += base;
    base += tot[c];
  }
  for (int i = i0; i < i1; ++i) {
    const int ci = cls(i);
    int p = 0;
#pragma unroll
    for (int c = 0; c < kOrderClasses; ++c)
      if (ci == c) p = pos[c]++;
    order[p] = i;
  }
}

}  // namespace

// ---- launchers ---------------------------------------------------------------------------
void launch_bsr_tiles(const int* block_indptr, int B, int Hkv, int Sq, int qbs, int tile_tokens,
                      TileRec* tmp, cudaStream_t st) {
  const int rows = B * Hkv * ceil_div(Sq, qbs);
  if (rows <= 0) return;
  bsr_tiles_kernel<<<ceil_div(rows, 256), 256, 0, st>>>(block_indptr, B, Hkv, Sq, qbs,
                                                        tile_tokens, tmp);
  count_launches(1);
}

bool bsr_plan_is_small(int B, int Hkv, int Sq, int qbs, int capacity, int max_cost) {
  const long long rows = static_cast<long long>(B) * Hkv * ceil_div(Sq, qbs);
  const long long smem = static_cast<long long>(capacity) * sizeof(TileRec) +
                         static_cast<long long>(max_cost + 1) * sizeof(int);
  return capacity > 0 && capacity <= kSortChunk && rows <= kSortChunk && smem <= 40 * 1024;
}

void launch_bsr_plan_small(const int* block_indptr, int B, int Hkv, int Sq, int qbs,
                           int tile_tokens, int capacity, int max_cost, TileRec* out,
                           uint32_t* status, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(capacity) * sizeof(TileRec) +
                      static_cast<size_t>(max_cost + 1) * sizeof(int);
  bsr_plan_small_kernel<<<1, kSortChunk, smem, st>>>(block_indptr, B, Hkv, Sq, qbs, tile_tokens,
                                                     max_cost, capacity, out, status);
  count_launches(1);
}

void launch_prefill_tiles(const int* qo_indptr, int q_len, const int* seq_lens, int B, int Hkv,
                          int tile_tokens, int causal, int window_left, int capacity,
                          int* tile_offsets, int* n_tiles, TileRec* tmp, uint32_t* status,
                          cudaStream_t st) {
  prefill_count_kernel<<<1, 1024, 0, st>>>(qo_indptr, q_len, B, Hkv, tile_tokens, capacity,
                                           tile_offsets, n_tiles, status);
  count_launches(1);
  if (B > 0) {
    launch_after_previous(prefill_fill_kernel, dim3(B), dim3(256), 0, st, qo_indptr, q_len,
                          seq_lens, Hkv, tile_tokens, causal, window_left, capacity,
                          static_cast<const int*>(tile_offsets), tmp);
    count_launches(1);
  }
}

size_t tile_sort_scratch_ints(int capacity, int max_cost) {
  const size_t nchunks = static_cast<size_t>(ceil_div(capacity > 0 ? capacity : 1, kSortChunk));
  return nchunks * static_cast<size_t>(max_cost + 1);
}

void launch_tile_sort(const TileRec* in, TileRec* out, const int* n_dev, int n_static,
                      int capacity, int max_cost, int* hist, int* offs, cudaStream_t st) {
  if (capacity <= 0) return;
  const int nchunks = ceil_div(capacity, kSortChunk);
  const size_t sm = static_cast<size_t>(max_cost + 1) * sizeof(int);
  launch_after_previous(sort_hist_kernel, dim3(nchunks), dim3(kSortChunk), sm, st, in, n_dev,
                        n_static, max_cost, hist);
  launch_after_previous(sort_offsets_kernel, dim3(1), dim3(1024), sm, st, nchunks, max_cost,
                        static_cast<const int*>(hist), offs);
  launch_after_previous(sort_scatter_kernel, dim3(nchunks), dim3(kSortChunk), sm, st, in, out,
                        n_dev, n_static, max_cost, static_cast<const int*>(offs));
  count_launches(3);
}

void launch_bitmap_plan(const uint8_t* sel, const int* lo, const int* hi, const int* bfirst,
                        const int* blast, int T, int NB, long long capacity, int* indptr,
                        int* indices, uint32_t* status, cudaStream_t st) {
  if (T <= 0) return;
  const int warps_per_cta = 8;
  const int grid = ceil_div(T, warps_per_cta);
  // counts are staged in indices' tail-free scratch: indptr[1..T] first holds the counts
  bitmap_scan_kernel<false><<<grid, 32 * warps_per_cta, 0, st>>>(
      sel, lo, hi, bfirst, blast, T, NB, indptr + 1, nullptr, nullptr, capacity);
  counts_to_indptr_kernel<<<1, 1024, 0, st>>>(indptr + 1, T, capacity, indptr, status);
  bitmap_scan_kernel<true><<<grid, 32 * warps_per_cta, 0, st>>>(
      sel, lo, hi, bfirst, blast, T, NB, nullptr, indptr, indices, capacity);
  count_launches(3);
}

void launch_indexed_plan(const int* idx, int K, const int* lo, const int* hi, const int* bfirst,
                         const int* blast, int T, int NB, long long capacity, int* indptr,
                         int* indices, uint32_t* status, cudaStream_t st) {
  if (T <= 0) return;
  const int warps_per_cta = 8;
  const int grid = ceil_div(T, warps_per_cta);
  indexed_scan_kernel<false><<<grid, 32 * warps_per_cta, 0, st>>>(
      idx, K, lo, hi, bfirst, blast, T, NB, indptr + 1, nullptr, nullptr, capacity, status);
  counts_to_indptr_kernel<<<1, 1024, 0, st>>>(indptr + 1, T, capacity, indptr, status);
  indexed_scan_kernel<true><<<grid, 32 * warps_per_cta, 0, st>>>(
      idx, K, lo, hi, bfirst, blast, T, NB, nullptr, indptr, indices, capacity, status);
  count_launches(3);
}

void launch_decode_plan(const int* seq_lens, const int* qo_indptr, int q_len, int max_q,
                        int total_q, int B, int Hkv, int chunk, int window_left, int max_splits,
                        int* split_offset, SplitItem* items, int* order, int* counters,
                        uint32_t* status, cudaStream_t st) {
  decode_plan_kernel<<<1, 1024, 0, st>>>(seq_lens, qo_indptr, q_len, max_q, total_q, B, Hkv,
                                         chunk, window_left, max_splits, split_offset, items,
                                         order, counters, status);
  count_launches(1);
}

}  // namespace pa
