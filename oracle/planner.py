"""Plain-Python oracle of the work planner (integer outputs, compared bit for bit).

TEST INFRASTRUCTURE ONLY: imported by the test suite, never by the library.

The pages fix what is computed, not how it is scheduled; the planner layout below is this
library's own contract and is restated here independently of the CUDA planner kernels.

M-tile rows pack (token, head-in-group) pairs: row m of a tile is token tok0 + m // G,
query head g * G + m % G, with G = Hq / Hkv.  A tile holds `tile_tokens` tokens of one
(request, KV head) and, for the block-sparse form, never crosses a query-block boundary.

Tile record (8 int32): b, g, tok0, ntok, kv_begin, kv_end, q_row0, 0
  block-sparse : kv_begin/kv_end bound the block_indices slice of the tile's BSR row;
                 q_row0 = b * Sq + tok0
  dense prefill: kv_begin/kv_end are 128-key tile numbers [first, end) covering the
                 visible key span of the tile's rows; q_row0 = qo_indptr[b] + tok0
Tiles are ordered by cost = kv_end - kv_begin, largest first; equal costs keep their
natural order, which is (b, g, q-block, m) for the block-sparse form and (b, g, m) for
the dense form.
"""
from __future__ import annotations

import numpy as np

from .attention import i64

KV_TILE = 128  # keys per dense-prefill KV tile


def _sort_tiles(recs):
    recs = np.asarray(recs, dtype=np.int64).reshape(-1, 8)
    cost = recs[:, 5] - recs[:, 4]
    order = sorted(range(len(recs)), key=lambda i: (-int(cost[i]), i))
    return recs[order].astype(np.int32)


def plan_bsr_tiles(B, Sq, Hq, Hkv, q_block_size, block_indptr, tile_tokens):
    """Tile list of the block-sparse form; see the module docstring for the record."""
    bptr = i64(block_indptr)
    nqb = -(-Sq // q_block_size)
    recs = []
    for b in range(B):
        for g in range(Hkv):
            for r in range(nqb):
                n_r = min(q_block_size, Sq - r * q_block_size)
                for m in range(-(-n_r // tile_tokens)):
                    tok0 = r * q_block_size + m * tile_tokens
                    ntok = min(tile_tokens, n_r - m * tile_tokens)
                    recs.append([b, g, tok0, ntok, bptr[b, g, r], bptr[b, g, r + 1],
                                 b * Sq + tok0, 0])
    return _sort_tiles(recs)


def bsr_tile_capacity(B, Sq, Hkv, q_block_size, tile_tokens):
    nqb = -(-Sq // q_block_size)
    n = 0
    for r in range(nqb):
        n_r = min(q_block_size, Sq - r * q_block_size)
        n += -(-n_r // tile_tokens)
    return B * Hkv * n


def plan_prefill_tiles(Hkv, qo_indptr, seq_lens_kv, tile_tokens, mask_type="dense",
                       window_left=-1):
    """Tile list of the dense packed-Q prefill form.

    The keys a tile can see run from lo = max(0, p(tok0) - window_left) (0 without a
    window) to hi = min(len_kv, p(tok0 + ntok - 1) + 1) under the causal mask (len_kv
    otherwise); kv tiles are [lo // 128, ceil(hi / 128)), or empty when hi <= lo.
    """
    qo, lens = i64(qo_indptr), i64(seq_lens_kv)
    recs = []
    for b in range(len(lens)):
        nq, L = int(qo[b + 1] - qo[b]), int(lens[b])
        for g in range(Hkv):
            for m in range(-(-nq // tile_tokens)):
                tok0 = m * tile_tokens
                ntok = min(tile_tokens, nq - tok0)
                p0 = L - nq + tok0
                p1 = p0 + ntok - 1
                hi = min(L, p1 + 1) if mask_type == "causal" else L
                lo = max(0, p0 - window_left) if (mask_type == "causal" and window_left >= 0) \
                    else 0
                if hi <= lo:
                    kb = ke = 0
                else:
                    kb, ke = lo // KV_TILE, -(-hi // KV_TILE)
                recs.append([b, g, tok0, ntok, kb, ke, int(qo[b]) + tok0, 0])
    return _sort_tiles(recs)


def decode_split_chunk(B, Hkv, max_seq_len, num_sms):
    """Keys per split-KV partition, from static arguments only: 128 x max(1, floor(B * Hkv *
    ceil(max_seq_len / 128) / (16 * num_sms))), capped at ceil(max_seq_len / 128) tiles."""
    tiles = max(1, -(-max_seq_len // 128))
    ct = max(1, (B * Hkv * tiles) // (16 * num_sms))
    return 128 * min(ct, tiles)


def plan_decode(seq_lens, Hkv, chunk, window_left=-1, q_lens=None):
    """Split-KV work list.  Request b with L keys and nq queries (q_lens[b], default 1) has
    its visible keys in [lo, L): lo = max(0, L - nq - window_left) with a window (the first
    key the earliest query, at position L - nq, keeps), else 0.  [lo, L) is cut at
    multiples of `chunk`: splits s in [lo // chunk, max(ceil(L / chunk), lo // chunk + 1)).
    split_offset is the exclusive prefix sum of the split counts; item Hkv * split_offset[b]
    + g * n_b + k is (b, g, kv_begin, kv_end) of the k-th split, kv_begin = max(s * chunk,
    lo) and kv_end = min((s + 1) * chunk, L)."""
    lens = i64(seq_lens)
    B = lens.size
    nqs = np.ones(B, np.int64) if q_lens is None else i64(q_lens)
    counts, firsts = [], []
    for L, nq in zip(lens, nqs):
        L, nq = int(L), int(nq)
        lo = max(0, L - nq - window_left) if window_left >= 0 else 0
        s0 = lo // chunk
        s1 = max(-(-L // chunk), s0 + 1)
        counts.append(s1 - s0)
        firsts.append((s0, lo))
    split_offset = np.zeros(B + 1, dtype=np.int64)
    split_offset[1:] = np.cumsum(counts)
    items = np.zeros((Hkv * int(split_offset[-1]), 4), dtype=np.int64)
    for b in range(B):
        L = int(lens[b])
        s0, lo = firsts[b]
        n = counts[b]
        for g in range(Hkv):
            for k in range(n):
                s = s0 + k
                items[Hkv * split_offset[b] + g * n + k] = [b, g, max(s * chunk, lo),
                                                             min((s + 1) * chunk, L)]
    return split_offset.astype(np.int32), items.astype(np.int32)


ORDER_CLASSES = 8  # size classes of the split-KV claim order


def decode_work_order(items, chunk):
    """Order in which the split-KV work items are claimed: by size class
    min(7, 8 * (kv_end - kv_begin) // chunk), largest class first; items of one class keep
    their list order.  The longest splits start first and the short tails of the requests
    fill the end of the launch."""
    items = np.asarray(items, dtype=np.int64).reshape(-1, 4)
    size = items[:, 3] - items[:, 2]
    cls = np.clip((ORDER_CLASSES * size) // chunk, 0, ORDER_CLASSES - 1)
    return np.array(sorted(range(len(items)), key=lambda i: (-int(cls[i]), i)), dtype=np.int32)


def plan_bitmap(sel_blocks, lo, hi, block_first, block_last):
    """Per-query CSR of selected global block IDs (ascending): block g is listed for query
    t iff sel_blocks[t, g] != 0 and [block_first[g], block_last[g]] meets [lo[t], hi[t]]."""
    sel = sel_blocks.numpy() if hasattr(sel_blocks, "numpy") else np.asarray(sel_blocks)
    lo_, hi_ = i64(lo), i64(hi)
    first, last = i64(block_first), i64(block_last)
    T = lo_.size
    indptr = np.zeros(T + 1, dtype=np.int64)
    parts = []
    for t in range(T):
        g = np.nonzero(sel[t])[0]
        g = g[np.maximum(first[g], lo_[t]) <= np.minimum(last[g], hi_[t])]
        parts.append(g)
        indptr[t + 1] = indptr[t] + g.size
    indices = np.concatenate(parts) if parts else np.zeros(0, np.int64)
    return indptr.astype(np.int32), indices.astype(np.int32)


def plan_indexed(sel_indices, lo, hi, block_first, block_last):
    """Per-query CSR of the indexed form: row t keeps, in the caller's order, the entries g of
    sel_indices[t] with 0 <= g < NB whose span [block_first[g], block_last[g]] meets
    [lo[t], hi[t]]; every other entry is dropped."""
    idx = sel_indices.numpy() if hasattr(sel_indices, "numpy") else np.asarray(sel_indices)
    lo_, hi_ = i64(lo), i64(hi)
    first, last = i64(block_first), i64(block_last)
    NB = first.size
    T = lo_.size
    indptr = np.zeros(T + 1, dtype=np.int64)
    parts = []
    for t in range(T):
        keep = [int(g) for g in idx[t]
                if 0 <= int(g) < NB and max(first[g], lo_[t]) <= min(last[g], hi_[t])]
        parts.append(np.array(keep, dtype=np.int64))
        indptr[t + 1] = indptr[t] + len(keep)
    indices = np.concatenate(parts) if parts else np.zeros(0, np.int64)
    return indptr.astype(np.int32), indices.astype(np.int32)
