"""Float64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's CPU
baseline leg import this module; the library's CUDA path never does, and the two share no
code.  Everything here is plain NumPy float64 on the exact (bf16-valued) inputs: the
logical K/V of each request is materialised from its pages, the visibility of every
(query row, head, key) triple is decided from the pages' selection and mask rules, and a
masked softmax is taken directly.

Sources (FlashInfer API pages):
  [BSA]  flashinfer.attention.prims_ts.block_sparse_attention_with_paged_kv_cache
  [PRE]  flashinfer.attention.prims_ts.batch_prefill_with_paged_kv_cache
  [QSA]  flashinfer.qsa.qsa_forward
  [DEC]  flashinfer.attention.prims_ts.prims_ts_batch_decode_with_kv_cache
  [SAGE] flashinfer.cute_dsl.sparse.bsa_attn_sm120.bsa_attn_sm120_blk64_sage_fwd

Readings where the pages are silent:
  * query position: query i of a request with len_q queries and len_kv keys sits at
    p(i) = len_kv - len_q + i (bottom-right aligned);
  * GQA: query head h reads KV head h // (Hq / Hkv);
  * combined cache axis 1: index 0 = K, 1 = V;
  * kv_valid_bits: bit (j & 31) of uint32 word (j >> 5), 1 = live token;
  * LSE is the natural log of sum_j exp(scale * q.k_j) over visible keys (sm_scale
    included, output_scale excluded);
  * window_left = w >= 0 keeps keys p - w <= j <= p (w + 1 keys);
  * output_scale / bmm2_scale multiply the normalised output;
  * a row with no visible key gives O = 0 exactly and LSE = -inf (the rule [QSA] states,
    applied to every form);
  * [QSA] sel_blocks columns are global block IDs whose token spans are
    [block_first[g], block_last[g]]; only lo/hi and the bitmap decide visibility.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def f64(x) -> np.ndarray:
    """Exact float64 copy of a (bf16/fp32) tensor or array."""
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def i64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def u32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x).view(np.uint32)


def bf16_round(x: np.ndarray) -> torch.Tensor:
    """Round float64 values to bf16, nearest-even (torch's conversion)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16)


# ----------------------------------------------------------------------------------------
# The masked softmax: the definition every form reduces to.
# ----------------------------------------------------------------------------------------

def masked_softmax_attention(q, keys, vals, visible, scale, out_scale=1.0):
    """q [n, G, D] (G query heads sharing one KV head), keys/vals [L, D], visible [n, L].

    s_j = scale * q . k_j on visible keys; LSE = log sum_j exp(s_j); O = out_scale *
    sum_j exp(s_j - LSE) v_j.  Rows with no visible key: O = 0, LSE = -inf.
    Returns O [n, G, D], LSE [n, G].
    """
    n, G, D = q.shape
    L = keys.shape[0]
    out = np.zeros((n, G, D))
    lse = np.full((n, G), -np.inf)
    if n == 0 or L == 0:
        return out, lse
    s = np.matmul(q.reshape(n * G, D), keys.T).reshape(n, G, L) * scale
    s = np.where(visible[:, None, :], s, -np.inf)
    live = visible.any(axis=1)
    if not live.any():
        return out, lse
    s = s[live]
    m = s.max(axis=2, keepdims=True)
    e = np.exp(s - m)
    e = np.where(visible[live][:, None, :], e, 0.0)
    l = e.sum(axis=2)
    vis_vals = np.where(visible[live].any(axis=0)[:, None], vals, 0.0)
    o = np.matmul(e.reshape(-1, L), vis_vals).reshape(e.shape[0], G, D) / l[..., None]
    out[live] = o * out_scale
    lse[live] = m[..., 0] + np.log(l)
    return out, lse


# ----------------------------------------------------------------------------------------
# Materialising the logical K/V of one request from its pages.
# ----------------------------------------------------------------------------------------

def gather_pages(pool, page_ids, length):
    """pool [P, Hkv, ps, D] (float64); logical token j lives in page page_ids[j // ps],
    slot j % ps.  Returns [length, Hkv, D]."""
    ps = pool.shape[2]
    j = np.arange(length)
    pid = np.asarray(page_ids, dtype=np.int64)[j // ps]
    return pool[pid, :, j % ps, :]


def split_pools(kv_cache=None, k_cache=None, v_cache=None):
    """(K pool, V pool) as float64 [P, Hkv, ps, D]; a combined cache [P, 2, Hkv, ps, D] holds
    K at axis-1 index 0 and V at index 1."""
    if kv_cache is not None:
        c = f64(kv_cache)
        return c[:, 0], c[:, 1]
    return f64(k_cache), f64(v_cache)


def valid_token_mask(words_row, length):
    """Bool [length] from one request's uint32 validity words (LSB-first)."""
    j = np.arange(length)
    return ((words_row[j >> 5] >> (j & 31).astype(np.uint32)) & 1).astype(bool)


# ----------------------------------------------------------------------------------------
# [BSA] block-sparse attention over a CSR-paged cache
# ----------------------------------------------------------------------------------------

def block_sparse_attention(q, kv_indptr, kv_indices, block_indptr, block_indices, q_block_size,
                           kv_block_size, seq_lens_kv, *, kv_cache=None, k_cache=None,
                           v_cache=None, kv_valid_bits=None, mask_type="dense", sm_scale=None,
                           rows=None):
    """[BSA] forward: q [B, Sq, Hq, D]; K/V gathered through paged_kv_indptr/indices.

    Row (b, i) with KV head g sees key j iff j < seq_lens_kv[b], j // kv_block_size is
    listed in block_indices[block_indptr[b, g, i // q_block_size] :
    block_indptr[b, g, i // q_block_size + 1]], the validity bit of j is set (when
    kv_valid_bits is given) and, for mask_type "causal", j <= p(i).
    rows: optional list of (b, i) to compute; other rows are returned as NaN.
    Returns O float64 [B, Sq, Hq, D] and LSE float64 [B, Sq, Hq].
    """
    qf = f64(q)
    B, Sq, Hq, D = qf.shape
    Kp, Vp = split_pools(kv_cache, k_cache, v_cache)
    Hkv = Kp.shape[1]
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if sm_scale is None else float(sm_scale)
    indptr, indices = i64(kv_indptr), i64(kv_indices)
    bptr, bidx = i64(block_indptr), i64(block_indices)
    lens = i64(seq_lens_kv)
    words = u32(kv_valid_bits) if kv_valid_bits is not None else None
    qbs, kvbs = int(q_block_size), int(kv_block_size)
    nqb = -(-Sq // qbs)
    want = None
    if rows is not None:
        want = {}
        for b, i in rows:
            want.setdefault(int(b), set()).add(int(i))
    out = np.full((B, Sq, Hq, D), np.nan if rows is not None else 0.0)
    lse = np.full((B, Sq, Hq), np.nan if rows is not None else -np.inf)
    for b in range(B):
        if want is not None and b not in want:
            continue
        L = int(lens[b])
        pages = indices[indptr[b]:indptr[b + 1]]
        K = gather_pages(Kp, pages, L)
        V = gather_pages(Vp, pages, L)
        live = valid_token_mask(words[b], L) if words is not None else np.ones(L, bool)
        for g in range(Hkv):
            for r in range(nqb):
                i_all = np.arange(r * qbs, min((r + 1) * qbs, Sq))
                if want is not None:
                    i_all = np.array([i for i in i_all if i in want[b]], dtype=np.int64)
                if i_all.size == 0:
                    continue
                sel = np.zeros(L, bool)
                for c in bidx[bptr[b, g, r]:bptr[b, g, r + 1]]:
                    sel[c * kvbs:min((c + 1) * kvbs, L)] = True
                sel &= live
                keys = np.nonzero(sel)[0]
                vis = np.ones((i_all.size, keys.size), bool)
                if mask_type == "causal":
                    p = L - Sq + i_all
                    vis &= keys[None, :] <= p[:, None]
                o, s = masked_softmax_attention(qf[b, i_all, g * G:(g + 1) * G], K[keys, g],
                                                V[keys, g], vis, scale)
                out[b, i_all, g * G:(g + 1) * G] = o
                lse[b, i_all, g * G:(g + 1) * G] = s
    return out, lse


# ----------------------------------------------------------------------------------------
# [PRE] packed-Q prefill over separate HND pools with a row-strided page table
# ----------------------------------------------------------------------------------------

def batch_prefill(q, k_cache, v_cache, qo_indptr, block_tables, seq_lens_kv, *,
                  mask_type="dense", window_left=-1, sm_scale=None, output_scale=1.0,
                  rows=None):
    """[PRE] forward: q [total_q, Hq, D]; request b owns rows qo_indptr[b]:qo_indptr[b+1] and
    pages block_tables[b, :].  Key j is visible to local query i iff j < len_kv and, for
    "causal", j <= p(i) and (window_left >= 0) j >= p(i) - window_left.
    rows: optional list of packed row indices.  Returns O [total_q, Hq, D], LSE [total_q, Hq].
    """
    if window_left >= 0 and mask_type != "causal":
        raise ValueError("window_left >= 0 requires the causal mask")
    qf = f64(q)
    T, Hq, D = qf.shape
    Kp, Vp = f64(k_cache), f64(v_cache)
    Hkv = Kp.shape[1]
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if sm_scale is None else float(sm_scale)
    qo = i64(qo_indptr)
    tables = i64(block_tables)
    lens = i64(seq_lens_kv)
    want = set(int(r) for r in rows) if rows is not None else None
    out = np.full((T, Hq, D), np.nan if rows is not None else 0.0)
    lse = np.full((T, Hq), np.nan if rows is not None else -np.inf)
    for b in range(len(lens)):
        r0, r1 = int(qo[b]), int(qo[b + 1])
        loc = np.arange(r1 - r0)
        if want is not None:
            loc = np.array([i for i in loc if (r0 + i) in want], dtype=np.int64)
        if loc.size == 0:
            continue
        L = int(lens[b])
        K = gather_pages(Kp, tables[b], L)
        V = gather_pages(Vp, tables[b], L)
        keys = np.arange(L)
        vis = np.ones((loc.size, L), bool)
        if mask_type == "causal":
            p = L - (r1 - r0) + loc
            vis &= keys[None, :] <= p[:, None]
            if window_left >= 0:
                vis &= keys[None, :] >= (p - window_left)[:, None]
        for g in range(Hkv):
            o, s = masked_softmax_attention(qf[r0 + loc, g * G:(g + 1) * G], K[:, g], V[:, g],
                                            vis, scale, output_scale)
            out[r0 + loc, g * G:(g + 1) * G] = o
            lse[r0 + loc, g * G:(g + 1) * G] = s
    return out, lse


# ----------------------------------------------------------------------------------------
# [DEC] decode over a CSR-paged cache: one query, SQ fixed queries, or packed queries
# ----------------------------------------------------------------------------------------

def batch_decode(query, kv_indptr, kv_indices, seq_lens, *, kv_cache=None, k_cache=None,
                 v_cache=None, bmm1_scale=None, bmm2_scale=1.0, mask_type="dense",
                 window_left=-1, seq_len_q=1, qo_indptr=None, rows=None):
    """[DEC] forward (signature and notes on seq_len_q / qo_indptr).  Query layouts:

      * seq_len_q = 1, no qo_indptr: query [B, Hq, D]; O [B, Hq, D], LSE [B, Hq];
      * seq_len_q = SQ > 1: token-major query [B, SQ, Hq, D]; O and LSE [B, SQ, ...];
      * qo_indptr given: packed query [total_q, Hq, D], request b owning rows
        qo_indptr[b]:qo_indptr[b+1]; O [total_q, Hq, D], LSE [total_q, Hq].

    Query i of a request with nq queries and L keys sits at p = L - nq + i: keys j < L are
    candidates, the causal mask keeps j <= p, and window_left = w >= 0 keeps j >= p - w.
    With one query p = L - 1, so the causal mask keeps every live key.  bmm1_scale is the
    softmax scale (default 1/sqrt(D)); bmm2_scale multiplies the normalised output.
    rows: optional list of request indices to evaluate (the rest is NaN)."""
    if window_left >= 0 and mask_type != "causal":
        raise ValueError("window_left >= 0 requires the causal mask")
    qf = f64(query)
    lens = i64(seq_lens)
    B = lens.size
    if qo_indptr is not None:
        qo = i64(qo_indptr)
        qp = qf
    elif seq_len_q > 1:
        qo = np.arange(B + 1, dtype=np.int64) * seq_len_q
        qp = qf.reshape((B * seq_len_q,) + qf.shape[2:])
    else:
        qo = np.arange(B + 1, dtype=np.int64)
        qp = qf
    T, Hq, D = qp.shape
    Kp, Vp = split_pools(kv_cache, k_cache, v_cache)
    Hkv = Kp.shape[1]
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if bmm1_scale is None else float(bmm1_scale)
    indptr, indices = i64(kv_indptr), i64(kv_indices)
    want = set(int(r) for r in rows) if rows is not None else None
    out = np.full((T, Hq, D), np.nan if rows is not None else 0.0)
    lse = np.full((T, Hq), np.nan if rows is not None else -np.inf)
    for b in range(B):
        if want is not None and b not in want:
            continue
        r0, r1 = int(qo[b]), int(qo[b + 1])
        L = int(lens[b])
        pages = indices[indptr[b]:indptr[b + 1]]
        K = gather_pages(Kp, pages, L)
        V = gather_pages(Vp, pages, L)
        keys = np.arange(L)
        p = L - (r1 - r0) + np.arange(r1 - r0)
        vis = np.ones((r1 - r0, L), bool)
        if mask_type == "causal":
            vis &= keys[None, :] <= p[:, None]
            if window_left >= 0:
                vis &= keys[None, :] >= (p - window_left)[:, None]
        for g in range(Hkv):
            o, s = masked_softmax_attention(qp[r0:r1, g * G:(g + 1) * G], K[:, g], V[:, g],
                                            vis, scale, bmm2_scale)
            out[r0:r1, g * G:(g + 1) * G] = o
            lse[r0:r1, g * G:(g + 1) * G] = s
    if qo_indptr is None and seq_len_q > 1:
        return out.reshape(B, seq_len_q, Hq, D), lse.reshape(B, seq_len_q, Hq)
    return out, lse


def decode_visible_pairs(Hq, seq_lens, q_lens, mask_type="dense", window_left=-1):
    """Visible (query row, query head, key) triples of a [DEC] problem whose request b has
    q_lens[b] queries (the counting rule of the forward above)."""
    lens = i64(seq_lens)
    nq = i64(q_lens)
    qo = np.zeros(lens.size + 1, dtype=np.int64)
    qo[1:] = np.cumsum(nq)
    return prefill_visible_pairs(Hq, qo, lens, mask_type, window_left)


def merge_partials(o_parts, lse_parts):
    """Combine attention results over disjoint key subsets (split-KV).

    o_parts [S, ..., D] are the per-subset normalised outputs and lse_parts [S, ...] their
    natural-log normalisers; LSE = log sum_s exp(LSE_s) and O = sum_s exp(LSE_s - LSE) O_s.
    Subsets with LSE_s = -inf contribute nothing; if all are -inf the result is 0 / -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe)
    tot = w.sum(axis=0)
    lse = np.where(tot > 0, m_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    o = np.where((tot > 0)[..., None],
                 (w[..., None] * np.nan_to_num(o_parts)).sum(axis=0)
                 / np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    return o, lse


# ----------------------------------------------------------------------------------------
# [QSA] per-query block-bitmap attention on packed, non-paged K/V
# ----------------------------------------------------------------------------------------

def token_block_map(block_first, block_last, T):
    """Global block holding each packed token (-1 where no block covers it)."""
    first, last = i64(block_first), i64(block_last)
    blk = np.full(T, -1, dtype=np.int64)
    for g in range(first.size):
        blk[first[g]:last[g] + 1] = g
    return blk


def qsa_forward(q, k, v, sel_blocks, lo, hi, blk_base, tok_base, block_first, block_last,
                scale=0.0625, block_size=4, rows=None):
    """[QSA] forward.  Query token t with KV head g sees key token j iff lo[t] <= j <= hi[t]
    and sel_blocks[t, blk(j)] != 0, where blk(j) is the global block whose inclusive span
    [block_first, block_last] holds j.  blk_base / tok_base do not change the result.
    Returns (out bf16 [T, Hq, D], out_fp32 [T, Hq, D], lse fp32 [Hq, T]) as torch tensors
    plus the float64 output and LSE ([T, Hq, D], [Hq, T]).
    """
    if block_size != 4:
        raise ValueError("block_size must be 4")
    qf, kf, vf = f64(q), f64(k), f64(v)
    T, Hq, D = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    sel = sel_blocks.numpy() if isinstance(sel_blocks, torch.Tensor) else np.asarray(sel_blocks)
    lo_, hi_ = i64(lo), i64(hi)
    blk = token_block_map(block_first, block_last, T)
    ts = range(T) if rows is None else [int(t) for t in rows]
    out = np.full((T, Hq, D), np.nan if rows is not None else 0.0)
    lse = np.full((Hq, T), np.nan if rows is not None else -np.inf)
    for t in ts:
        j = np.arange(max(lo_[t], 0), min(hi_[t], T - 1) + 1)
        j = j[blk[j] >= 0]
        j = j[sel[t, blk[j]] != 0]
        vis = np.ones((1, j.size), bool)
        for g in range(Hkv):
            o, s = masked_softmax_attention(qf[t, None, g * G:(g + 1) * G], kf[j, g], vf[j, g],
                                            vis, float(scale))
            out[t, g * G:(g + 1) * G] = o[0]
            lse[g * G:(g + 1) * G, t] = s[0]
    return out, lse


def qsa_indexed_forward(q, k, v, sel_indices, lo, hi, block_first, block_last, scale=0.0625,
                        block_size=4, rows=None):
    """Indexed form of [QSA] (the notes name qsa_indexed_forward for callers that already hold
    each query's selected block indices).  Row t of sel_indices [T, K] lists global block ids;
    entries outside [0, NB) are unused.  Query token t sees key token j iff lo[t] <= j <= hi[t]
    and j lies in the span [block_first[g], block_last[g]] of a listed block g (the listed
    blocks of a row are distinct).  Returns the float64 output [T, Hq, D] and LSE [Hq, T]."""
    if block_size != 4:
        raise ValueError("block_size must be 4")
    qf, kf, vf = f64(q), f64(k), f64(v)
    T, Hq, D = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    idx = sel_indices.numpy() if isinstance(sel_indices, torch.Tensor) else np.asarray(sel_indices)
    first, last = i64(block_first), i64(block_last)
    NB = first.size
    lo_, hi_ = i64(lo), i64(hi)
    ts = range(T) if rows is None else [int(t) for t in rows]
    out = np.full((T, Hq, D), np.nan if rows is not None else 0.0)
    lse = np.full((Hq, T), np.nan if rows is not None else -np.inf)
    for t in ts:
        spans = []
        for g in idx[t]:
            g = int(g)
            if 0 <= g < NB:
                a, e = max(first[g], lo_[t]), min(last[g], hi_[t])
                if a <= e:
                    spans.append(np.arange(a, e + 1))
        j = np.sort(np.concatenate(spans)) if spans else np.zeros(0, np.int64)
        vis = np.ones((1, j.size), bool)
        for g in range(Hkv):
            o, s = masked_softmax_attention(qf[t, None, g * G:(g + 1) * G], kf[j, g], vf[j, g],
                                            vis, float(scale))
            out[t, g * G:(g + 1) * G] = o[0]
            lse[g * G:(g + 1) * G, t] = s[0]
    return out, lse


# ----------------------------------------------------------------------------------------
# [SAGE] prequantized block-sparse attention
# ----------------------------------------------------------------------------------------

def fp8_e4m3_to_f64(codes):
    """Decode FP8 E4M3 bytes (the e4m3fn format: 1 sign, 4 exponent bits with bias 7, 3
    mantissa bits, no infinities, S.1111.111 = NaN) to float64 (torch's conversion)."""
    t = codes if isinstance(codes, torch.Tensor) else torch.from_numpy(np.asarray(codes))
    return t.contiguous().view(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def sage_block_sparse_attention(q_int8, k_int8, v_fp8, q_scale, k_scale, v_scale,
                                q2k_block_index, block_sparse_num, block_sizes=None,
                                q2k_block_nums=None, softmax_scale=None):
    """[SAGE] forward on the dequantized values (signature, parameters and notes).

    q = q_int8 * q_scale[b, h, i // 32] (four scales per 128 queries), k = k_int8 *
    k_scale[b, h, j // 64] (one per 64-key block), v[j, d] = e4m3(v_fp8[b, h, d, j]) *
    v_scale[b, h, d].  Query block r = i // 64 selects the first n_r entries of
    q2k_block_index[b, h, r] (n_r = q2k_block_nums[b, h, r], else block_sparse_num); key j of
    selected block c is visible iff j < Sk and j - 64 c < block_sizes[c] (block_sizes given as
    [NB], [B, NB] or [B, H, NB]; all 64 when omitted).  No causal mask (non-causal forward).
    O = softmax(softmax_scale * q k^T) v over the visible keys; a row with none gives exactly
    0.  Returns O [B, H, Sq, 128] in float64."""
    qi = f64(q_int8)
    ki = f64(k_int8)
    vf = fp8_e4m3_to_f64(v_fp8)
    B, H, Sq, D = qi.shape
    Sk = ki.shape[2]
    qs, ks, vs = f64(q_scale), f64(k_scale), f64(v_scale)
    idx = i64(q2k_block_index)
    NB = -(-Sk // 64)
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    if block_sizes is None:
        bs = np.full((B, H, NB), 64, dtype=np.int64)
    else:
        bsz = i64(block_sizes)
        # [NB] is shared by all (b, h); [B, NB] is per batch, shared by the heads
        if bsz.ndim == 1:
            full = bsz[None, None, :]
        elif bsz.ndim == 2:
            full = bsz[:, None, :]
        else:
            full = bsz
        bs = np.broadcast_to(full, (B, H, bsz.shape[-1]))
    nums = i64(q2k_block_nums) if q2k_block_nums is not None else None
    out = np.zeros((B, H, Sq, D))
    for b in range(B):
        for h in range(H):
            q = qi[b, h] * qs[b, h][np.arange(Sq) // 32][:, None]
            k = ki[b, h] * ks[b, h][np.arange(Sk) // 64][:, None]
            v = vf[b, h, :, :Sk].T * vs[b, h][None, :]
            for r in range(-(-Sq // 64)):
                rows = np.arange(r * 64, min(Sq, r * 64 + 64))
                n = int(nums[b, h, r]) if nums is not None else int(block_sparse_num)
                keys = []
                for c in idx[b, h, r, :n]:
                    c = int(c)
                    if 0 <= c < NB:
                        keys.extend(j for j in range(64 * c, min(Sk, 64 * c + 64))
                                    if j - 64 * c < bs[b, h, c])
                keys = np.array(sorted(keys), dtype=np.int64)
                vis = np.ones((rows.size, keys.size), bool)
                o, _ = masked_softmax_attention(q[rows][:, None, :], k[keys], v[keys], vis, scale)
                out[b, h, rows] = o[:, 0]
    return out


# ----------------------------------------------------------------------------------------
# Work accounting: exact visible-pair counts (FLOPs = 4 * D * pairs).
# ----------------------------------------------------------------------------------------

def bsr_visible_pairs(B, Sq, Hq, Hkv, block_indptr, block_indices, q_block_size, kv_block_size,
                      seq_lens_kv, kv_valid_bits=None, mask_type="dense"):
    """Number of visible (row, query head, key) triples of a [BSA] problem."""
    G = Hq // Hkv
    bptr, bidx, lens = i64(block_indptr), i64(block_indices), i64(seq_lens_kv)
    words = u32(kv_valid_bits) if kv_valid_bits is not None else None
    qbs, kvbs = int(q_block_size), int(kv_block_size)
    total = 0
    for b in range(B):
        L = int(lens[b])
        live = valid_token_mask(words[b], L) if words is not None else np.ones(L, bool)
        for g in range(Hkv):
            for r in range(-(-Sq // qbs)):
                sel = np.zeros(L, bool)
                for c in bidx[bptr[b, g, r]:bptr[b, g, r + 1]]:
                    sel[c * kvbs:min((c + 1) * kvbs, L)] = True
                sel &= live
                keys = np.nonzero(sel)[0]
                i = np.arange(r * qbs, min((r + 1) * qbs, Sq))
                if mask_type == "causal":
                    p = L - Sq + i
                    total += int(np.searchsorted(keys, p, side="right").sum()) * G
                else:
                    total += keys.size * i.size * G
    return total


def prefill_visible_pairs(Hq, qo_indptr, seq_lens_kv, mask_type="dense", window_left=-1):
    qo, lens = i64(qo_indptr), i64(seq_lens_kv)
    total = 0
    for b in range(len(lens)):
        nq, L = int(qo[b + 1] - qo[b]), int(lens[b])
        if mask_type != "causal":
            total += nq * L
            continue
        p = L - nq + np.arange(nq)
        hi = np.minimum(p, L - 1) + 1
        lo = np.maximum(p - window_left, 0) if window_left >= 0 else np.zeros_like(p)
        total += int(np.maximum(hi - lo, 0).sum())
    return total * Hq


def qsa_visible_pairs(Hq, sel_blocks, lo, hi, block_first, block_last):
    sel = sel_blocks.numpy() if isinstance(sel_blocks, torch.Tensor) else np.asarray(sel_blocks)
    lo_, hi_ = i64(lo), i64(hi)
    first, last = i64(block_first), i64(block_last)
    T = lo_.size
    total = 0
    for t in range(T):
        g = np.nonzero(sel[t])[0]
        a = np.maximum(first[g], lo_[t])
        e = np.minimum(last[g], hi_[t])
        total += int(np.maximum(e - a + 1, 0).sum())
    return total * Hq


def qsa_indexed_visible_pairs(Hq, sel_indices, lo, hi, block_first, block_last):
    idx = sel_indices.numpy() if isinstance(sel_indices, torch.Tensor) else np.asarray(sel_indices)
    lo_, hi_ = i64(lo), i64(hi)
    first, last = i64(block_first), i64(block_last)
    NB = first.size
    total = 0
    for t in range(lo_.size):
        g = idx[t].astype(np.int64)
        g = g[(g >= 0) & (g < NB)]
        total += int(np.maximum(np.minimum(last[g], hi_[t]) - np.maximum(first[g], lo_[t]) + 1,
                                0).sum())
    return total * Hq
