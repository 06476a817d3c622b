"""Seeded synthetic inputs for paged-KV attention.

This module only draws inputs: page pools, page tables, query tensors and the sparse
selections (BSR rows, per-query block bitmaps).  It holds none of the attention
arithmetic; the same generated tensors feed the CUDA path and the float64 checker.

All randomness comes from a seeded ``torch.Generator`` (CPU) and a seeded
``numpy.random.Generator``; every tensor is created on the CPU.  Q/K/V are i.i.d.
N(0, 1) rounded to bf16.  Pages that no request owns, table entries past a request's
live pages, and the slots past the last live token of every request's last page are
filled with NaN, so that a read of memory the method never uses shows up in the output.

Workload names follow the tensor contracts of the FlashInfer pages
``block_sparse_attention_with_paged_kv_cache``, ``batch_prefill_with_paged_kv_cache``,
``prims_ts_batch_decode_with_kv_cache`` and ``qsa_forward``.
"""
from __future__ import annotations

import math

import numpy as np
import torch

NAN = float("nan")


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def assign_pages(gen: torch.Generator, lens, page_size: int, num_pages: int | None = None,
                 spare_frac: float = 0.10):
    """Give each request disjoint physical page IDs from one seeded permutation.

    Request b takes the next ceil(len_b / page_size) entries of the permutation.
    Returns (num_pages, list of int64 page-id tensors, spare page ids).
    """
    need = [_ceil_div(int(n), page_size) for n in lens]
    total = sum(need)
    if num_pages is None:
        num_pages = max(1, math.ceil(total * (1.0 + spare_frac)))
    if total > num_pages:
        raise ValueError("not enough pages")
    perm = torch.randperm(num_pages, generator=gen)
    out, off = [], 0
    for n in need:
        out.append(perm[off:off + n].clone())
        off += n
    spare = perm[off:].clone()
    return num_pages, out, spare


def _poison(pool_k: torch.Tensor, pool_v: torch.Tensor, pages, lens, spare, page_size: int):
    """NaN-fill spare pages and the unused tail slots of each request's last page.

    pool_k / pool_v are [P, Hkv, ps, D] views (for a combined cache, the K and V halves).
    """
    if spare.numel():
        pool_k[spare] = NAN
        pool_v[spare] = NAN
    for pids, n in zip(pages, lens):
        n = int(n)
        if pids.numel() == 0:
            continue
        tail = n - (pids.numel() - 1) * page_size
        if tail < page_size:
            last = int(pids[-1])
            pool_k[last, :, tail:, :] = NAN
            pool_v[last, :, tail:, :] = NAN


def _csr(pages):
    indptr = [0]
    for p in pages:
        indptr.append(indptr[-1] + p.numel())
    indices = torch.cat(pages) if pages else torch.zeros(0, dtype=torch.int64)
    return (torch.tensor(indptr, dtype=torch.int32), indices.to(torch.int32))


def make_page_pools(gen, lens, Hkv, D, page_size, num_pages=None, combined=False,
                    spare_frac=0.10, poison=True):
    """Random K/V page pools plus a per-request page assignment.

    Returns dict(k_cache, v_cache | kv_cache, pages, spare, num_pages).  Separate pools are
    [P, Hkv, ps, D]; a combined cache is [P, 2, Hkv, ps, D] with index 0 = K, 1 = V.
    """
    P, pages, spare = assign_pages(gen, lens, page_size, num_pages, spare_frac)
    out = {"pages": pages, "spare": spare, "num_pages": P}
    if combined:
        cache = _normal_bf16(gen, (P, 2, Hkv, page_size, D))
        if poison:
            _poison(cache[:, 0], cache[:, 1], pages, lens, spare, page_size)
        out["kv_cache"] = cache
    else:
        k = _normal_bf16(gen, (P, Hkv, page_size, D))
        v = _normal_bf16(gen, (P, Hkv, page_size, D))
        if poison:
            _poison(k, v, pages, lens, spare, page_size)
        out["k_cache"], out["v_cache"] = k, v
    return out


# ----------------------------------------------------------------------------------------
# Block-sparse (BSR) selections
# ----------------------------------------------------------------------------------------

def _qblock_positions(L: int, Sq: int, r: int, qbs: int):
    """Logical positions of the first and last query of q-block r (queries are the last Sq
    positions of the request's KV sequence)."""
    first = L - Sq + r * qbs
    last = L - Sq + min((r + 1) * qbs, Sq) - 1
    return first, last


def bsr_select(rng: np.random.Generator, B, Hkv, Sq, seq_lens, qbs, kvbs, policy, **kw):
    """Build block_indptr [B, Hkv, nqb+1] and block_indices (sorted per row).

    policy:
      "diag_bernoulli": blocks meeting [p_first, p_last] kept; every earlier block (entirely
          before p_first) kept with probability kw["p"] (default 0.5).
      "sink_recent_random": block 0, the kw["n_recent"] most recent blocks up to
          p_last // kvbs, and kw["n_random"] distinct uniform draws from the blocks between.
      "causal_all": every block that meets [0, p_last].
      "all": every block that meets [0, len).
      "random": each block of [0, ceil(len/kvbs)) kept with probability kw["p"].
      "empty": no blocks.
    Offsets run over all (b, g, r) rows in row-major order.
    """
    nqb = _ceil_div(Sq, qbs)
    indptr = np.zeros((B, Hkv, nqb + 1), dtype=np.int64)
    rows = []
    off = 0
    for b in range(B):
        L = int(seq_lens[b])
        nblk = _ceil_div(L, kvbs)
        for g in range(Hkv):
            for r in range(nqb):
                indptr[b, g, r] = off
                first, last = _qblock_positions(L, Sq, r, qbs)
                if policy == "diag_bernoulli":
                    p = kw.get("p", 0.5)
                    c0, c1 = max(first, 0) // kvbs, max(last, 0) // kvbs
                    earlier = np.arange(0, c0)
                    keep = earlier[rng.random(earlier.size) < p]
                    sel = np.concatenate([keep, np.arange(c0, c1 + 1)])
                elif policy == "sink_recent_random":
                    n_recent, n_random = kw["n_recent"], kw["n_random"]
                    lastb = max(last, 0) // kvbs
                    recent = np.arange(max(0, lastb - n_recent + 1), lastb + 1)
                    pool = np.arange(1, max(1, lastb - n_recent + 1))
                    k = min(n_random, pool.size)
                    extra = rng.choice(pool, size=k, replace=False) if k else np.zeros(0, np.int64)
                    sel = np.unique(np.concatenate([[0], recent, extra]))
                elif policy == "causal_all":
                    sel = np.arange(0, max(last, -1) // kvbs + 1) if last >= 0 else np.zeros(0)
                elif policy == "all":
                    sel = np.arange(0, nblk)
                elif policy == "random":
                    cand = np.arange(0, nblk)
                    sel = cand[rng.random(cand.size) < kw.get("p", 0.5)]
                elif policy == "empty":
                    sel = np.zeros(0)
                else:
                    raise ValueError(policy)
                sel = np.unique(sel.astype(np.int64))
                rows.append(sel)
                off += sel.size
            indptr[b, g, nqb] = off
    indices = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    return (torch.from_numpy(indptr.astype(np.int32)),
            torch.from_numpy(indices.astype(np.int32)))


def valid_bits_drop(rng: np.random.Generator, seq_lens, max_seq_len: int, frac: float):
    """uint32 token-validity words [B, ceil(max_seq_len/32)] (stored as int32 bit patterns).

    Bit (j & 31) of word (j >> 5) is 1 for a live token; a seeded round(frac * len) of each
    request's tokens are cleared; bits at j >= len stay 0.
    """
    B = len(seq_lens)
    W = _ceil_div(max_seq_len, 32)
    words = np.zeros((B, W), dtype=np.uint32)
    for b in range(B):
        L = int(seq_lens[b])
        live = np.ones(L, dtype=bool)
        k = int(round(frac * L))
        if k:
            live[rng.choice(L, size=k, replace=False)] = False
        bits = np.zeros(W * 32, dtype=np.uint32)
        bits[:L] = live
        words[b] = (bits.reshape(W, 32) << np.arange(32, dtype=np.uint32)).sum(axis=1,
                                                                              dtype=np.uint32)
    return torch.from_numpy(words.view(np.int32))


def make_bsr_problem(seed, B, Sq, Hq, Hkv, D, seq_lens, page_size, qbs, kvbs, *,
                     num_pages=None, combined=False, policy="diag_bernoulli",
                     valid_drop=0.0, mask_type="causal", spare_frac=0.10, **policy_kw):
    """A complete input set for block-sparse paged attention (fixed-Q [B, Sq, Hq, D])."""
    gen = _gen(seed)
    rng = np.random.default_rng(seed)
    seq_lens = [int(x) for x in seq_lens]
    q = _normal_bf16(gen, (B, Sq, Hq, D))
    pools = make_page_pools(gen, seq_lens, Hkv, D, page_size, num_pages, combined, spare_frac)
    kv_indptr, kv_indices = _csr(pools["pages"])
    block_indptr, block_indices = bsr_select(rng, B, Hkv, Sq, seq_lens, qbs, kvbs, policy,
                                             **policy_kw)
    max_len = max(seq_lens) if seq_lens else 0
    prob = dict(form="bsr", q=q, kv_indptr=kv_indptr, kv_indices=kv_indices,
                block_indptr=block_indptr, block_indices=block_indices,
                q_block_size=qbs, kv_block_size=kvbs, page_size=page_size,
                seq_lens_kv=torch.tensor(seq_lens, dtype=torch.int32),
                max_seq_len_kv=max_len, mask_type=mask_type,
                sm_scale=1.0 / math.sqrt(D), num_pages=pools["num_pages"],
                kv_valid_bits=None, spare_pages=pools["spare"])
    if combined:
        prob["kv_cache"] = pools["kv_cache"]
    else:
        prob["k_cache"], prob["v_cache"] = pools["k_cache"], pools["v_cache"]
    if valid_drop > 0:
        prob["kv_valid_bits"] = valid_bits_drop(rng, seq_lens, max_len, valid_drop)
    return prob


# ----------------------------------------------------------------------------------------
# Packed-Q paged prefill
# ----------------------------------------------------------------------------------------

def make_prefill_problem(seed, q_lens, prefix_lens, Hq, Hkv, D, page_size, *, mask_type="causal",
                         window_left=-1, output_scale=1.0, spare_frac=0.10):
    """Packed-Q prefill over separate HND pools with a row-strided block_tables [B, C].

    KV length = query length + cached prefix; queries are the last q_len KV positions.
    Table entries past a request's live pages point at a spare (NaN) page.
    """
    gen = _gen(seed)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(a) + int(b) for a, b in zip(q_lens, prefix_lens)]
    B = len(q_lens)
    total_q = sum(q_lens)
    q = _normal_bf16(gen, (total_q, Hq, D))
    need = [_ceil_div(n, page_size) for n in kv_lens]
    P = max(1, math.ceil(sum(need) * (1.0 + spare_frac))) + 1
    pools = make_page_pools(gen, kv_lens, Hkv, D, page_size, P, False)
    spare = pools["spare"]
    filler = int(spare[0]) if spare.numel() else 0
    C = max(1, max(need) if need else 1)
    tables = torch.full((B, C), filler, dtype=torch.int32)
    for b, p in enumerate(pools["pages"]):
        tables[b, :p.numel()] = p.to(torch.int32)
    qo_indptr = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32))
    return dict(form="prefill", q=q, k_cache=pools["k_cache"], v_cache=pools["v_cache"],
                qo_indptr=qo_indptr, block_tables=tables,
                seq_lens_kv=torch.tensor(kv_lens, dtype=torch.int32), page_size=page_size,
                mask_type=mask_type, window_left=int(window_left), sm_scale=1.0 / math.sqrt(D),
                output_scale=float(output_scale), num_pages=P, spare_pages=spare)


# ----------------------------------------------------------------------------------------
# CSR paged decode
# ----------------------------------------------------------------------------------------

def make_decode_problem(seed, seq_lens, Hq, Hkv, D, page_size, *, combined=True, spare_frac=0.10,
                        mask_type="dense", window_left=-1, bmm2_scale=1.0, seq_len_q=1,
                        q_lens=None):
    """Decode over a CSR page table, combined or separate cache.  Queries: [B, Hq, D] for
    one query per request; [B, SQ, Hq, D] for seq_len_q = SQ > 1; packed [total_q, Hq, D]
    with qo_indptr when q_lens (queries of each request) is given."""
    gen = _gen(seed)
    seq_lens = [int(x) for x in seq_lens]
    B = len(seq_lens)
    if q_lens is not None:
        q_lens = [int(x) for x in q_lens]
        if len(q_lens) != B or min(q_lens, default=1) < 1:
            raise ValueError("q_lens needs one positive count per request")
        q = _normal_bf16(gen, (sum(q_lens), Hq, D))
        qo = torch.zeros(B + 1, dtype=torch.int32)
        qo[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
        sq, max_sq = 1, max(q_lens, default=1)
    elif seq_len_q > 1:
        q = _normal_bf16(gen, (B, seq_len_q, Hq, D))
        qo, sq, max_sq = None, int(seq_len_q), int(seq_len_q)
    else:
        q = _normal_bf16(gen, (B, Hq, D))
        qo, sq, max_sq = None, 1, 1
    pools = make_page_pools(gen, seq_lens, Hkv, D, page_size, None, combined, spare_frac)
    kv_indptr, kv_indices = _csr(pools["pages"])
    prob = dict(form="decode", q=q, kv_indptr=kv_indptr, kv_indices=kv_indices,
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                max_seq_len=max(seq_lens) if seq_lens else 1, page_size=page_size,
                mask_type=mask_type, window_left=int(window_left),
                sm_scale=1.0 / math.sqrt(D), bmm2_scale=float(bmm2_scale),
                seq_len_q=sq, qo_indptr=qo, max_seq_len_q=max_sq,
                q_lens=q_lens if q_lens is not None else [sq] * B,
                num_pages=pools["num_pages"], spare_pages=pools["spare"])
    if combined:
        prob["kv_cache"] = pools["kv_cache"]
    else:
        prob["k_cache"], prob["v_cache"] = pools["k_cache"], pools["v_cache"]
    return prob


# ----------------------------------------------------------------------------------------
# Per-query block bitmap (packed, non-paged K/V)
# ----------------------------------------------------------------------------------------

def make_qsa_problem(seed, seq_lens, Hq, Hkv, D, *, block_size=4, n_near=16, n_random=256,
                     scale=None):
    """Packed sequences with a per-query block bitmap.

    Block numbering restarts at each sequence (every sequence length is a multiple of the
    block size, so no block straddles two sequences); global block g covers tokens
    [block_size*g, block_size*g + block_size - 1].  lo[t] = first token of t's sequence,
    hi[t] = t.  Row t selects the block holding t and the n_near - 1 blocks before it
    (clipped at the sequence start) plus min(n_random, available) distinct uniform blocks
    earlier in the same sequence.
    """
    gen = _gen(seed)
    rng = np.random.default_rng(seed)
    seq_lens = [int(x) for x in seq_lens]
    for n in seq_lens:
        if n % block_size:
            raise ValueError("sequence lengths must be multiples of block_size")
    T = sum(seq_lens)
    NB = T // block_size
    q = _normal_bf16(gen, (T, Hq, D))
    k = _normal_bf16(gen, (T, Hkv, D))
    v = _normal_bf16(gen, (T, Hkv, D))
    sel = np.zeros((T, NB), dtype=np.uint8)
    lo = np.zeros(T, np.int32)
    hi = np.arange(T, dtype=np.int32)
    tok_base = np.zeros(T, np.int32)
    blk_base = np.zeros(T, np.int32)
    t0 = 0
    for n in seq_lens:
        nb = n // block_size
        b0 = t0 // block_size
        loc = np.arange(n) // block_size                      # local block of each query
        lo[t0:t0 + n] = t0
        tok_base[t0:t0 + n] = t0
        blk_base[t0:t0 + n] = b0
        rows = np.arange(t0, t0 + n)
        for d in range(n_near):                               # nearest blocks
            lb = loc - d
            ok = lb >= 0
            sel[rows[ok], b0 + lb[ok]] = 1
        avail = np.maximum(loc - n_near + 1, 0)               # earlier blocks: [0, avail)
        if n_random > 0 and nb > n_near:
            chunk = 2048
            for s in range(0, n, chunk):
                e = min(n, s + chunk)
                u = rng.random((e - s, nb))
                u[np.arange(nb)[None, :] >= avail[s:e, None]] = np.inf
                kk = min(n_random, nb)
                part = np.argpartition(u, kk - 1, axis=1)[:, :kk]
                take = np.take_along_axis(u, part, axis=1) < np.inf
                rr = np.repeat(rows[s:e, None], kk, axis=1)
                sel[rr[take], b0 + part[take]] = 1
        t0 += n
    block_first = (np.arange(NB) * block_size).astype(np.int32)
    block_last = (block_first + block_size - 1).astype(np.int32)
    return dict(form="qsa", q=q, k=k, v=v, sel_blocks=torch.from_numpy(sel),
                lo=torch.from_numpy(lo), hi=torch.from_numpy(hi),
                blk_base=torch.from_numpy(blk_base), tok_base=torch.from_numpy(tok_base),
                block_first=torch.from_numpy(block_first),
                block_last=torch.from_numpy(block_last),
                scale=(1.0 / math.sqrt(D)) if scale is None else float(scale),
                block_size=block_size)


def make_qsa_indexed_problem(seed, seq_lens, Hq, Hkv, D, *, block_size=4, n_near=16,
                             n_random=256, scale=None, extra_cols=0, junk=0.0):
    """The selection of make_qsa_problem given as index rows (the indexed form):
    sel_indices [T, K] int32, row t holding its selected global block ids and -1 for unused
    entries, all in a seeded random order.  K = the largest row count + extra_cols.  A
    fraction `junk` of the unused entries hold instead the id of a block past hi[t] (a
    listed block with no visible key)."""
    p = make_qsa_problem(seed, seq_lens, Hq, Hkv, D, block_size=block_size, n_near=n_near,
                         n_random=n_random, scale=scale)
    sel = p["sel_blocks"].numpy()
    T, NB = sel.shape
    rng = np.random.default_rng(seed + 7)
    r, c = np.nonzero(sel)
    counts = np.bincount(r, minlength=T)
    K = max(1, int(counts.max(initial=0)) + int(extra_cols))
    start = np.concatenate([[0], np.cumsum(counts)])
    idx = np.full((T, K), -1, dtype=np.int32)
    idx[r, np.arange(r.size) - start[r]] = c
    if junk > 0:
        hi_blk = p["hi"].numpy().astype(np.int64) // block_size
        free = np.arange(K)[None, :] >= counts[:, None]
        pick = free & (rng.random((T, K)) < junk)
        cand = hi_blk[:, None] + 1 + rng.integers(0, 8, size=(T, K))
        pick &= cand < NB
        idx[pick] = cand[pick].astype(np.int32)
    idx = np.take_along_axis(idx, np.argsort(rng.random((T, K)), axis=1), axis=1)
    p = dict(p, form="qsa_indexed", sel_indices=torch.from_numpy(np.ascontiguousarray(idx)))
    del p["sel_blocks"]
    return p


# ----------------------------------------------------------------------------------------
# Prequantized block-sparse attention (int8 Q/K, FP8 E4M3 V)
# ----------------------------------------------------------------------------------------

def make_sage_problem(seed, B, H, Sq, Sk, *, capacity=8, uniform=None, sizes="none",
                      empty_rows=0.0, D=128):
    """Q, K, V drawn N(0, 1) and quantized as a Sage quantizer would: Q to int8 with one scale
    per 32 queries, K to int8 with one scale per 64-key block (scale = max |x| / 127, round to
    nearest), V to FP8 E4M3 with one scale per channel (max |v| / 448), stored HDS
    [B, H, D, ceil(Sk / 64) * 64] (the padding columns are 0).  Query block r of (b, h) selects
    distinct uniform KV blocks: `uniform` of them each (block_sparse_num) or a per-row count
    uniform in [0, capacity] (q2k_block_nums; a fraction empty_rows of rows select none).
    sizes: "none" (block_sizes omitted), "nb" [NB], "bnb" [B, NB] or "bhnb" [B, H, NB] with
    uniform valid-token counts in [1, 64] (the last block never above Sk - 64 (NB - 1))."""
    gen = _gen(seed)
    rng = np.random.default_rng(seed)
    QB, NB = -(-Sq // 64), -(-Sk // 64)
    q = torch.randn((B, H, Sq, D), generator=gen, dtype=torch.float32)
    k = torch.randn((B, H, Sk, D), generator=gen, dtype=torch.float32)
    v = torch.randn((B, H, Sk, D), generator=gen, dtype=torch.float32)
    QG = -(-Sq // 128) * 4
    qp = torch.zeros((B, H, QG * 32, D))
    qp[:, :, :Sq] = q
    q_scale = (qp.abs().reshape(B, H, QG, 32 * D).amax(-1) / 127.0).clamp_min(1e-8)
    q_int8 = torch.round(qp / q_scale.repeat_interleave(32, dim=2)[..., None])[:, :, :Sq]
    kp = torch.zeros((B, H, NB * 64, D))
    kp[:, :, :Sk] = k
    k_scale = (kp.abs().reshape(B, H, NB, 64 * D).amax(-1) / 127.0).clamp_min(1e-8)
    k_int8 = torch.round(kp / k_scale.repeat_interleave(64, dim=2)[..., None])[:, :, :Sk]
    v_scale = (v.abs().amax(2) / 448.0).clamp_min(1e-8)                      # [B, H, D]
    vq = (v / v_scale[:, :, None, :]).to(torch.float8_e4m3fn)               # [B, H, Sk, D]
    v_hds = torch.zeros((B, H, D, NB * 64), dtype=torch.uint8)
    v_hds[:, :, :, :Sk] = vq.view(torch.uint8).transpose(2, 3)
    cap = capacity if uniform is None else max(capacity, uniform)
    idx = np.zeros((B, H, QB, cap), dtype=np.int32)
    nums = np.zeros((B, H, QB), dtype=np.int32)
    for b in range(B):
        for h in range(H):
            for r in range(QB):
                n = uniform if uniform is not None else int(rng.integers(0, min(capacity, NB) + 1))
                if uniform is None and rng.random() < empty_rows:
                    n = 0
                n = min(n, NB)
                idx[b, h, r, :n] = rng.choice(NB, size=n, replace=False)
                idx[b, h, r, n:] = rng.integers(0, NB, size=cap - n)   # unused entries
                nums[b, h, r] = n
    last = Sk - 64 * (NB - 1)
    block_sizes = None
    if sizes != "none":
        shape = {"nb": (NB,), "bnb": (B, NB), "bhnb": (B, H, NB)}[sizes]
        bsz = rng.integers(1, 65, size=shape).astype(np.int32)
        bsz[..., NB - 1] = np.minimum(bsz[..., NB - 1], last)
        block_sizes = torch.from_numpy(bsz)
    return dict(form="sage", q_int8=q_int8.to(torch.int8), k_int8=k_int8.to(torch.int8),
                v_fp8=v_hds, q_scale=q_scale.float(), k_scale=k_scale.float(),
                v_scale=v_scale.float(), q2k_block_index=torch.from_numpy(idx),
                block_sparse_num=int(uniform) if uniform is not None else 0,
                q2k_block_nums=None if uniform is not None else torch.from_numpy(nums),
                block_sizes=block_sizes, softmax_scale=1.0 / math.sqrt(D), Sq=Sq, Sk=Sk)


# ----------------------------------------------------------------------------------------
# The named workloads
# ----------------------------------------------------------------------------------------

def tiny_bsr(seed=1001):
    """Tiny block-sparse paged prefill: B=2, Hq=8, Hkv=2, D=128, lens {256, 200}, Sq=128,
    separate pools [64, 2, 16, 128], q/kv block 64, diagonal + p=0.5 earlier, causal."""
    return make_bsr_problem(seed, B=2, Sq=128, Hq=8, Hkv=2, D=128, seq_lens=[256, 200],
                            page_size=16, qbs=64, kvbs=64, num_pages=64, combined=False,
                            policy="diag_bernoulli", p=0.5, mask_type="causal")


def decode_b64(seed=1002):
    """Paged decode: B=64, Hq=32, Hkv=8, D=128, lens U[512, 8192], combined cache ps=16,
    +10% spare pages, CSR table, dense mask."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=64, endpoint=True)
    return make_decode_problem(seed, lens, Hq=32, Hkv=8, D=128, page_size=16, combined=True)


def decode_b64_sq4(seed=1002, seq_len_q=4):
    """Multi-query decode (speculative verification): the decode_b64 cache and lengths with
    seq_len_q = 4 queries per request, query [64, 4, 32, 128], causal mask."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=64, endpoint=True)
    return make_decode_problem(seed, lens, Hq=32, Hkv=8, D=128, page_size=16, combined=True,
                               mask_type="causal", seq_len_q=seq_len_q)


def prefill_b16(seed=1003, window_left=-1):
    """Dense causal packed-Q prefill: B=16, q_len U[128, 2048], prefix U[0, 2048],
    Hq=32, Hkv=8, D=128, separate HND pools ps=32, row-strided block_tables."""
    rng = np.random.default_rng(seed)
    q_lens = rng.integers(128, 2048, size=16, endpoint=True)
    prefix = rng.integers(0, 2048, size=16, endpoint=True)
    return make_prefill_problem(seed, q_lens, prefix, Hq=32, Hkv=8, D=128, page_size=32,
                                mask_type="causal", window_left=window_left)


def prefill_b16_d256(seed=1003, window_left=-1):
    """prefill_b16 (the same query lengths, prefixes and heads) with head dimension 256."""
    rng = np.random.default_rng(seed)
    q_lens = rng.integers(128, 2048, size=16, endpoint=True)
    prefix = rng.integers(0, 2048, size=16, endpoint=True)
    return make_prefill_problem(seed, q_lens, prefix, Hq=32, Hkv=8, D=256, page_size=32,
                                mask_type="causal", window_left=window_left)


def long_bsr(seed=1004, S=65536, Hq=64, Hkv=8):
    """Long-context block-sparse prefill: B=1, Sq=Skv=S, page 64, q block 128, kv block 64,
    sink + 16 recent + 48 random earlier blocks per row, causal, 1% invalid tokens."""
    return make_bsr_problem(seed, B=1, Sq=S, Hq=Hq, Hkv=Hkv, D=128, seq_lens=[S], page_size=64,
                            qbs=128, kvbs=64, combined=False, policy="sink_recent_random",
                            n_recent=16, n_random=48, valid_drop=0.01, mask_type="causal")


def qsa_t32k(seed=1005, lens=(4096, 8192, 8192, 12288)):
    """Per-query bitmap sparse attention: T=32768 packed (4096/8192/8192/12288), Hq=24,
    Hkv=2, D=256, block 4, 16 nearest + 256 random earlier blocks, scale 1/16."""
    return make_qsa_problem(seed, list(lens), Hq=24, Hkv=2, D=256, block_size=4, n_near=16,
                            n_random=256, scale=1.0 / 16)


def qsa_t32k_indexed(seed=1005, lens=(4096, 8192, 8192, 12288)):
    """qsa_t32k's selection as index rows (indexed form): sel_indices [32768, 272] int32, each
    row's selected block ids in a seeded random order (rows with fewer blocks padded with -1)."""
    return make_qsa_indexed_problem(seed, list(lens), Hq=24, Hkv=2, D=256, block_size=4,
                                    n_near=16, n_random=256, scale=1.0 / 16)


def sage_b2h16(seed=1006):
    """Prequantized block-sparse attention: B=2, H=16, Sq=Sk=4096, D=128, 16 distinct uniform
    64-key blocks per 64-query block (block_sparse_num, uniform), no block sizes."""
    return make_sage_problem(seed, B=2, H=16, Sq=4096, Sk=4096, capacity=16, uniform=16,
                             sizes="none")
