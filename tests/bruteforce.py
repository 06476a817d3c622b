"""A second, deliberately naive route to the attention definition, for pinning the oracle.

Pure Python loops over every (request, query, head, key) on tiny inputs: each key's
visibility is decided from the raw page-table/selection/mask rules with integer
arithmetic, keys are fetched one page lookup at a time, and the softmax is taken with
math.fsum / math.exp.  Nothing here is shared with the oracle.
"""
import math

import numpy as np


def _vec(t):
    return [float(x) for x in t]


def _softmax_row(q, keys, vals, scale, out_scale=1.0):
    """q: list[D]; keys/vals: list of list[D].  Returns (o list[D], lse)."""
    if not keys:
        return [0.0] * len(q), -math.inf
    s = [scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    tot = math.fsum(w)
    D = len(q)
    o = [out_scale * math.fsum(w[n] * vals[n][d] for n in range(len(w))) / tot for d in range(D)]
    return o, m + math.log(tot)


def _bit(words, b, j):
    word = int(words[b][j // 32]) & 0xFFFFFFFF
    return (word >> (j % 32)) & 1


def bsa_visible(prob, b, i, h):
    """Visible logical key positions of row (b, i), query head h, in a block-sparse problem."""
    q = prob["q"]
    B, Sq, Hq, D = q.shape
    Hkv = (prob["k_cache"] if "k_cache" in prob else prob["kv_cache"][:, 0]).shape[1]
    G = Hq // Hkv
    g = h // G
    L = int(prob["seq_lens_kv"][b])
    qbs, kvbs = prob["q_block_size"], prob["kv_block_size"]
    r = i // qbs
    lo, hi = int(prob["block_indptr"][b, g, r]), int(prob["block_indptr"][b, g, r + 1])
    blocks = [int(x) for x in prob["block_indices"][lo:hi]]
    words = None
    if prob.get("kv_valid_bits") is not None:
        words = prob["kv_valid_bits"].numpy().view(np.uint32)
    out = []
    for j in range(L):
        if (j // kvbs) not in blocks:
            continue
        if words is not None and not _bit(words, b, j):
            continue
        if prob["mask_type"] == "causal" and j > L - Sq + i:
            continue
        out.append(j)
    return out


def _kv_row(prob, b, j, kv_head, which):
    ps = prob["page_size"]
    if "kv_indptr" in prob:
        page = int(prob["kv_indices"][int(prob["kv_indptr"][b]) + j // ps])
    else:
        page = int(prob["block_tables"][b, j // ps])
    if "kv_cache" in prob:
        t = prob["kv_cache"][page, 0 if which == "k" else 1, kv_head, j % ps]
    else:
        t = prob["k_cache" if which == "k" else "v_cache"][page, kv_head, j % ps]
    return _vec(t.float())


def bsa_bruteforce(prob):
    q = prob["q"]
    B, Sq, Hq, D = q.shape
    Hkv = (prob["k_cache"] if "k_cache" in prob else prob["kv_cache"][:, 0]).shape[1]
    G = Hq // Hkv
    scale = prob["sm_scale"]
    O = np.zeros((B, Sq, Hq, D))
    LSE = np.zeros((B, Sq, Hq))
    for b in range(B):
        for i in range(Sq):
            for h in range(Hq):
                js = bsa_visible(prob, b, i, h)
                keys = [_kv_row(prob, b, j, h // G, "k") for j in js]
                vals = [_kv_row(prob, b, j, h // G, "v") for j in js]
                o, s = _softmax_row(_vec(q[b, i, h].float()), keys, vals, scale)
                O[b, i, h], LSE[b, i, h] = o, s
    return O, LSE


def prefill_visible(prob, b, i):
    """Visible keys of local query i of request b in a packed prefill problem."""
    qo = prob["qo_indptr"]
    nq = int(qo[b + 1]) - int(qo[b])
    L = int(prob["seq_lens_kv"][b])
    p = L - nq + i
    w = prob["window_left"]
    out = []
    for j in range(L):
        if prob["mask_type"] == "causal":
            if j > p:
                continue
            if w >= 0 and j < p - w:
                continue
        out.append(j)
    return out


def prefill_bruteforce(prob):
    q = prob["q"]
    T, Hq, D = q.shape
    Hkv = prob["k_cache"].shape[1]
    G = Hq // Hkv
    O = np.zeros((T, Hq, D))
    LSE = np.zeros((T, Hq))
    qo = prob["qo_indptr"]
    for b in range(len(prob["seq_lens_kv"])):
        for i in range(int(qo[b + 1]) - int(qo[b])):
            js = prefill_visible(prob, b, i)
            for h in range(Hq):
                keys = [_kv_row(prob, b, j, h // G, "k") for j in js]
                vals = [_kv_row(prob, b, j, h // G, "v") for j in js]
                o, s = _softmax_row(_vec(q[int(qo[b]) + i, h].float()), keys, vals,
                                    prob["sm_scale"], prob["output_scale"])
                O[int(qo[b]) + i, h], LSE[int(qo[b]) + i, h] = o, s
    return O, LSE


def qsa_visible(prob, t):
    first = [int(x) for x in prob["block_first"]]
    last = [int(x) for x in prob["block_last"]]
    sel = prob["sel_blocks"]
    out = []
    for j in range(int(prob["lo"][t]), int(prob["hi"][t]) + 1):
        for g in range(len(first)):
            if first[g] <= j <= last[g]:
                if int(sel[t, g]) != 0:
                    out.append(j)
                break
    return out


def qsa_bruteforce(prob):
    q, k, v = prob["q"], prob["k"], prob["v"]
    T, Hq, D = q.shape
    G = Hq // k.shape[1]
    O = np.zeros((T, Hq, D))
    LSE = np.zeros((Hq, T))
    for t in range(T):
        js = qsa_visible(prob, t)
        for h in range(Hq):
            keys = [_vec(k[j, h // G].float()) for j in js]
            vals = [_vec(v[j, h // G].float()) for j in js]
            o, s = _softmax_row(_vec(q[t, h].float()), keys, vals, prob["scale"])
            O[t, h], LSE[h, t] = o, s
    return O, LSE


def decode_visible(prob, b, i):
    """Visible keys of query i of request b in a decode problem (one, fixed or packed
    queries): the query sits at len - nq + i."""
    nq = int(prob["q_lens"][b])
    L = int(prob["seq_lens"][b])
    p = L - nq + i
    w = prob["window_left"]
    out = []
    for j in range(L):
        if prob["mask_type"] == "causal":
            if j > p:
                continue
            if w >= 0 and j < p - w:
                continue
        out.append(j)
    return out


def decode_bruteforce(prob):
    """O and LSE in the query's own layout ([B, Hq, D], [B, SQ, Hq, D] or packed)."""
    q = prob["q"]
    Hq, D = q.shape[-2], q.shape[-1]
    Hkv = (prob["k_cache"] if "k_cache" in prob else prob["kv_cache"][:, 0]).shape[1]
    G = Hq // Hkv
    qrows = q.reshape(-1, Hq, D)
    O = np.zeros((qrows.shape[0], Hq, D))
    LSE = np.zeros((qrows.shape[0], Hq))
    row = 0
    for b in range(len(prob["seq_lens"])):
        for i in range(int(prob["q_lens"][b])):
            js = decode_visible(prob, b, i)
            for h in range(Hq):
                keys = [_kv_row(prob, b, j, h // G, "k") for j in js]
                vals = [_kv_row(prob, b, j, h // G, "v") for j in js]
                o, s = _softmax_row(_vec(qrows[row, h].float()), keys, vals, prob["sm_scale"],
                                    prob["bmm2_scale"])
                O[row, h], LSE[row, h] = o, s
            row += 1
    return O.reshape(tuple(q.shape)), LSE.reshape(tuple(q.shape[:-1]))


def qsa_indexed_visible(prob, t):
    """Visible key tokens of query t in the indexed form: walk the keys in [lo, hi] and keep
    those whose block (found by scanning the spans) is listed in row t."""
    first = [int(x) for x in prob["block_first"]]
    last = [int(x) for x in prob["block_last"]]
    listed = set(int(g) for g in prob["sel_indices"][t])
    out = []
    for j in range(int(prob["lo"][t]), int(prob["hi"][t]) + 1):
        for g in range(len(first)):
            if first[g] <= j <= last[g]:
                if g in listed:
                    out.append(j)
                break
    return out


def qsa_indexed_bruteforce(prob):
    q, k, v = prob["q"], prob["k"], prob["v"]
    T, Hq, D = q.shape
    G = Hq // k.shape[1]
    O = np.zeros((T, Hq, D))
    LSE = np.zeros((Hq, T))
    for t in range(T):
        js = qsa_indexed_visible(prob, t)
        for h in range(Hq):
            keys = [_vec(k[j, h // G].float()) for j in js]
            vals = [_vec(v[j, h // G].float()) for j in js]
            o, s = _softmax_row(_vec(q[t, h].float()), keys, vals, prob["scale"])
            O[t, h], LSE[h, t] = o, s
    return O, LSE


def e4m3_value(code):
    """FP8 E4M3 (e4m3fn) from its bit fields: sign, 4-bit exponent with bias 7 (0 =
    subnormal), 3-bit mantissa; S.1111.111 is NaN and there is no infinity."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _sage_block_size(prob, b, h, c):
    bs = prob["block_sizes"]
    if bs is None:
        return 64
    if bs.dim() == 1:
        return int(bs[c])
    if bs.dim() == 2:
        return int(bs[b, c])
    return int(bs[b, h, c])


def sage_visible(prob, b, h, i):
    """Visible keys of query i of (b, h) in the prequantized form: walk every key and keep
    those whose 64-key block is among the row's first n listed ids and whose offset inside
    the block is below the block's size."""
    Sk = prob["k_int8"].shape[2]
    r = i // 64
    n = (int(prob["q2k_block_nums"][b, h, r]) if prob["q2k_block_nums"] is not None
         else int(prob["block_sparse_num"]))
    listed = [int(c) for c in prob["q2k_block_index"][b, h, r, :n]]
    out = []
    for j in range(Sk):
        c = j // 64
        if c in listed and j - 64 * c < _sage_block_size(prob, b, h, c):
            out.append(j)
    return out


def sage_bruteforce(prob):
    """Dequantized block-sparse attention by plain loops (bit-level FP8 decoding)."""
    qi, ki, vh = prob["q_int8"], prob["k_int8"], prob["v_fp8"]
    B, H, Sq, D = qi.shape
    O = np.zeros((B, H, Sq, D))
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                qs = float(prob["q_scale"][b, h, i // 32])
                q = [int(x) * qs for x in qi[b, h, i]]
                keys, vals = [], []
                for j in sage_visible(prob, b, h, i):
                    ks = float(prob["k_scale"][b, h, j // 64])
                    keys.append([int(x) * ks for x in ki[b, h, j]])
                    vals.append([e4m3_value(vh[b, h, d, j]) * float(prob["v_scale"][b, h, d])
                                 for d in range(D)])
                o, _ = _softmax_row(q, keys, vals, prob["softmax_scale"])
                O[b, h, i] = o
    return O
