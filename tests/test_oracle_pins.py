"""Pins of the float64 oracle against things other than itself (CPU only).

* a naive brute-force route (tests/bruteforce.py) on tiny inputs;
* torch's scaled_dot_product_attention in float64 with an explicit boolean mask;
* hand-derived closed forms (tests/golden/closed_form_cases.json);
* invariants: page order, combined vs separate pools, all-blocks BSR = dense causal
  prefill = decode, GQA = MHA with repeated KV heads, NaN in unused pages, split-KV merge,
  bitmap form = block-sparse form on the same selection;
* closed forms: uniform V, q = 0 (LSE = log #visible), a single visible key, two equal keys.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests import bruteforce as BF

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def _close(a, b, tol=1e-12):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(np.where(both_inf, 0.0, a))), "unexpected non-finite"
    assert d.max(initial=0.0) <= tol, d.max()


def _run_bsa(p, **kw):
    return A.block_sparse_attention(
        p["q"], p["kv_indptr"], p["kv_indices"], p["block_indptr"], p["block_indices"],
        p["q_block_size"], p["kv_block_size"], p["seq_lens_kv"], kv_cache=p.get("kv_cache"),
        k_cache=p.get("k_cache"), v_cache=p.get("v_cache"), kv_valid_bits=p.get("kv_valid_bits"),
        mask_type=p["mask_type"], sm_scale=p["sm_scale"], **kw)


def _run_prefill(p, **kw):
    return A.batch_prefill(p["q"], p["k_cache"], p["v_cache"], p["qo_indptr"], p["block_tables"],
                           p["seq_lens_kv"], mask_type=p["mask_type"],
                           window_left=p["window_left"], sm_scale=p["sm_scale"],
                           output_scale=p["output_scale"], **kw)


def _run_decode(p, **kw):
    return A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                          kv_cache=p.get("kv_cache"), k_cache=p.get("k_cache"),
                          v_cache=p.get("v_cache"), bmm1_scale=p["sm_scale"],
                          bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                          window_left=p["window_left"], seq_len_q=p.get("seq_len_q", 1),
                          qo_indptr=p.get("qo_indptr"), **kw)


def _run_qsa(p, **kw):
    return A.qsa_forward(p["q"], p["k"], p["v"], p["sel_blocks"], p["lo"], p["hi"], p["blk_base"],
                         p["tok_base"], p["block_first"], p["block_last"], p["scale"],
                         p["block_size"], **kw)


# ----------------------------------------------------------------------------------------
# brute force
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed,policy,mask,drop,combined", [
    (1, "random", "causal", 0.2, False),
    (2, "diag_bernoulli", "causal", 0.0, True),
    (3, "random", "dense", 0.3, False),
    (4, "all", "dense", 0.0, True),
])
def test_bsa_matches_bruteforce(seed, policy, mask, drop, combined):
    p = W.make_bsr_problem(seed, B=2, Sq=6, Hq=4, Hkv=2, D=8, seq_lens=[13, 9], page_size=4,
                           qbs=4, kvbs=4, combined=combined, policy=policy, p=0.5,
                           valid_drop=drop, mask_type=mask)
    o, s = _run_bsa(p)
    ob, sb = BF.bsa_bruteforce(p)
    _close(o, ob)
    _close(s, sb)


@pytest.mark.parametrize("seed,mask,window,oscale", [
    (5, "causal", -1, 1.0), (6, "causal", 3, 1.0), (7, "dense", -1, 0.5), (8, "causal", 0, 2.0)])
def test_prefill_matches_bruteforce(seed, mask, window, oscale):
    p = W.make_prefill_problem(seed, q_lens=[3, 5, 1], prefix_lens=[4, 0, 6], Hq=4, Hkv=1, D=8,
                               page_size=4, mask_type=mask, window_left=window,
                               output_scale=oscale)
    o, s = _run_prefill(p)
    ob, sb = BF.prefill_bruteforce(p)
    _close(o, ob)
    _close(s, sb)


@pytest.mark.parametrize("seed,kw", [
    (5, dict(seq_lens=[9, 14], mask_type="dense")),
    (6, dict(seq_lens=[9, 14], mask_type="causal", window_left=3, combined=False)),
    (7, dict(seq_lens=[7, 12], seq_len_q=3, mask_type="causal")),
    (8, dict(seq_lens=[7, 12], seq_len_q=3, mask_type="dense", bmm2_scale=0.5)),
    (9, dict(seq_lens=[5, 13, 6], q_lens=[1, 4, 2], mask_type="causal", window_left=2)),
    (10, dict(seq_lens=[2, 10], q_lens=[3, 1], mask_type="causal", combined=False)),
])
def test_decode_matches_bruteforce(seed, kw):
    """One, fixed and packed query layouts; request 0 of the last case has more queries
    than keys, so its first query sits before the first key and sees nothing."""
    kw = dict(kw)
    lens = kw.pop("seq_lens")
    p = W.make_decode_problem(seed, lens, Hq=4, Hkv=2, D=8, page_size=4, **kw)
    o, s = _run_decode(p)
    ob, sb = BF.decode_bruteforce(p)
    _close(o, ob)
    _close(s, sb)


def test_qsa_matches_bruteforce():
    p = W.make_qsa_problem(9, [16, 24], Hq=4, Hkv=2, D=8, block_size=4, n_near=2, n_random=2)
    o, s = _run_qsa(p)
    ob, sb = BF.qsa_bruteforce(p)
    _close(o, ob)
    _close(s, sb)


# ----------------------------------------------------------------------------------------
# library special case: torch SDPA in float64 with an explicit mask
# ----------------------------------------------------------------------------------------

def _run_qsa_indexed(p, **kw):
    return A.qsa_indexed_forward(p["q"], p["k"], p["v"], p["sel_indices"], p["lo"], p["hi"],
                                 p["block_first"], p["block_last"], p["scale"], p["block_size"],
                                 **kw)


@pytest.mark.parametrize("extra,junk", [(0, 0.0), (3, 0.5)])
def test_qsa_indexed_matches_bruteforce(extra, junk):
    p = W.make_qsa_indexed_problem(37, [16, 12], Hq=2, Hkv=1, D=8, block_size=4, n_near=2,
                                   n_random=2, extra_cols=extra, junk=junk)
    o, s = _run_qsa_indexed(p)
    ob, sb = BF.qsa_indexed_bruteforce(p)
    _close(o, ob)
    _close(s, sb)


def test_qsa_indexed_equals_bitmap_form():
    """The same selection as index rows (any order, padded, with listed blocks past hi) and
    as a bitmap gives the same result."""
    kw = dict(Hq=4, Hkv=2, D=16, block_size=4, n_near=3, n_random=4)
    pi = W.make_qsa_indexed_problem(38, [24, 40], extra_cols=5, junk=0.3, **kw)
    pb = W.make_qsa_problem(38, [24, 40], **kw)
    o_i, s_i = _run_qsa_indexed(pi)
    o_b, s_b = _run_qsa(pb)
    _close(o_i, o_b, 1e-13)
    _close(s_i, s_b, 1e-13)


def _run_sage(p, **kw):
    return A.sage_block_sparse_attention(p["q_int8"], p["k_int8"], p["v_fp8"], p["q_scale"],
                                         p["k_scale"], p["v_scale"], p["q2k_block_index"],
                                         p["block_sparse_num"], p["block_sizes"],
                                         p["q2k_block_nums"], p["softmax_scale"], **kw)


def test_fp8_e4m3_decoding_follows_the_format():
    codes = np.arange(256, dtype=np.uint8)
    got = A.fp8_e4m3_to_f64(codes)
    want = np.array([BF.e4m3_value(c) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


@pytest.mark.parametrize("kw", [
    dict(B=1, H=2, Sq=70, Sk=150, capacity=2, sizes="bhnb", empty_rows=0.3),
    dict(B=2, H=1, Sq=64, Sk=64, uniform=1, sizes="nb"),
    dict(B=1, H=1, Sq=33, Sk=190, uniform=2, sizes="none"),
    dict(B=2, H=3, Sq=40, Sk=130, capacity=3, sizes="bnb"),     # [B, NB]: per batch
    dict(B=2, H=2, Sq=20, Sk=130, capacity=3, sizes="bnb"),     # B = H must not mix them up
])
def test_sage_matches_bruteforce(kw):
    p = W.make_sage_problem(45, D=8, **kw)
    _close(_run_sage(p), BF.sage_bruteforce(p), 1e-12)


def test_sage_with_unit_scales_equals_block_sparse_form():
    """Unit scales make the dequantized values the integers and the FP8 values themselves:
    the result is then the [BSA] forward (non-causal, 64-query and 64-key blocks, one KV head
    per (b, h)) on those values."""
    p = W.make_sage_problem(46, B=1, H=2, Sq=100, Sk=180, capacity=3, sizes="none", D=8)
    p["q_scale"] = torch.ones_like(p["q_scale"])
    p["k_scale"] = torch.ones_like(p["k_scale"])
    p["v_scale"] = torch.ones_like(p["v_scale"])
    o = _run_sage(p)
    B, H, Sq, D = p["q_int8"].shape
    Sk = p["k_int8"].shape[2]
    NB = -(-Sk // 64)
    vf = A.fp8_e4m3_to_f64(p["v_fp8"])[:, :, :, :Sk]
    for h in range(H):
        # one request of the [BSA] form: identity pages of 64 keys
        kc = torch.zeros((NB, 1, 64, D), dtype=torch.float64)
        vc = torch.zeros((NB, 1, 64, D), dtype=torch.float64)
        kc.view(NB * 64, D)[:Sk] = p["k_int8"][0, h].double()
        vc.view(NB * 64, D)[:Sk] = torch.from_numpy(vf[0, h].T.copy())
        nums = p["q2k_block_nums"][0, h]
        ptr = np.concatenate([[0], np.cumsum(nums.numpy())]).reshape(1, 1, -1)
        ids = torch.cat([p["q2k_block_index"][0, h, r, :int(nums[r])] for r in range(nums.numel())])
        ob, _ = A.block_sparse_attention(
            p["q_int8"][0:1, h][:, :, None, :].double(), torch.tensor([0, NB]), torch.arange(NB),
            torch.from_numpy(ptr), ids, 64, 64, torch.tensor([Sk]), k_cache=kc, v_cache=vc,
            mask_type="dense", sm_scale=p["softmax_scale"])
        _close(o[0, h], ob[0, :, 0], 1e-12)


def test_sage_zero_query_gives_the_mean_of_visible_values():
    """q = 0: O = the mean of the visible dequantized V rows, an integer count that pins the
    block selection, the counts and the block sizes; a row selecting nothing is exactly 0."""
    p = W.make_sage_problem(47, B=1, H=1, Sq=128, Sk=250, capacity=3, sizes="bhnb",
                            empty_rows=0.3, D=8)
    p["q_int8"] = torch.zeros_like(p["q_int8"])
    o = _run_sage(p)
    vf = A.fp8_e4m3_to_f64(p["v_fp8"])[0, 0] * p["v_scale"][0, 0].double().numpy()[:, None]
    for r in range(2):
        n = int(p["q2k_block_nums"][0, 0, r])
        js = [j for c in p["q2k_block_index"][0, 0, r, :n].tolist()
              for j in range(64 * c, min(250, 64 * c + int(p["block_sizes"][0, 0, c])))]
        rows = o[0, 0, 64 * r:64 * r + 64]
        if not js:
            assert np.all(rows == 0.0)
        else:
            _close(rows, np.broadcast_to(vf[:, js].mean(axis=1), rows.shape), 1e-13)


def test_prefill_matches_torch_sdpa():
    p = W.make_prefill_problem(11, q_lens=[7, 12], prefix_lens=[9, 3], Hq=6, Hkv=2, D=16,
                               page_size=8, mask_type="causal", window_left=5)
    o, s = _run_prefill(p)
    G = 3
    qo = p["qo_indptr"]
    for b in range(2):
        r0, r1 = int(qo[b]), int(qo[b + 1])
        L = int(p["seq_lens_kv"][b])
        pages = p["block_tables"][b].long()
        j = torch.arange(L)
        K = p["k_cache"].double()[pages[j // 8], :, j % 8]          # [L, Hkv, D]
        V = p["v_cache"].double()[pages[j // 8], :, j % 8]
        Kh = K.repeat_interleave(G, dim=1).permute(1, 0, 2)         # [Hq, L, D]
        Vh = V.repeat_interleave(G, dim=1).permute(1, 0, 2)
        Q = p["q"].double()[r0:r1].permute(1, 0, 2)                  # [Hq, nq, D]
        pos = L - (r1 - r0) + torch.arange(r1 - r0)
        mask = (j[None, :] <= pos[:, None]) & (j[None, :] >= pos[:, None] - 5)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, Kh, Vh, attn_mask=mask,
                                                               scale=p["sm_scale"])
        _close(o[r0:r1], ref.permute(1, 0, 2).numpy(), 1e-12)
        sc = (Q @ Kh.transpose(1, 2)) * p["sm_scale"]
        lse = torch.logsumexp(sc.masked_fill(~mask, -math.inf), dim=-1).permute(1, 0)
        _close(s[r0:r1], lse.numpy(), 1e-12)


# ----------------------------------------------------------------------------------------
# hand-derived closed forms
# ----------------------------------------------------------------------------------------

def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp, "log": math.log,
                                                   "inf": math.inf}))


def _golden_cases():
    with open(GOLDEN) as f:
        g = json.load(f)
    return g, [c["name"] for c in g["cases"]]


@pytest.mark.parametrize("name", _golden_cases()[1])
def test_golden_closed_forms(name):
    g, _ = _golden_cases()
    case = next(c for c in g["cases"] if c["name"] == name)
    keys = torch.tensor(g["keys"], dtype=torch.bfloat16)
    vals = torch.tensor(g["values"], dtype=torch.bfloat16)
    L, D = keys.shape
    nq = len(case["queries"])
    q = torch.tensor(case["queries"], dtype=torch.bfloat16)
    # one page per token, pages stored in reverse order to exercise the table
    pool_k = keys.flip(0)[:, None, None, :].contiguous()            # [P=L, Hkv=1, ps=1, D]
    pool_v = vals.flip(0)[:, None, None, :].contiguous()
    pages = torch.arange(L - 1, -1, -1, dtype=torch.int32)
    if case["form"] == "prefill":
        o, s = A.batch_prefill(q[:, None, :], pool_k, pool_v, torch.tensor([0, nq]),
                               pages[None, :], torch.tensor([L]), mask_type=case["mask"],
                               window_left=case["window_left"], sm_scale=case["scale"],
                               output_scale=case["output_scale"])
        o, s = o[:, 0], s[:, 0]
    elif case["form"] == "decode":
        o, s = A.batch_decode(q[:, None, :], torch.tensor([0, L]), pages, torch.tensor([L]),
                              k_cache=pool_k, v_cache=pool_v, bmm1_scale=case["scale"],
                              mask_type=case["mask"], window_left=case["window_left"])
        o, s = o[:, 0], s[:, 0]
    else:
        bl = case["blocks"]
        bptr = np.concatenate([[0], np.cumsum([len(x) for x in bl])]).reshape(1, 1, -1)
        bidx = torch.tensor([x for r in bl for x in r], dtype=torch.int32)
        vb = None
        if case["valid_bits"] is not None:
            vb = torch.tensor(np.array(case["valid_bits"], np.uint32).view(np.int32))[None]
        o, s = A.block_sparse_attention(q[None, :, None, :], torch.tensor([0, L]), pages,
                                        torch.tensor(bptr), bidx, case["q_block_size"],
                                        case["kv_block_size"], torch.tensor([L]),
                                        k_cache=pool_k, v_cache=pool_v, kv_valid_bits=vb,
                                        mask_type=case["mask"], sm_scale=case["scale"])
        o, s = o[0, :, 0], s[0, :, 0]
    for i, e in enumerate(case["expect"]):
        _close(s[i], _eval(e["lse"]), 1e-14)
        _close(o[i], [_eval(x) for x in e["o"]], 1e-14)


# ----------------------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------------------

def _identity_pages(p):
    """Same logical K/V with every request's pages laid out consecutively."""
    ps = p["page_size"]
    lens = [int(x) for x in p["seq_lens_kv"]]
    pools = [p["k_cache"], p["v_cache"]] if "k_cache" in p else [p["kv_cache"][:, 0],
                                                                 p["kv_cache"][:, 1]]
    new_k, new_v, indptr, indices = [], [], [0], []
    for b, L in enumerate(lens):
        pg = p["kv_indices"][int(p["kv_indptr"][b]):int(p["kv_indptr"][b + 1])].long()
        for t in pg:
            indices.append(len(new_k))
            new_k.append(pools[0][t])
            new_v.append(pools[1][t])
        indptr.append(len(indices))
    q = dict(p)
    q.pop("kv_cache", None)
    q["k_cache"], q["v_cache"] = torch.stack(new_k), torch.stack(new_v)
    q["kv_indptr"] = torch.tensor(indptr, dtype=torch.int32)
    q["kv_indices"] = torch.tensor(indices, dtype=torch.int32)
    return q


def test_page_order_and_combined_pools_do_not_matter():
    p = W.make_bsr_problem(21, B=2, Sq=20, Hq=4, Hkv=2, D=16, seq_lens=[50, 37], page_size=8,
                           qbs=8, kvbs=8, combined=True, policy="random", p=0.6,
                           valid_drop=0.1, mask_type="causal")
    o1, s1 = _run_bsa(p)
    o2, s2 = _run_bsa(_identity_pages(p))
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
    assert not np.isnan(o1).any()


def test_nan_in_unused_pages_is_never_read():
    p = W.make_bsr_problem(22, B=2, Sq=9, Hq=2, Hkv=1, D=8, seq_lens=[21, 10], page_size=8,
                           qbs=4, kvbs=8, policy="all", mask_type="causal")
    o1, s1 = _run_bsa(p)
    assert not np.isnan(o1).any() and not np.isnan(s1).any()
    q = dict(p)
    q["k_cache"] = p["k_cache"].clone()
    q["k_cache"][p["spare_pages"].long()] = 7.0
    o2, s2 = _run_bsa(q)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_all_blocks_bsr_equals_prefill_equals_decode():
    lens = [40, 29]
    Sq = 1
    p = W.make_bsr_problem(23, B=2, Sq=Sq, Hq=4, Hkv=2, D=16, seq_lens=lens, page_size=8,
                           qbs=1, kvbs=8, policy="causal_all", mask_type="causal")
    o_bsa, s_bsa = _run_bsa(p)
    # the same pages as a row-strided table for the prefill form
    tables = torch.zeros(2, 5, dtype=torch.int32)
    for b in range(2):
        pg = p["kv_indices"][int(p["kv_indptr"][b]):int(p["kv_indptr"][b + 1])]
        tables[b, :pg.numel()] = pg
    pre = dict(q=p["q"].reshape(2, 4, 16), k_cache=p["k_cache"], v_cache=p["v_cache"],
               qo_indptr=torch.tensor([0, 1, 2]), block_tables=tables,
               seq_lens_kv=p["seq_lens_kv"], mask_type="causal", window_left=-1,
               sm_scale=p["sm_scale"], output_scale=1.0)
    o_pre, s_pre = _run_prefill(pre)
    _close(o_bsa.reshape(2, 4, 16), o_pre)
    _close(s_bsa.reshape(2, 4), s_pre)
    dec = dict(q=p["q"].reshape(2, 4, 16), kv_indptr=p["kv_indptr"], kv_indices=p["kv_indices"],
               seq_lens=p["seq_lens_kv"], k_cache=p["k_cache"], v_cache=p["v_cache"],
               sm_scale=p["sm_scale"], bmm2_scale=1.0, mask_type="dense", window_left=-1)
    o_dec, s_dec = _run_decode(dec)
    _close(o_dec, o_pre)
    _close(s_dec, s_pre)


def test_dense_bsr_with_longer_queries_equals_prefill():
    lens, Sq = [45, 33], 12
    p = W.make_bsr_problem(24, B=2, Sq=Sq, Hq=4, Hkv=2, D=16, seq_lens=lens, page_size=8,
                           qbs=4, kvbs=8, policy="all", mask_type="causal")
    o_bsa, s_bsa = _run_bsa(p)
    tables = torch.zeros(2, 6, dtype=torch.int32)
    for b in range(2):
        pg = p["kv_indices"][int(p["kv_indptr"][b]):int(p["kv_indptr"][b + 1])]
        tables[b, :pg.numel()] = pg
    pre = dict(q=p["q"].reshape(2 * Sq, 4, 16), k_cache=p["k_cache"], v_cache=p["v_cache"],
               qo_indptr=torch.tensor([0, Sq, 2 * Sq]), block_tables=tables,
               seq_lens_kv=p["seq_lens_kv"], mask_type="causal", window_left=-1,
               sm_scale=p["sm_scale"], output_scale=1.0)
    o_pre, s_pre = _run_prefill(pre)
    _close(o_bsa.reshape(2 * Sq, 4, 16), o_pre)
    _close(s_bsa.reshape(2 * Sq, 4), s_pre)


def test_empty_rows_are_exactly_zero_and_minus_inf():
    p = W.make_bsr_problem(25, B=1, Sq=8, Hq=2, Hkv=1, D=8, seq_lens=[16], page_size=4,
                           qbs=4, kvbs=4, policy="empty", mask_type="dense")
    o, s = _run_bsa(p)
    assert np.all(o == 0.0) and np.all(np.isneginf(s))
    # a causal row whose selected blocks all lie after its position is empty too
    p = W.make_bsr_problem(26, B=1, Sq=4, Hq=2, Hkv=1, D=8, seq_lens=[16], page_size=4,
                           qbs=4, kvbs=4, policy="all", mask_type="causal")
    p["block_indptr"] = torch.tensor([[[0, 1]]], dtype=torch.int32)
    p["block_indices"] = torch.tensor([3], dtype=torch.int32)
    p["seq_lens_kv"] = torch.tensor([16], dtype=torch.int32)
    o, s = _run_bsa(p)                  # queries at 12..15, block 3 = keys 12..15
    assert np.all(np.isfinite(s))
    p["block_indices"] = torch.tensor([4], dtype=torch.int32)     # beyond the live length
    o, s = _run_bsa(p)
    assert np.all(o == 0.0) and np.all(np.isneginf(s))


def test_gqa_equals_mha_with_repeated_kv_heads():
    G = 3
    p = W.make_bsr_problem(27, B=2, Sq=10, Hq=6, Hkv=2, D=8, seq_lens=[30, 17], page_size=4,
                           qbs=5, kvbs=4, policy="random", p=0.7, valid_drop=0.1,
                           mask_type="causal")
    o1, s1 = _run_bsa(p)
    m = dict(p)
    m["k_cache"] = p["k_cache"].repeat_interleave(G, dim=1)
    m["v_cache"] = p["v_cache"].repeat_interleave(G, dim=1)
    m["block_indptr"] = None
    rows_ptr, rows_idx, off = [], [], 0
    bptr, bidx = p["block_indptr"], p["block_indices"]
    nqb = bptr.shape[2] - 1
    ptr = np.zeros((2, 6, nqb + 1), np.int64)
    for b in range(2):
        for h in range(6):
            for r in range(nqb):
                ptr[b, h, r] = off
                sl = bidx[int(bptr[b, h // G, r]):int(bptr[b, h // G, r + 1])]
                rows_idx.append(sl)
                off += sl.numel()
            ptr[b, h, nqb] = off
    m["block_indptr"] = torch.tensor(ptr.astype(np.int32))
    m["block_indices"] = torch.cat(rows_idx)
    o2, s2 = _run_bsa(m)
    _close(o1, o2)
    _close(s1, s2)


def test_split_kv_merge_equals_unsplit():
    rng = np.random.default_rng(28)
    q = rng.standard_normal((1, 4, 16))
    K = rng.standard_normal((100, 16))
    V = rng.standard_normal((100, 16))
    vis = np.ones((1, 100), bool)
    o_full, s_full = A.masked_softmax_attention(q, K, V, vis, 0.25)
    for cuts in ([0, 100], [0, 37, 100], [0, 10, 20, 30, 99, 100], [0, 0, 50, 100]):
        parts = [A.masked_softmax_attention(q, K[a:b], V[a:b], vis[:, a:b], 0.25)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        o, s = A.merge_partials([x[0] for x in parts], [x[1] for x in parts])
        _close(o, o_full)
        _close(s, s_full)


def test_bitmap_form_equals_block_sparse_form():
    """One sequence; query t selects blocks of 4 tokens and sees lo = 0 .. hi = t.  The same
    selection as BSR rows of one query (q_block_size 1, kv_block_size 4) under the causal
    mask gives the same result."""
    p = W.make_qsa_problem(29, [32], Hq=4, Hkv=2, D=8, block_size=4, n_near=2, n_random=3)
    o1, s1 = _run_qsa(p)
    T = 32
    sel = p["sel_blocks"].numpy()
    ptr = np.zeros((1, 2, T + 1), np.int64)
    idx, off = [], 0
    for g in range(2):
        for t in range(T):
            ptr[0, g, t] = off
            blocks = np.nonzero(sel[t])[0]
            idx.extend(blocks.tolist())
            off += blocks.size
        ptr[0, g, T] = off
    k_pool = p["k"].reshape(8, 4, 2, 8).permute(0, 2, 1, 3).contiguous()    # pages of 4 tokens
    v_pool = p["v"].reshape(8, 4, 2, 8).permute(0, 2, 1, 3).contiguous()
    o2, s2 = A.block_sparse_attention(p["q"][None], torch.tensor([0, 8]),
                                      torch.arange(8, dtype=torch.int32),
                                      torch.tensor(ptr.astype(np.int32)),
                                      torch.tensor(idx, dtype=torch.int32), 1, 4,
                                      torch.tensor([T]), k_cache=k_pool, v_cache=v_pool,
                                      mask_type="causal", sm_scale=p["scale"])
    _close(o1, o2[0])
    _close(s1, s2[0].T)


# ----------------------------------------------------------------------------------------
# closed forms on random problems
# ----------------------------------------------------------------------------------------

def test_uniform_v_gives_v():
    p = W.make_prefill_problem(31, q_lens=[5, 9], prefix_lens=[3, 11], Hq=4, Hkv=2, D=8,
                               page_size=4, mask_type="causal", window_left=4,
                               output_scale=1.5)
    v = p["v_cache"].clone()
    row = torch.randn(2, 8).to(torch.bfloat16)
    v[:] = row[None, :, None, :]
    p["v_cache"] = v
    o, _ = _run_prefill(p)
    expect = 1.5 * row.double().numpy()[np.arange(4) // 2]
    _close(o, np.broadcast_to(expect, o.shape))


def test_zero_query_counts_visible_keys():
    """q = 0 makes every visible score 0: LSE = log(#visible) and O = mean of visible v.
    The count comes from the brute-force visibility rules."""
    p = W.make_bsr_problem(32, B=2, Sq=7, Hq=4, Hkv=2, D=8, seq_lens=[25, 12], page_size=4,
                           qbs=3, kvbs=4, policy="random", p=0.5, valid_drop=0.25,
                           mask_type="causal")
    p["q"] = torch.zeros_like(p["q"])
    o, s = _run_bsa(p)
    for b in range(2):
        for i in range(7):
            for h in range(4):
                js = BF.bsa_visible(p, b, i, h)
                if not js:
                    assert o[b, i, h].tolist() == [0.0] * 8 and s[b, i, h] == -math.inf
                    continue
                _close(s[b, i, h], math.log(len(js)), 1e-14)
                vals = np.array([BF._kv_row(p, b, j, h // 2, "v") for j in js])
                _close(o[b, i, h], vals.mean(axis=0), 1e-13)
    pq = W.make_qsa_problem(33, [20, 12], Hq=2, Hkv=1, D=8, block_size=4, n_near=1, n_random=2)
    pq["q"] = torch.zeros_like(pq["q"])
    _, s = _run_qsa(pq)
    for t in range(32):
        n = len(BF.qsa_visible(pq, t))
        _close(s[:, t], [math.log(n) if n else -math.inf] * 2, 1e-14)


def test_zero_query_decode_counts_visible_keys():
    """q = 0 in multi-query decode: LSE = log of the number of visible keys, which for query
    i of nq at position p = L - nq + i is min(p, L - 1) + 1 - max(0, p - w) under the causal
    mask (L without it)."""
    lens, q_lens, w = [11, 6, 20], [3, 6, 1], 4
    for mask, win in (("causal", -1), ("causal", w), ("dense", -1)):
        p = W.make_decode_problem(34, lens, Hq=2, Hkv=1, D=8, page_size=4, q_lens=q_lens,
                                  mask_type=mask, window_left=win)
        p["q"] = torch.zeros_like(p["q"])
        _, s = _run_decode(p)
        row = 0
        for L, nq in zip(lens, q_lens):
            for i in range(nq):
                pos = L - nq + i
                if mask == "causal":
                    n = min(pos, L - 1) + 1 - (max(0, pos - win) if win >= 0 else 0)
                else:
                    n = L
                _close(s[row], [math.log(n) if n > 0 else -math.inf] * 2, 1e-14)
                row += 1


def test_multi_query_decode_equals_prefill():
    """Decode with packed queries over a CSR table and prefill over the same pages as a
    row-strided table are the same computation."""
    lens, q_lens = [23, 9, 31], [4, 9, 2]
    p = W.make_decode_problem(35, lens, Hq=4, Hkv=2, D=16, page_size=8, q_lens=q_lens,
                              mask_type="causal", window_left=5, combined=False,
                              bmm2_scale=1.25)
    o_dec, s_dec = _run_decode(p)
    C = max(-(-L // 8) for L in lens)
    tables = torch.zeros(len(lens), C, dtype=torch.int32)
    for b in range(len(lens)):
        pg = p["kv_indices"][int(p["kv_indptr"][b]):int(p["kv_indptr"][b + 1])]
        tables[b, :len(pg)] = pg
    o_pre, s_pre = A.batch_prefill(p["q"], p["k_cache"], p["v_cache"], p["qo_indptr"], tables,
                                   p["seq_lens"], mask_type="causal", window_left=5,
                                   sm_scale=p["sm_scale"], output_scale=1.25)
    _close(o_dec, o_pre, 0)
    _close(s_dec, s_pre, 0)


def test_fixed_and_packed_decode_layouts_agree():
    lens = [17, 5]
    p = W.make_decode_problem(36, lens, Hq=4, Hkv=1, D=8, page_size=4, seq_len_q=3,
                              mask_type="causal", window_left=6)
    o_fix, s_fix = _run_decode(p)
    packed = dict(p, q=p["q"].reshape(6, 4, 8), seq_len_q=1,
                  qo_indptr=torch.tensor([0, 3, 6], dtype=torch.int32))
    o_pk, s_pk = _run_decode(packed)
    _close(o_fix.reshape(6, 4, 8), o_pk, 0)
    _close(s_fix.reshape(6, 4), s_pk, 0)


def test_single_and_duplicate_keys():
    q = np.array([[[0.5, -1.0, 2.0]]])
    K = np.array([[1.0, 2.0, 3.0], [1.0, 2.0, 3.0], [4.0, 0.0, 1.0]])
    V = np.array([[1.0, 0.0, 0.0], [1.0, 0.0, 0.0], [0.0, 5.0, 0.0]])
    s0 = 0.7 * (0.5 - 2.0 + 6.0)
    o, s = A.masked_softmax_attention(q, K, V, np.array([[True, False, False]]), 0.7)
    _close(o[0, 0], V[0], 0)
    _close(s[0, 0], s0, 1e-15)
    o, s = A.masked_softmax_attention(q, K, V, np.array([[True, True, False]]), 0.7)
    _close(s[0, 0], s0 + math.log(2.0), 1e-14)
    _close(o[0, 0], V[0], 1e-15)


# ----------------------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin above
# ----------------------------------------------------------------------------------------

def test_planted_causal_off_by_one_is_caught(monkeypatch):
    p = W.make_prefill_problem(41, q_lens=[4], prefix_lens=[3], Hq=2, Hkv=1, D=8, page_size=4,
                               mask_type="causal")
    ref_o, _ = BF.prefill_bruteforce(p)
    real = A.masked_softmax_attention

    def shifted(q, keys, vals, visible, scale, out_scale=1.0):
        vis = visible.copy()
        vis[:, 1:] |= visible[:, :-1]          # lets each row see one key past its position
        return real(q, keys, vals, vis, scale, out_scale)

    monkeypatch.setattr(A, "masked_softmax_attention", shifted)
    o, _ = _run_prefill(p)
    assert np.abs(o - ref_o).max() > 1e-3


def test_planted_top_left_decode_alignment_is_caught(monkeypatch):
    """Placing multi-query decode queries at positions 0..nq-1 (top-left) instead of the
    last nq positions must disagree with the brute force."""
    p = W.make_decode_problem(43, [10], Hq=2, Hkv=1, D=8, page_size=4, seq_len_q=3,
                              mask_type="causal")
    ob, _ = BF.decode_bruteforce(p)
    o, _ = _run_decode(p)
    _close(o, ob)
    real = A.masked_softmax_attention

    def top_left(q, keys, vals, visible, scale, out_scale=1.0):
        n, L = visible.shape
        vis = np.arange(L)[None, :] <= np.arange(n)[:, None]
        return real(q, keys, vals, vis, scale, out_scale)

    monkeypatch.setattr(A, "masked_softmax_attention", top_left)
    o2, _ = _run_decode(p)
    assert np.abs(o2 - ob).max() > 1e-3


def test_planted_gqa_mapping_is_caught():
    p = W.make_bsr_problem(42, B=1, Sq=4, Hq=4, Hkv=2, D=8, seq_lens=[8], page_size=4, qbs=4,
                           kvbs=4, policy="all", mask_type="dense")
    o, _ = _run_bsa(p)
    ob, _ = BF.bsa_bruteforce(p)
    _close(o, ob)
    # reading KV head h % Hkv instead of h // G gives a different answer
    swapped = dict(p)
    swapped["q"] = p["q"][:, :, [0, 2, 1, 3]]
    o2, _ = _run_bsa(swapped)
    assert np.abs(o2[:, :, [0, 2, 1, 3]] - ob).max() > 1e-3


def test_planted_exclusive_hi_is_caught():
    """Reading the bitmap form's hi as an exclusive bound (keys lo .. hi - 1) must disagree
    with the brute force, which keeps hi itself ([QSA] lo/hi are inclusive)."""
    p = W.make_qsa_problem(46, [20, 12], Hq=4, Hkv=2, D=8, block_size=4, n_near=2, n_random=2)
    ob, sb = BF.qsa_bruteforce(p)
    o, s = _run_qsa(p)
    _close(o, ob)
    excl = dict(p, hi=p["hi"] - 1)                # the oracle fed the misreading
    o2, s2 = _run_qsa(excl)
    fin = np.isfinite(sb) & np.isfinite(np.asarray(s2))
    assert np.abs(np.asarray(s2)[fin] - np.asarray(sb)[fin]).max() > 1e-3


def test_planted_msb_first_valid_bits_are_caught():
    """Reading kv_valid_bits most significant bit first must disagree with the brute force,
    which takes bit j & 31 of word j >> 5, least significant first."""
    p = W.make_bsr_problem(47, B=1, Sq=8, Hq=2, Hkv=1, D=8, seq_lens=[40], page_size=8, qbs=4,
                           kvbs=8, policy="all", valid_drop=0.3, mask_type="causal")
    ob, _ = BF.bsa_bruteforce(p)
    o, _ = _run_bsa(p)
    _close(o, ob)
    w = p["kv_valid_bits"].numpy().view(np.uint32)
    rev = np.zeros_like(w)
    for k in range(32):                            # bit k moves to bit 31 - k
        rev |= ((w >> np.uint32(k)) & np.uint32(1)) << np.uint32(31 - k)
    o2, _ = _run_bsa(dict(p, kv_valid_bits=torch.from_numpy(rev.view(np.int32))))
    assert np.abs(o2 - ob).max() > 1e-3


def test_planted_query_scale_group_is_caught():
    """Using one query scale per 64 queries (column i // 64) instead of per 32 (column
    i // 32) must disagree with the brute force."""
    p = W.make_sage_problem(48, D=8, B=1, H=1, Sq=96, Sk=128, uniform=2, sizes="none")
    ref = BF.sage_bruteforce(p)
    _close(_run_sage(p), ref, 1e-12)
    qs = p["q_scale"].clone()
    ncol = qs.shape[-1]
    qs_wrong = qs[..., [min(c // 2, ncol - 1) for c in range(ncol)]]
    assert not torch.equal(qs_wrong, qs)
    assert np.abs(_run_sage(dict(p, q_scale=qs_wrong)) - ref).max() > 1e-3


def test_planted_merge_weights_are_caught():
    """Merging split-KV partials with weights exp(LSE_s) left unnormalised (or with equal
    weights) must disagree with the unsplit softmax that the merge pin compares against."""
    rng = np.random.default_rng(49)
    q = rng.standard_normal((1, 2, 16))
    K = rng.standard_normal((60, 16))
    V = rng.standard_normal((60, 16))
    vis = np.ones((1, 60), bool)
    o_full, _ = A.masked_softmax_attention(q, K, V, vis, 0.25)
    parts = [A.masked_softmax_attention(q, K[a:b], V[a:b], vis[:, a:b], 0.25)
             for a, b in ((0, 17), (17, 60))]
    o_parts = np.stack([x[0] for x in parts])
    lse = np.stack([x[1] for x in parts])
    unnormalised = (np.exp(lse)[..., None] * o_parts).sum(0)
    equal = o_parts.mean(0)
    assert np.abs(unnormalised - o_full).max() > 1e-3
    assert np.abs(equal - o_full).max() > 1e-3
    o, _ = A.merge_partials([x[0] for x in parts], [x[1] for x in parts])
    _close(o, o_full)


def test_planted_window_of_w_keys_is_caught():
    """A window of w keys (p - w < j) instead of w + 1 (p - w <= j, the query's own position
    counted inside it) must disagree with the brute force, for prefill and for decode."""
    p = W.make_prefill_problem(50, q_lens=[5, 3], prefix_lens=[6, 2], Hq=2, Hkv=1, D=8,
                               page_size=4, mask_type="causal", window_left=3)
    ob, _ = BF.prefill_bruteforce(p)
    o, _ = _run_prefill(p)
    _close(o, ob)
    o2, _ = _run_prefill(dict(p, window_left=2))
    assert np.abs(o2 - ob).max() > 1e-3
    d = W.make_decode_problem(51, [9, 14], Hq=2, Hkv=1, D=8, page_size=4, q_lens=[1, 3],
                              mask_type="causal", window_left=4)
    db, _ = BF.decode_bruteforce(d)
    o, _ = _run_decode(d)
    _close(o, db)
    o2, _ = _run_decode(dict(d, window_left=3))
    assert np.abs(o2 - db).max() > 1e-3
