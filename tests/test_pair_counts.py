"""Pins of the visible-pair counters (CPU only).

Every TFLOPS figure the benchmark prints is 4 * D times a count of visible (query row, query
head, key) triples.  The oracle's counters (oracle/attention.py) and the benchmark's own
restatements (bench.py) are each checked here against two routes that share nothing with
them:

* the brute-force visibility of tests/bruteforce.py, which walks every key of every row with
  the pages' integer rules, summed over rows and heads;
* the q = 0 closed form of the oracle's forward: with every score 0, LSE = ln(#visible keys),
  so the sum of exp(LSE) over rows and heads is the count.

The cases cover valid bits, causal and window masks, empty rows, a ragged last block, more
queries than keys, and index rows padded with -1, ids >= NB and listed blocks past hi.
"""
import numpy as np
import pytest
import torch

import bench
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests import bruteforce as BF


def _lse_count(lse):
    """sum exp(LSE) over finite entries, rounded (LSE = ln n exactly up to rounding)."""
    lse = np.asarray(lse, np.float64)
    tot = float(np.exp(lse[np.isfinite(lse)]).sum())
    n = int(round(tot))
    assert abs(tot - n) < 1e-6 * max(1, n)
    return n


def _zero_q(p, key="q"):
    p = dict(p)
    p[key] = torch.zeros_like(p[key])
    return p


# ----------------------------------------------------------------------------------------
# [BSA] block-sparse
# ----------------------------------------------------------------------------------------

BSR_CASES = [
    # causal, valid bits, ragged last block (lens not multiples of kvbs), random selection
    dict(seed=51, B=2, Sq=10, Hq=4, Hkv=2, D=8, seq_lens=[23, 14], page_size=4, qbs=4, kvbs=8,
         policy="random", p=0.5, valid_drop=0.2, mask_type="causal"),
    # dense mask, every block, GQA group 3
    dict(seed=52, B=1, Sq=7, Hq=6, Hkv=2, D=8, seq_lens=[19], page_size=4, qbs=3, kvbs=4,
         policy="all", mask_type="dense"),
    # diagonal + earlier blocks, the last q-block ragged, combined pool
    dict(seed=53, B=2, Sq=9, Hq=2, Hkv=1, D=8, seq_lens=[30, 9], page_size=8, qbs=4, kvbs=8,
         policy="diag_bernoulli", p=0.5, mask_type="causal", combined=True),
    # empty rows everywhere
    dict(seed=54, B=1, Sq=5, Hq=2, Hkv=1, D=8, seq_lens=[12], page_size=4, qbs=4, kvbs=4,
         policy="empty", mask_type="causal"),
    # sparse random selection with many rows selecting nothing, valid bits, dense mask
    dict(seed=55, B=2, Sq=8, Hq=4, Hkv=4, D=8, seq_lens=[17, 26], page_size=4, qbs=2, kvbs=4,
         policy="random", p=0.2, valid_drop=0.3, mask_type="dense"),
]


def _bsr_brute_count(p):
    B, Sq, Hq, _ = p["q"].shape
    return sum(len(BF.bsa_visible(p, b, i, h))
               for b in range(B) for i in range(Sq) for h in range(Hq))


@pytest.mark.parametrize("case", BSR_CASES)
def test_bsr_pair_counters(case):
    case = dict(case)
    p = W.make_bsr_problem(case.pop("seed"), **case)
    B, Sq, Hq, _ = p["q"].shape
    Hkv = (p["k_cache"] if "k_cache" in p else p["kv_cache"][:, 0]).shape[1]
    want = _bsr_brute_count(p)
    got = A.bsr_visible_pairs(B, Sq, Hq, Hkv, p["block_indptr"], p["block_indices"],
                              p["q_block_size"], p["kv_block_size"], p["seq_lens_kv"],
                              p["kv_valid_bits"], p["mask_type"])
    assert got == want
    assert bench.bsr_pairs(p) == want
    pz = _zero_q(p)
    _, lse = A.block_sparse_attention(
        pz["q"], pz["kv_indptr"], pz["kv_indices"], pz["block_indptr"], pz["block_indices"],
        pz["q_block_size"], pz["kv_block_size"], pz["seq_lens_kv"], kv_cache=pz.get("kv_cache"),
        k_cache=pz.get("k_cache"), v_cache=pz.get("v_cache"),
        kv_valid_bits=pz.get("kv_valid_bits"), mask_type=pz["mask_type"], sm_scale=pz["sm_scale"])
    assert _lse_count(lse) == want


def test_bsr_cases_cover_empty_rows_and_valid_bits():
    """The cases above include rows with no selected block and cleared valid bits."""
    empty, cleared = 0, 0
    for case in BSR_CASES:
        case = dict(case)
        p = W.make_bsr_problem(case.pop("seed"), **case)
        bp = p["block_indptr"].numpy()
        empty += int((bp[..., 1:] == bp[..., :-1]).sum())
        if p["kv_valid_bits"] is not None:
            cleared += 1
    assert empty > 0 and cleared > 0


# ----------------------------------------------------------------------------------------
# [PRE] packed prefill and [DEC] decode
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("mask,window", [("causal", -1), ("causal", 0), ("causal", 3),
                                         ("dense", -1)])
def test_prefill_pair_counters(mask, window):
    p = W.make_prefill_problem(56, q_lens=[3, 6, 1, 5], prefix_lens=[4, 0, 7, 2], Hq=4, Hkv=2,
                               D=8, page_size=4, mask_type=mask, window_left=window)
    qo = p["qo_indptr"]
    want = sum(len(BF.prefill_visible(p, b, i))
               for b in range(len(p["seq_lens_kv"]))
               for i in range(int(qo[b + 1]) - int(qo[b]))) * 4
    assert A.prefill_visible_pairs(4, qo, p["seq_lens_kv"], mask, window) == want
    assert bench.prefill_pairs(p) == want
    pz = _zero_q(p)
    _, lse = A.batch_prefill(pz["q"], pz["k_cache"], pz["v_cache"], pz["qo_indptr"],
                             pz["block_tables"], pz["seq_lens_kv"], mask_type=mask,
                             window_left=window, sm_scale=pz["sm_scale"])
    assert _lse_count(lse) == want


@pytest.mark.parametrize("kw", [
    dict(seq_lens=[9, 14, 1], mask_type="dense"),
    dict(seq_lens=[9, 14], seq_len_q=3, mask_type="causal"),
    dict(seq_lens=[5, 13, 6], q_lens=[1, 4, 2], mask_type="causal", window_left=2),
    # request 0 has more queries than keys: its first query sees nothing
    dict(seq_lens=[2, 10], q_lens=[3, 1], mask_type="causal"),
    dict(seq_lens=[8, 3], q_lens=[2, 2], mask_type="dense"),
])
def test_decode_pair_counter(kw):
    kw = dict(kw)
    lens = kw.pop("seq_lens")
    p = W.make_decode_problem(57, lens, Hq=4, Hkv=2, D=8, page_size=4, **kw)
    want = sum(len(BF.decode_visible(p, b, i))
               for b in range(len(lens)) for i in range(int(p["q_lens"][b]))) * 4
    got = A.decode_visible_pairs(4, p["seq_lens"], p["q_lens"], p["mask_type"],
                                 p["window_left"])
    assert got == want
    pz = _zero_q(p)
    _, lse = A.batch_decode(pz["q"], pz["kv_indptr"], pz["kv_indices"], pz["seq_lens"],
                            kv_cache=pz.get("kv_cache"), k_cache=pz.get("k_cache"),
                            v_cache=pz.get("v_cache"), bmm1_scale=pz["sm_scale"],
                            mask_type=pz["mask_type"], window_left=pz["window_left"],
                            seq_len_q=pz.get("seq_len_q", 1), qo_indptr=pz.get("qo_indptr"))
    assert _lse_count(lse) == want


def test_decode_bytes_follow_the_lengths():
    """Decode moves len * Hkv * D * 2 (K and V) * 2 bytes per request, whatever the queries."""
    p = W.make_decode_problem(58, [10, 20, 1], Hq=4, Hkv=2, D=128, page_size=16)
    assert bench.decode_kv_bytes(p) == (10 + 20 + 1) * 2 * 128 * 2 * 2


# ----------------------------------------------------------------------------------------
# [QSA] bitmap and indexed forms
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("lens,near,rand", [([16, 24], 2, 2), ([12, 8, 20], 1, 3)])
def test_qsa_pair_counters(lens, near, rand):
    p = W.make_qsa_problem(59, lens, Hq=4, Hkv=2, D=8, block_size=4, n_near=near, n_random=rand)
    T = int(sum(lens))
    want = sum(len(BF.qsa_visible(p, t)) for t in range(T)) * 4
    assert A.qsa_visible_pairs(4, p["sel_blocks"], p["lo"], p["hi"], p["block_first"],
                               p["block_last"]) == want
    assert bench.qsa_pairs(p) == want
    pz = _zero_q(p)
    _, lse = A.qsa_forward(pz["q"], pz["k"], pz["v"], pz["sel_blocks"], pz["lo"], pz["hi"],
                           pz["blk_base"], pz["tok_base"], pz["block_first"], pz["block_last"],
                           pz["scale"], pz["block_size"])
    assert _lse_count(lse) == want


@pytest.mark.parametrize("extra,junk,oob", [(0, 0.0, False), (3, 0.5, False), (4, 0.3, True)])
def test_qsa_indexed_pair_counters(extra, junk, oob):
    p = W.make_qsa_indexed_problem(60, [16, 12, 8], Hq=2, Hkv=1, D=8, block_size=4, n_near=2,
                                   n_random=2, extra_cols=extra, junk=junk)
    if oob:
        # ids at or past NB in some padding entries: outside the contract, never visible
        idx = p["sel_indices"].clone()
        NB = p["block_first"].numel()
        pad = (idx < 0).nonzero()
        for n, (t, c) in enumerate(pad.tolist()[::2]):
            idx[t, c] = NB + n % 3
        p = dict(p, sel_indices=idx)
        assert (idx >= NB).any()
    T = p["lo"].numel()
    want = sum(len(BF.qsa_indexed_visible(p, t)) for t in range(T)) * 2
    assert A.qsa_indexed_visible_pairs(2, p["sel_indices"], p["lo"], p["hi"], p["block_first"],
                                       p["block_last"]) == want
    assert bench.qsa_indexed_pairs(p) == want
    pz = _zero_q(p)
    _, lse = A.qsa_indexed_forward(pz["q"], pz["k"], pz["v"], pz["sel_indices"], pz["lo"],
                                   pz["hi"], pz["block_first"], pz["block_last"], pz["scale"],
                                   pz["block_size"])
    assert _lse_count(lse) == want


# ----------------------------------------------------------------------------------------
# [SAGE] prequantized block-sparse
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("kw", [
    dict(B=1, H=2, Sq=70, Sk=150, capacity=2, sizes="bhnb", empty_rows=0.3),
    dict(B=2, H=1, Sq=64, Sk=64, uniform=1, sizes="nb"),
    dict(B=1, H=1, Sq=33, Sk=190, uniform=2, sizes="none"),
    dict(B=2, H=3, Sq=40, Sk=130, capacity=3, sizes="bnb"),
])
def test_sage_pair_counter(kw):
    p = W.make_sage_problem(61, D=8, **kw)
    B, H, Sq, _ = p["q_int8"].shape
    want = sum(len(BF.sage_visible(p, b, h, i))
               for b in range(B) for h in range(H) for i in range(Sq))
    assert bench.sage_pairs(p) == want


# ----------------------------------------------------------------------------------------
# planted mistakes in the counters are caught
# ----------------------------------------------------------------------------------------

def test_planted_counter_mistakes_are_caught():
    """Plausible misreadings of the rules give counts that the brute force rejects: valid
    bits ignored, queries aligned top-left instead of bottom-right, and a window of w keys
    instead of w + 1."""
    case = dict(BSR_CASES[0])
    p = W.make_bsr_problem(case.pop("seed"), **case)
    B, Sq, Hq, _ = p["q"].shape
    want = _bsr_brute_count(p)
    no_bits = A.bsr_visible_pairs(B, Sq, Hq, 2, p["block_indptr"], p["block_indices"],
                                  p["q_block_size"], p["kv_block_size"], p["seq_lens_kv"],
                                  None, p["mask_type"])
    assert no_bits != want
    pf = W.make_prefill_problem(62, q_lens=[3, 6], prefix_lens=[4, 2], Hq=2, Hkv=1, D=8,
                                page_size=4, mask_type="causal", window_left=-1)
    qo = pf["qo_indptr"]
    nq = qo[1:] - qo[:-1]

    def brute(prob):
        return sum(len(BF.prefill_visible(prob, b, i))
                   for b in range(2) for i in range(int(nq[b]))) * 2

    want = brute(pf)
    # top-left: query i sees keys 0..i, the bottom-right count of a request with nq keys
    top_left = A.prefill_visible_pairs(2, qo, nq, "causal", -1)
    assert top_left != want
    w = 2
    want_w = brute(dict(pf, window_left=w))
    assert A.prefill_visible_pairs(2, qo, pf["seq_lens_kv"], "causal", w) == want_w
    assert A.prefill_visible_pairs(2, qo, pf["seq_lens_kv"], "causal", w - 1) != want_w


# ----------------------------------------------------------------------------------------
# block-granular counts (the benchmark's secondary figure)
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", BSR_CASES)
def test_bsr_block_pairs(case):
    """Every listed block taken whole for every row of its q-block: a loop over (row, head)
    of the row's block count times the block size; never below the visible count."""
    case = dict(case)
    p = W.make_bsr_problem(case.pop("seed"), **case)
    B, Sq, Hq, _ = p["q"].shape
    Hkv = (p["k_cache"] if "k_cache" in p else p["kv_cache"][:, 0]).shape[1]
    G, qbs, kvbs = Hq // Hkv, p["q_block_size"], p["kv_block_size"]
    bp = p["block_indptr"].numpy()
    want = sum(int(bp[b, h // G, i // qbs + 1] - bp[b, h // G, i // qbs]) * kvbs
               for b in range(B) for i in range(Sq) for h in range(Hq))
    assert bench.bsr_block_pairs(p) == want
    assert want >= _bsr_brute_count(p)


def test_bsr_block_pairs_equal_visible_without_masks():
    """Every block, dense mask, no valid bits, lengths whole blocks: nothing is cut."""
    p = W.make_bsr_problem(63, B=2, Sq=6, Hq=4, Hkv=2, D=8, seq_lens=[16, 8], page_size=4,
                           qbs=3, kvbs=4, policy="all", mask_type="dense")
    assert p["kv_valid_bits"] is None
    assert bench.bsr_block_pairs(p) == bench.bsr_pairs(p) == _bsr_brute_count(p)


@pytest.mark.parametrize("mask,window,D", [("causal", -1, 128), ("causal", 37, 128),
                                           ("dense", -1, 128), ("causal", 100, 256)])
def test_prefill_tile_pairs_follow_the_planner(mask, window, D):
    """The dense prefill count is the oracle planner's tile list (work tiles of 2 x 128 / G
    tokens, one sub-tile for D = 256) times 128 keys per KV tile and the tile's rows."""
    from oracle import planner
    p = W.make_prefill_problem(64, q_lens=[130, 7, 300], prefix_lens=[0, 260, 45], Hq=8,
                               Hkv=2, D=D, page_size=32, mask_type=mask, window_left=window)
    G = 4
    T = (128 // G) * (1 if D == 256 else 2)
    recs = np.asarray(planner.plan_prefill_tiles(2, p["qo_indptr"], p["seq_lens_kv"], T,
                                                 mask, window))
    want = int(((recs[:, 5] - recs[:, 4]) * 128 * recs[:, 3]).sum()) * G
    assert bench.prefill_tile_pairs(p) == want
    assert want >= bench.prefill_pairs(p)


def test_qsa_block_pairs():
    """Selected blocks that meet [lo, hi], whole: a loop over (token, block); the indexed form
    of the same selection gives the same count."""
    p = W.make_qsa_problem(65, [16, 24], Hq=4, Hkv=2, D=8, block_size=4, n_near=2, n_random=2)
    sel = p["sel_blocks"].numpy()
    lo, hi = p["lo"].numpy(), p["hi"].numpy()
    first, last = p["block_first"].numpy(), p["block_last"].numpy()
    want = 0
    for t in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            if sel[t, g] and max(first[g], lo[t]) <= min(last[g], hi[t]):
                want += int(last[g] - first[g] + 1)
    want *= 4
    assert bench.qsa_block_pairs(p) == want
    assert want >= bench.qsa_pairs(p)
    pi = W.make_qsa_indexed_problem(66, [16, 12, 8], Hq=2, Hkv=1, D=8, block_size=4, n_near=2,
                                    n_random=2, extra_cols=3, junk=0.5)
    idx = pi["sel_indices"].numpy()
    NB = pi["block_first"].numel()
    as_bitmap = np.zeros((idx.shape[0], NB), np.uint8)
    for t, c in zip(*np.nonzero((idx >= 0) & (idx < NB))):
        as_bitmap[t, idx[t, c]] = 1
    pb = dict(pi, sel_blocks=torch.from_numpy(as_bitmap))
    assert bench.qsa_indexed_block_pairs(pi) == bench.qsa_block_pairs(pb)


@pytest.mark.parametrize("kw", [
    dict(B=1, H=2, Sq=70, Sk=150, capacity=2, sizes="bhnb", empty_rows=0.3),
    dict(B=1, H=1, Sq=33, Sk=190, uniform=2, sizes="none"),
])
def test_sage_block_pairs(kw):
    """Each listed 64-key block taken whole for every query of its 64-query block."""
    p = W.make_sage_problem(67, D=8, **kw)
    B, H, Sq, _ = p["q_int8"].shape
    nums = p["q2k_block_nums"]
    want = 0
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                n = int(nums[b, h, i // 64]) if nums is not None else p["block_sparse_num"]
                want += 64 * n
    assert bench.sage_block_pairs(p) == want
    assert want >= bench.sage_pairs(p)
