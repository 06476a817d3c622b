"""The benchmark's oracle samples are faithful slices of their workloads (CPU only): the
oracle on a slice equals the oracle on the same rows of the whole problem, so the rate timed
on a slice is the oracle's rate on the workload's own rows.  Also pins the bitmap form's
gathered-byte count against a loop over (token, block)."""
import numpy as np

import bench
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W


def _bsa(p):
    return A.block_sparse_attention(
        p["q"], p["kv_indptr"], p["kv_indices"], p["block_indptr"], p["block_indices"],
        p["q_block_size"], p["kv_block_size"], p["seq_lens_kv"], kv_cache=p.get("kv_cache"),
        k_cache=p.get("k_cache"), v_cache=p.get("v_cache"), kv_valid_bits=p.get("kv_valid_bits"),
        mask_type=p["mask_type"], sm_scale=p["sm_scale"])


def test_bsr_query_block_slice_keeps_positions():
    p = W.make_bsr_problem(71, B=2, Sq=40, Hq=4, Hkv=2, D=16, seq_lens=[70, 45], page_size=8,
                           qbs=8, kvbs=8, policy="random", p=0.6, valid_drop=0.1,
                           mask_type="causal")
    o, s = _bsa(p)
    sub = bench.bsr_qblock_slice(p, 2, 4)
    o2, s2 = _bsa(sub)
    assert np.allclose(o2, o[:, 16:32], atol=1e-12, rtol=0)
    assert np.array_equal(np.isneginf(s2), np.isneginf(s[:, 16:32]))
    fin = np.isfinite(s2)
    assert np.allclose(s2[fin], s[:, 16:32][fin], atol=1e-12, rtol=0)


def test_prefill_subbatch_equals_its_rows():
    p = W.make_prefill_problem(72, [9, 20, 5], [7, 0, 30], Hq=4, Hkv=2, D=16, page_size=8,
                               mask_type="causal", window_left=6)
    kw = dict(mask_type="causal", window_left=6, sm_scale=p["sm_scale"])
    o, s = A.batch_prefill(p["q"], p["k_cache"], p["v_cache"], p["qo_indptr"],
                           p["block_tables"], p["seq_lens_kv"], **kw)
    sub = bench.prefill_subbatch(p, [0, 2])
    o2, s2 = A.batch_prefill(sub["q"], sub["k_cache"], sub["v_cache"], sub["qo_indptr"],
                             sub["block_tables"], sub["seq_lens_kv"], **kw)
    rows = list(range(0, 9)) + list(range(29, 34))
    assert np.allclose(o2, o[rows], atol=1e-12, rtol=0)
    assert np.allclose(s2, s[rows], atol=1e-12, rtol=0)
    assert bench.prefill_pairs(sub) == A.prefill_visible_pairs(4, sub["qo_indptr"],
                                                               sub["seq_lens_kv"], "causal", 6)


def test_qsa_last_sequence_equals_its_rows():
    p = W.make_qsa_problem(73, [16, 24, 32], Hq=4, Hkv=2, D=8, block_size=4, n_near=2,
                           n_random=3)
    args = lambda q: (q["q"], q["k"], q["v"], q["sel_blocks"], q["lo"], q["hi"],  # noqa: E731
                      q["blk_base"], q["tok_base"], q["block_first"], q["block_last"],
                      q["scale"], q["block_size"])
    o, s = A.qsa_forward(*args(p))
    seq = bench.qsa_last_sequence(p)
    o2, s2 = A.qsa_forward(*args(seq))
    assert np.allclose(o2, o[40:], atol=1e-12, rtol=0)
    assert np.allclose(s2, s[:, 40:], atol=1e-12, rtol=0)
    rows = [0, 5, 31]
    assert bench.qsa_pairs(bench.qsa_rows(seq, rows)) == sum(len(_visible(seq, t)) * 4
                                                             for t in rows)
    pi = W.make_qsa_indexed_problem(73, [16, 24, 32], Hq=4, Hkv=2, D=8, block_size=4, n_near=2,
                                    n_random=3, extra_cols=2, junk=0.5)
    seqi = bench.qsa_last_sequence(pi)
    oi, si = A.qsa_indexed_forward(seqi["q"], seqi["k"], seqi["v"], seqi["sel_indices"],
                                   seqi["lo"], seqi["hi"], seqi["block_first"],
                                   seqi["block_last"], seqi["scale"], seqi["block_size"])
    oi_full, _ = A.qsa_indexed_forward(pi["q"], pi["k"], pi["v"], pi["sel_indices"], pi["lo"],
                                       pi["hi"], pi["block_first"], pi["block_last"],
                                       pi["scale"], pi["block_size"])
    assert np.allclose(oi, oi_full[40:], atol=1e-12, rtol=0)


def _visible(p, t):
    first, last = p["block_first"].numpy(), p["block_last"].numpy()
    sel = p["sel_blocks"].numpy()
    return [j for j in range(int(p["lo"][t]), int(p["hi"][t]) + 1)
            for g in range(first.size) if first[g] <= j <= last[g] and sel[t, g]]


def test_qsa_gathered_bytes_counts_live_blocks():
    p = W.make_qsa_problem(74, [16, 24], Hq=4, Hkv=2, D=8, block_size=4, n_near=2, n_random=3)
    sel = p["sel_blocks"].numpy()
    first, last = p["block_first"].numpy(), p["block_last"].numpy()
    n = 0
    for t in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            if sel[t, g] and max(first[g], int(p["lo"][t])) <= min(last[g], int(p["hi"][t])):
                n += 1
    assert bench.qsa_gathered_bytes(p) == n * 4 * 2 * 8 * 2 * 2
    pi = W.make_qsa_indexed_problem(74, [16, 24], Hq=4, Hkv=2, D=8, block_size=4, n_near=2,
                                    n_random=3, extra_cols=2, junk=0.5)
    assert bench.qsa_gathered_bytes(pi) == n * 4 * 2 * 8 * 2 * 2
