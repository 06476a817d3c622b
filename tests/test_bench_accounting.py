"""The benchmark's own work counters agree with the oracle's exact visible-pair counts (CPU)."""
import numpy as np

import bench
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W


def test_bsr_pairs_match_oracle_count():
    for p in (W.tiny_bsr(),
              W.make_bsr_problem(3, B=2, Sq=50, Hq=8, Hkv=2, D=16, seq_lens=[90, 61], page_size=16,
                                 qbs=16, kvbs=16, policy="random", p=0.5, valid_drop=0.1,
                                 mask_type="causal"),
              W.make_bsr_problem(4, B=1, Sq=40, Hq=4, Hkv=4, D=16, seq_lens=[70], page_size=8,
                                 qbs=8, kvbs=8, policy="all", mask_type="dense")):
        B, Sq, Hq, _ = p["q"].shape
        Hkv = p["k_cache"].shape[1]
        ref = A.bsr_visible_pairs(B, Sq, Hq, Hkv, p["block_indptr"], p["block_indices"],
                                  p["q_block_size"], p["kv_block_size"], p["seq_lens_kv"],
                                  p["kv_valid_bits"], p["mask_type"])
        assert bench.bsr_pairs(p) == ref


def test_prefill_pairs_match_oracle_count():
    for w in (-1, 0, 17):
        p = W.make_prefill_problem(5, [30, 7, 64], [0, 50, 12], Hq=4, Hkv=2, D=16, page_size=16,
                                   mask_type="causal", window_left=w)
        ref = A.prefill_visible_pairs(4, p["qo_indptr"], p["seq_lens_kv"], "causal", w)
        assert bench.prefill_pairs(p) == ref


def test_qsa_pairs_match_oracle_count():
    p = W.make_qsa_problem(6, [64, 32], Hq=4, Hkv=1, D=16, block_size=4, n_near=3, n_random=4)
    ref = A.qsa_visible_pairs(4, p["sel_blocks"], p["lo"], p["hi"], p["block_first"],
                              p["block_last"])
    assert bench.qsa_pairs(p) == ref


def test_decode_bytes():
    p = W.make_decode_problem(7, [10, 20], Hq=4, Hkv=2, D=128, page_size=16)
    assert bench.decode_kv_bytes(p) == 30 * 2 * 128 * 2 * 2
