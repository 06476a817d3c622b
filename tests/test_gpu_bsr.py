"""GPU parity of the block-sparse paged attention path (device planner + tcgen05 kernel)
against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from oracle import planner as PL
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, read_ws, to_dev

pytestmark = pytest.mark.gpu


def _run(p):
    d = to_dev(p)
    cache = d["kv_cache"] if "kv_cache" in d else (d["k_cache"], d["v_cache"])
    B, Sq, Hq, D = p["q"].shape
    out = torch.full_like(d["q"], 5.0)
    lse = torch.full((B, Sq, Hq), 9.0, dtype=torch.float32, device=DEV)
    params = pkb.bsr_params(d["q"], cache, p["q_block_size"], p["kv_block_size"],
                            p["max_seq_len_kv"], has_valid_bits=p["kv_valid_bits"] is not None,
                            mask_type=p["mask_type"], sm_scale=p["sm_scale"])
    meta = pkb.bsr_meta(d["kv_indptr"], d["kv_indices"], d["block_indptr"], d["block_indices"],
                        d["seq_lens_kv"], d["kv_valid_bits"])
    pkb.paged_attn_validate_bsr(params, p["kv_indptr"], p["kv_indices"], p["block_indptr"],
                                p["block_indices"], p["seq_lens_kv"])
    ws = torch.empty(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    k, v = (cache, None) if not isinstance(cache, tuple) else cache
    pkb.paged_attn_plan(params, meta, ws)
    pkb.paged_attn_run(params, meta, d["q"], k, v, out, None, lse, ws)
    torch.cuda.synchronize()
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.OK, (rc, raw)
    return out, lse, ws, params


def _oracle(p, rows=None):
    return A.block_sparse_attention(
        p["q"], p["kv_indptr"], p["kv_indices"], p["block_indptr"], p["block_indices"],
        p["q_block_size"], p["kv_block_size"], p["seq_lens_kv"], kv_cache=p.get("kv_cache"),
        k_cache=p.get("k_cache"), v_cache=p.get("v_cache"), kv_valid_bits=p.get("kv_valid_bits"),
        mask_type=p["mask_type"], sm_scale=p["sm_scale"], rows=rows)


def _check_plan(p, ws, params):
    lay = pkb.plan_layout(params)
    B, Sq, Hq, _ = p["q"].shape
    Hkv = Hq // (Hq // params.num_kv_heads)
    recs = read_ws(ws, lay.tiles_offset, 8 * lay.tiles_capacity).numpy().reshape(-1, 8)
    ref = PL.plan_bsr_tiles(B, Sq, Hq, params.num_kv_heads, p["q_block_size"], p["block_indptr"],
                            lay.tile_tokens)
    assert np.array_equal(recs, ref)


def test_tiny_bsr_workload():
    p = W.tiny_bsr()
    out, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


CASES = [
    # (B, Sq, Hq, Hkv, lens, ps, qbs, kvbs, combined, policy, kw, drop, mask)
    (2, 100, 8, 2, [300, 129], 16, 64, 64, False, "random", {"p": 0.6}, 0.0, "causal"),
    (1, 77, 4, 1, [200], 32, 32, 32, True, "random", {"p": 0.5}, 0.05, "dense"),
    (3, 40, 16, 2, [40, 90, 64], 16, 16, 16, False, "all", {}, 0.0, "causal"),
    (2, 130, 8, 8, [130, 256], 64, 128, 128, False, "diag_bernoulli", {"p": 0.3}, 0.02, "causal"),
    (1, 64, 16, 2, [500], 64, 64, 192, False, "random", {"p": 0.7}, 0.0, "dense"),
    (2, 33, 8, 1, [100, 50], 16, 24, 8, True, "random", {"p": 0.5}, 0.1, "causal"),
    (2, 50, 4, 4, [80, 60], 16, 16, 64, False, "empty", {}, 0.0, "dense"),
    (1, 256, 64, 8, [700], 64, 128, 64, False, "sink_recent_random",
     {"n_recent": 3, "n_random": 2}, 0.01, "causal"),
    # page sizes that are not powers of two: 8-key pieces that never straddle a page
    (2, 40, 8, 2, [100, 77], 24, 16, 64, False, "random", {"p": 0.6}, 0.0, "causal"),
    (1, 30, 4, 1, [150], 40, 8, 8, True, "random", {"p": 0.5}, 0.1, "dense"),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_bsr_matches_oracle(case):
    B, Sq, Hq, Hkv, lens, ps, qbs, kvbs, comb, pol, kw, drop, mask = CASES[case]
    p = W.make_bsr_problem(200 + case, B=B, Sq=Sq, Hq=Hq, Hkv=Hkv, D=128, seq_lens=lens,
                           page_size=ps, qbs=qbs, kvbs=kvbs, combined=comb, policy=pol,
                           valid_drop=drop, mask_type=mask, **kw)
    out, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


def test_blocks_past_the_length_contribute_nothing():
    p = W.make_bsr_problem(230, B=1, Sq=64, Hq=4, Hkv=1, D=128, seq_lens=[150], page_size=16,
                           qbs=64, kvbs=64, policy="all", mask_type="dense")
    p["max_seq_len_kv"] = 400
    # row selects block 0 and block 5 (keys 320..383, all past the length)
    p["block_indptr"] = torch.tensor([[[0, 2]]], dtype=torch.int32)
    p["block_indices"] = torch.tensor([0, 5], dtype=torch.int32)
    out, lse, _, _ = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)


@pytest.mark.slow
def test_long_bsr_workload_sampled():
    """The 64K-token workload in its bench launch configuration.  Compared rows: every row of
    the last 8 work tiles in launch order (the cheapest tiles, which run at the tail of the
    persistent grid), one whole 128-row q-block, the edges of the first q-blocks, the last
    row, and the rows of random whole tiles up to at least 1,024 in all."""
    p = W.long_bsr()
    out, lse, ws, params = _run(p)
    _check_plan(p, ws, params)
    lay = pkb.plan_layout(params)
    recs = read_ws(ws, lay.tiles_offset, 8 * lay.tiles_capacity).numpy().reshape(-1, 8)
    S = p["q"].shape[1]
    rows = set()
    for b, g, tok0, ntok, *_ in recs[-8:]:
        assert b == 0
        rows |= set(range(int(tok0), int(tok0) + int(ntok)))
    qb = 300 * p["q_block_size"]
    rows |= set(range(qb, qb + p["q_block_size"]))
    rows |= {0, 1, 127, 128, S - 1}
    rng = np.random.default_rng(5)
    for t in rng.permutation(len(recs) - 8):        # whole random tiles
        if len(rows) >= 1024:
            break
        rows |= set(range(int(recs[t, 2]), int(recs[t, 2]) + int(recs[t, 3])))
    rows = sorted(rows)
    o_ref, l_ref = _oracle(p, rows=[(0, i) for i in rows])
    check_out(out[0, rows], o_ref[0, rows])
    check_lse(lse[0, rows], l_ref[0, rows])
