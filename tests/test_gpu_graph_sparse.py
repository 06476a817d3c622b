"""CUDA-graph capture and replay of the sparse forms (block-sparse, bitmap, prequantized): the
plan and the run are captured once, then the metadata is rewritten in place with another
selection of the same static shape before each replay, and every replay is checked against
the float64 oracle."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out

pytestmark = pytest.mark.gpu


def _capture(run):
    run()                                       # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    return g


def _into(dst, src):
    """Copy src into the front of the device buffer dst (the rest keeps its old contents)."""
    dst.view(-1)[:src.numel()].copy_(src.reshape(-1))


def test_bsr_graph_replay_with_new_selection():
    kw = dict(B=2, Sq=100, Hq=8, Hkv=2, D=128, seq_lens=[300, 129], page_size=16, qbs=64,
              kvbs=64, combined=False, mask_type="causal")
    probs = [W.make_bsr_problem(800, policy="random", p=0.7, **kw),
             W.make_bsr_problem(801, policy="random", p=0.3, valid_drop=0.1, **kw)]
    NI = max(p["block_indices"].numel() for p in probs)
    d = {k: v.to(DEV) for k, v in probs[0].items() if isinstance(v, torch.Tensor)}
    bidx = torch.zeros(max(NI, 1), dtype=torch.int32, device=DEV)
    vbits = torch.zeros_like(probs[1]["kv_valid_bits"], device=DEV)
    params = pkb.bsr_params(d["q"], (d["k_cache"], d["v_cache"]), 64, 64,
                            probs[0]["max_seq_len_kv"], has_valid_bits=True, mask_type="causal",
                            sm_scale=probs[0]["sm_scale"])
    meta = pkb.bsr_meta(d["kv_indptr"], d["kv_indices"], d["block_indptr"], bidx,
                        d["seq_lens_kv"], vbits)
    ws = torch.zeros(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=DEV)

    def run():
        pkb.paged_attn_plan(params, meta, ws)
        pkb.paged_attn_run(params, meta, d["q"], d["k_cache"], d["v_cache"], out, None, lse, ws)

    def stage(p):
        for name in ("q", "k_cache", "v_cache", "kv_indptr", "kv_indices", "block_indptr",
                     "seq_lens_kv"):
            d[name].copy_(p[name])
        _into(bidx, p["block_indices"])
        vb = p["kv_valid_bits"]
        vbits.copy_(vb if vb is not None else torch.full_like(vbits.cpu(), -1))

    stage(probs[0])
    g = _capture(run)
    for p in probs:
        stage(p)
        out.fill_(3.0)
        g.replay()
        torch.cuda.synchronize()
        rc, raw = pkb.paged_attn_workspace_status(ws)
        assert rc == pkb.OK, (rc, raw)
        o_ref, l_ref = A.block_sparse_attention(
            p["q"], p["kv_indptr"], p["kv_indices"], p["block_indptr"], p["block_indices"], 64,
            64, p["seq_lens_kv"], k_cache=p["k_cache"], v_cache=p["v_cache"],
            kv_valid_bits=p["kv_valid_bits"], mask_type="causal", sm_scale=p["sm_scale"])
        check_out(out, o_ref)
        check_lse(lse, l_ref)


def test_bitmap_graph_replay_with_new_selection():
    kw = dict(Hq=24, Hkv=2, D=256, block_size=4, scale=1.0 / 16)
    probs = [W.make_qsa_problem(802, [120, 80], n_near=4, n_random=10, **kw),
             W.make_qsa_problem(803, [120, 80], n_near=2, n_random=25, **kw)]
    d = {k: v.to(DEV) for k, v in probs[0].items() if isinstance(v, torch.Tensor)}
    T, Hq, D = probs[0]["q"].shape
    params = pkb.qsa_params(d["q"], d["k"], d["sel_blocks"].shape[1], scale=kw["scale"])
    meta = pkb.qsa_meta(d["sel_blocks"], d["lo"], d["hi"], d["blk_base"], d["tok_base"],
                        d["block_first"], d["block_last"])
    ws = torch.zeros(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(d["q"])
    lse = torch.empty(Hq, T, dtype=torch.float32, device=DEV)

    def run():
        pkb.paged_attn_plan(params, meta, ws)
        pkb.paged_attn_run(params, meta, d["q"], d["k"], d["v"], out, None, lse, ws)

    g = _capture(run)
    for p in probs:
        for name in ("q", "k", "v", "sel_blocks", "lo", "hi"):
            d[name].copy_(p[name])
        out.fill_(3.0)
        g.replay()
        torch.cuda.synchronize()
        rc, raw = pkb.paged_attn_workspace_status(ws)
        assert rc == pkb.OK, (rc, raw)
        o_ref, l_ref = A.qsa_forward(p["q"], p["k"], p["v"], p["sel_blocks"], p["lo"], p["hi"],
                                     p["blk_base"], p["tok_base"], p["block_first"],
                                     p["block_last"], p["scale"], p["block_size"])
        check_out(out, o_ref)
        check_lse(lse, l_ref)


def test_sage_graph_replay_with_new_selection():
    kw = dict(B=1, H=4, Sq=200, Sk=700, capacity=5, sizes="bhnb")
    probs = [W.make_sage_problem(804, **kw), W.make_sage_problem(805, empty_rows=0.3, **kw)]
    d = {k: v.to(DEV) for k, v in probs[0].items() if isinstance(v, torch.Tensor)}
    params = pkb.sage_params(d["q_int8"], d["k_int8"], d["q2k_block_index"], 0,
                             block_sizes=d["block_sizes"], softmax_scale=probs[0]["softmax_scale"])
    ws = torch.zeros(pkb.paged_sage_workspace_size(params), dtype=torch.uint8, device=DEV)
    out = torch.empty(probs[0]["q_int8"].shape, dtype=torch.bfloat16, device=DEV)

    def run():
        pkb.paged_sage_run(params, d["q_int8"], d["k_int8"], d["v_fp8"], d["q_scale"],
                           d["k_scale"], d["v_scale"], d["q2k_block_index"], d["q2k_block_nums"],
                           d["block_sizes"], out, ws)

    g = _capture(run)
    for p in probs:
        for name, v in d.items():
            v.copy_(p[name])
        out.fill_(3.0)
        g.replay()
        torch.cuda.synchronize()
        rc, raw = pkb.paged_attn_workspace_status(ws)
        assert rc == pkb.OK, (rc, raw)
        o_ref = A.sage_block_sparse_attention(
            p["q_int8"], p["k_int8"], p["v_fp8"], p["q_scale"], p["k_scale"], p["v_scale"],
            p["q2k_block_index"], p["block_sparse_num"], p["block_sizes"], p["q2k_block_nums"],
            p["softmax_scale"])
        check_out(out.reshape(-1, 1, 128), o_ref.reshape(-1, 1, 128))
