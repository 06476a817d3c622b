"""GPU parity of the indexed per-query block attention (index rows [T, K] -> device CSR ->
the same tcgen05 kernel as the bitmap form) against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from oracle import planner as PL
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, read_ws, to_dev

pytestmark = pytest.mark.gpu


def _run(p, idx=None, expect=pkb.OK):
    d = to_dev(p)
    sel = d["sel_indices"] if idx is None else idx.to(DEV)
    params = pkb.qsa_indexed_params(d["q"], d["k"], d["block_first"].numel(), sel.shape[1],
                                    scale=p["scale"])
    meta = pkb.qsa_indexed_meta(sel, d["lo"], d["hi"], d["block_first"], d["block_last"])
    T, Hq, D = p["q"].shape
    out = torch.full_like(d["q"], 5.0)
    out32 = torch.full(p["q"].shape, 6.0, dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, T), 7.0, dtype=torch.float32, device=DEV)
    ws = torch.empty(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    pkb.paged_attn_plan(params, meta, ws)
    pkb.paged_attn_run(params, meta, d["q"], d["k"], d["v"], out, out32, lse, ws)
    torch.cuda.synchronize()
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == expect, (rc, raw)
    return out, out32, lse, ws, params


def _oracle(p, idx=None):
    return A.qsa_indexed_forward(p["q"], p["k"], p["v"],
                                 p["sel_indices"] if idx is None else idx, p["lo"], p["hi"],
                                 p["block_first"], p["block_last"], p["scale"], p["block_size"])


def _check_plan(p, ws, params, idx=None):
    lay = pkb.plan_layout(params)
    T = p["q"].shape[0]
    indptr = read_ws(ws, lay.indptr_offset, T + 1).numpy()
    ref_ptr, ref_idx = PL.plan_indexed(p["sel_indices"] if idx is None else idx, p["lo"], p["hi"],
                                       p["block_first"], p["block_last"])
    assert np.array_equal(indptr, ref_ptr)
    got = read_ws(ws, lay.indices_offset, int(indptr[-1])).numpy()
    assert np.array_equal(got, ref_idx)


CASES = [
    # (seq lens, Hq, Hkv, n_near, n_random, extra columns, junk fraction)
    ([64, 128, 40], 24, 2, 4, 8, 0, 0.0),
    ([256], 12, 1, 16, 40, 7, 0.4),
    ([48, 8], 2, 2, 2, 100, 33, 0.2),        # index rows wider than one warp pass
    ([96, 40], 6, 3, 4, 10, 2, 0.5),         # odd Hkv > 1
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_qsa_indexed_matches_oracle(case):
    lens, Hq, Hkv, near, rand, extra, junk = CASES[case]
    p = W.make_qsa_indexed_problem(450 + case, lens, Hq=Hq, Hkv=Hkv, D=256, block_size=4,
                                   n_near=near, n_random=rand, scale=1.0 / 16,
                                   extra_cols=extra, junk=junk)
    out, out32, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_out(out32, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


def test_qsa_indexed_equals_bitmap_form_on_gpu():
    kw = dict(Hq=24, Hkv=2, D=256, block_size=4, n_near=8, n_random=30, scale=1.0 / 16)
    pi = W.make_qsa_indexed_problem(460, [200, 120], extra_cols=5, junk=0.3, **kw)
    pb = W.make_qsa_problem(460, [200, 120], **kw)
    o_i, _, l_i, _, _ = _run(pi)
    d = to_dev(pb)
    params = pkb.qsa_params(d["q"], d["k"], d["sel_blocks"].shape[1], scale=pb["scale"])
    meta = pkb.qsa_meta(d["sel_blocks"], d["lo"], d["hi"], d["blk_base"], d["tok_base"],
                        d["block_first"], d["block_last"])
    ws = torch.empty(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    o_b = torch.empty_like(d["q"])
    l_b = torch.empty_like(l_i)
    pkb.paged_attn_plan(params, meta, ws)
    pkb.paged_attn_run(params, meta, d["q"], d["k"], d["v"], o_b, None, l_b, ws)
    torch.cuda.synchronize()
    # the indexed rows are shuffled, so the blocks are visited in another order: equal up to
    # the reduction order
    check_out(o_i, o_b.float().cpu().numpy().astype(np.float64), max_abs=1e-2, mean_abs=1e-3)
    check_lse(l_i, l_b.cpu().numpy().astype(np.float64))


def test_qsa_indexed_out_of_range_ids_are_dropped_and_reported():
    p = W.make_qsa_indexed_problem(461, [64, 32], Hq=12, Hkv=1, D=256, block_size=4, n_near=3,
                                   n_random=6, scale=1.0 / 16, extra_cols=2)
    idx = p["sel_indices"].clone()
    NB = p["block_first"].numel()
    idx[5, 0] = NB
    idx[40, 1] = NB + 1000
    out, out32, lse, ws, params = _run(p, idx, expect=pkb.ERR_METADATA)
    o_ref, l_ref = _oracle(p, idx)          # the oracle ignores ids outside [0, NB) as well
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params, idx)


@pytest.mark.slow
def test_qsa_t32k_indexed_sampled():
    p = W.qsa_t32k_indexed()
    out, out32, lse, ws, params = _run(p)
    T = p["q"].shape[0]
    rows = sorted(set([0, 1, 4095, 4096, 12287, 12288, T - 1] +
                      list(np.random.default_rng(9).integers(0, T, 40))))
    o_ref, l_ref = A.qsa_indexed_forward(p["q"], p["k"], p["v"], p["sel_indices"], p["lo"],
                                         p["hi"], p["block_first"], p["block_last"], p["scale"],
                                         p["block_size"], rows=rows)
    check_out(out, o_ref, rows=rows)
    check_lse(lse[:, rows], l_ref[:, rows])
