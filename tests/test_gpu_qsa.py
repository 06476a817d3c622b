"""GPU parity of the per-query bitmap attention path (device bitmap planner + tcgen05 kernel)
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


def _run(p, max_blocks_per_query=0):
    d = to_dev(p)
    params = pkb.qsa_params(d["q"], d["k"], d["sel_blocks"].shape[1], scale=p["scale"],
                            max_blocks_per_query=max_blocks_per_query)
    meta = pkb.qsa_meta(d["sel_blocks"], d["lo"], d["hi"], d["blk_base"], d["tok_base"],
                        d["block_first"], d["block_last"])
    T, Hq, D = p["q"].shape
    out = torch.full_like(d["q"], 5.0)
    out32 = torch.full(p["q"].shape, 6.0, dtype=torch.float32, device=DEV)
    lse = torch.full((Hq, T), 7.0, dtype=torch.float32, device=DEV)
    ws = torch.empty(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    pkb.paged_attn_plan(params, meta, ws)
    pkb.paged_attn_run(params, meta, d["q"], d["k"], d["v"], out, out32, lse, ws)
    torch.cuda.synchronize()
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.OK, (rc, raw)
    return out, out32, lse, ws, params


def _oracle(p, rows=None):
    return A.qsa_forward(p["q"], p["k"], p["v"], p["sel_blocks"], p["lo"], p["hi"], p["blk_base"],
                         p["tok_base"], p["block_first"], p["block_last"], p["scale"],
                         p["block_size"], rows=rows)


def _check_plan(p, ws, params):
    lay = pkb.plan_layout(params)
    T = p["q"].shape[0]
    indptr = read_ws(ws, lay.indptr_offset, T + 1).numpy()
    ref_ptr, ref_idx = PL.plan_bitmap(p["sel_blocks"], p["lo"], p["hi"], p["block_first"],
                                      p["block_last"])
    assert np.array_equal(indptr, ref_ptr)
    idx = read_ws(ws, lay.indices_offset, int(indptr[-1])).numpy()
    assert np.array_equal(idx, ref_idx)


CASES = [
    # (seq lens, Hq, Hkv, n_near, n_random, lo shift)
    ([64, 128, 40], 24, 2, 4, 8, False),
    ([256], 12, 1, 16, 40, False),
    ([100, 60], 16, 1, 3, 5, True),
    ([48, 8], 2, 2, 2, 100, True),
    ([520], 24, 2, 16, 256, False),
    ([96, 40], 6, 3, 4, 10, False),    # odd Hkv > 1: the last head has no partner
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_qsa_matches_oracle(case):
    lens, Hq, Hkv, near, rand, shift = CASES[case]
    p = W.make_qsa_problem(400 + case, lens, Hq=Hq, Hkv=Hkv, D=256, block_size=4, n_near=near,
                           n_random=rand, scale=1.0 / 16)
    if shift:   # lo inside a block, some rows with lo > hi (empty)
        T = p["q"].shape[0]
        p["lo"] = p["lo"] + torch.tensor([(t * 7) % 5 for t in range(T)], dtype=torch.int32)
    out, out32, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_out(out32, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


def test_qsa_unselected_nonfinite_tokens_do_not_leak():
    # 3-token blocks: the 4th token of every 4-token span belongs to no block, so no query
    # may see it.  It is NaN in K and V; a kernel that loads whole spans must mask it out of
    # both S and the V accumulation.
    p = W.make_qsa_problem(420, [64, 36], Hq=8, Hkv=2, D=256, block_size=4, n_near=3,
                           n_random=6, scale=1.0 / 16)
    p["block_last"] = p["block_first"] + 2
    T = p["q"].shape[0]
    unused = torch.arange(3, T, 4)
    p["k"][unused] = float("nan")
    p["v"][unused] = float("nan")
    out, out32, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    assert np.isfinite(o_ref).all()
    check_out(out, o_ref)
    check_out(out32, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


def test_qsa_capacity_overflow_is_reported():
    p = W.make_qsa_problem(410, [64], Hq=2, Hkv=1, D=256, block_size=4, n_near=4, n_random=8)
    d = to_dev(p)
    params = pkb.qsa_params(d["q"], d["k"], d["sel_blocks"].shape[1], max_blocks_per_query=1)
    meta = pkb.qsa_meta(d["sel_blocks"], d["lo"], d["hi"], d["blk_base"], d["tok_base"],
                        d["block_first"], d["block_last"])
    ws = torch.empty(pkb.paged_attn_workspace_size(params), dtype=torch.uint8, device=DEV)
    pkb.paged_attn_plan(params, meta, ws)
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.ERR_CAPACITY


@pytest.mark.slow
def test_qsa_t32k_workload_sampled():
    """The 32K-token workload in its bench launch configuration.  Compared tokens: the first
    and last 8 of every packed sequence (short and full-length selections) and random tokens
    up to at least 512 in all."""
    p = W.qsa_t32k()
    out, out32, lse, ws, params = _run(p, max_blocks_per_query=272)
    _check_plan(p, ws, params)
    T = p["q"].shape[0]
    starts = np.unique(p["tok_base"].numpy())
    ends = np.concatenate([starts[1:], [T]])
    rows = set()
    for a, e in zip(starts.tolist(), ends.tolist()):
        rows |= set(range(a, a + 8)) | set(range(e - 8, e))
    rng = np.random.default_rng(11)
    while len(rows) < 512:
        rows.add(int(rng.integers(0, T)))
    rows = sorted(rows)
    o_ref, l_ref = _oracle(p, rows=rows)
    check_out(out[rows], o_ref[rows])
    check_out(out32[rows], o_ref[rows])
    check_lse(lse[:, rows], l_ref[:, rows])
