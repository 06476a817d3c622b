"""GPU parity of the split-KV paged decode path (plan + partial kernel + merge) against the
float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from oracle import planner as PL
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, read_ws, to_dev

pytestmark = pytest.mark.gpu


def _run(p, split_chunk=0, stream=None):
    d = to_dev(p)
    if "kv_cache" in d:
        cache = d["kv_cache"]
    else:
        cache = (d["k_cache"], d["v_cache"])
    B, Hq, _ = p["q"].shape
    lse = torch.full((B, Hq), 7.0, dtype=torch.float32, device=DEV)
    out = torch.full_like(d["q"], 3.0)
    params = pkb.decode_params(d["q"], cache, p["max_seq_len"], bmm1_scale=p["sm_scale"],
                               bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                               window_left=p["window_left"], split_chunk=split_chunk)
    ws = torch.empty(pkb.paged_decode_workspace_size(params), dtype=torch.uint8, device=DEV)
    k, v = (cache, None) if not isinstance(cache, tuple) else cache
    pkb.paged_decode_run(params, d["q"], k, v, d["kv_indptr"], d["kv_indices"], d["seq_lens"],
                         out, lse, ws, stream)
    torch.cuda.synchronize()
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.OK, (rc, raw)
    return out, lse, ws, params


def _oracle(p):
    return A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                          kv_cache=p.get("kv_cache"), k_cache=p.get("k_cache"),
                          v_cache=p.get("v_cache"), bmm1_scale=p["sm_scale"],
                          bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                          window_left=p["window_left"])


CASES = [
    # (lens, Hq, Hkv, page_size, combined, mask, window, bmm2, split_chunk)
    ([1, 2, 15, 16, 17, 63, 64, 65, 300], 8, 2, 16, True, "dense", -1, 1.0, 128),
    ([1000, 129, 7], 32, 8, 16, True, "dense", -1, 1.0, 0),
    ([513, 2048, 77], 4, 4, 32, False, "causal", -1, 0.5, 256),
    ([900, 5, 1500], 16, 1, 64, True, "causal", 100, 1.0, 128),
    ([700, 3000], 16, 2, 128, False, "causal", 0, 2.0, 384),
    ([4100, 31], 8, 1, 8, True, "dense", -1, 1.0, 0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_matches_oracle(case):
    lens, Hq, Hkv, ps, comb, mask, win, s2, chunk = CASES[case]
    p = W.make_decode_problem(100 + case, lens, Hq=Hq, Hkv=Hkv, D=128, page_size=ps,
                              combined=comb, mask_type=mask, window_left=win, bmm2_scale=s2)
    out, lse, ws, params = _run(p, chunk)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    # the split plan is bit-exact against the planner oracle
    lay = pkb.plan_layout(params)
    B = len(lens)
    off = read_ws(ws, lay.split_offset_offset, B + 1).numpy()
    off_ref, items_ref = PL.plan_decode(lens, Hkv, lay.split_chunk, win)
    assert np.array_equal(off, off_ref)
    items = read_ws(ws, lay.items_offset, 4 * Hkv * int(off[-1])).numpy().reshape(-1, 4)
    assert np.array_equal(items, items_ref)
    order = read_ws(ws, lay.order_offset, len(items_ref)).numpy()
    assert np.array_equal(order, PL.decode_work_order(items_ref, lay.split_chunk))
    if chunk:
        assert lay.split_chunk == chunk


def test_split_count_does_not_change_the_result():
    p = W.make_decode_problem(120, [5000, 2500, 800], Hq=8, Hkv=2, D=128, page_size=16)
    outs = [_run(p, c)[:2] for c in (128, 1024, 8192)]
    o_ref, l_ref = _oracle(p)
    for o, l in outs:
        check_out(o, o_ref)
        check_lse(l, l_ref)


def test_auto_chunk_matches_formula():
    p = W.make_decode_problem(121, [100, 9000], Hq=32, Hkv=8, D=128, page_size=16)
    d = to_dev(p)
    params = pkb.decode_params(d["q"], d["kv_cache"], 8192 + 1000)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert pkb.paged_decode_split_chunk(params) == PL.decode_split_chunk(2, 8, 9192, sms)


@pytest.mark.slow
def test_decode_b64_full_workload():
    p = W.decode_b64()
    out, lse, ws, params = _run(p, 0)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    lay = pkb.plan_layout(params)
    off = read_ws(ws, lay.split_offset_offset, 65).numpy()
    off_ref, items_ref = PL.plan_decode(p["seq_lens"], 8, lay.split_chunk)
    assert np.array_equal(off, off_ref)
    items = read_ws(ws, lay.items_offset, 4 * 8 * int(off[-1])).numpy().reshape(-1, 4)
    assert np.array_equal(items, items_ref)
