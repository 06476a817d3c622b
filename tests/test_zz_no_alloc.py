"""The decode entry point that allocates nothing (scratch in a fixed array inside the
library).  It exists for callers that cannot allocate device memory when they call in: code
running inside a custom allocator or an out-of-memory handler, plugins whose host framework
owns every device allocation, runtimes whose pool forbids allocations after start-up.

Its results must match the float64 oracle and the regular workspace-based decode on
consecutive calls, so that leftovers of one call in the shared scratch never leak into the
next; the call must leave the device's free memory unchanged; and its status word must be
readable.  Collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, to_dev

pytestmark = pytest.mark.gpu


def _params(p, d, split_chunk):
    return pkb.decode_params(d["q"], d["kv_cache"], p["max_seq_len"], bmm1_scale=p["sm_scale"],
                             mask_type=p["mask_type"], window_left=p["window_left"],
                             split_chunk=split_chunk, seq_len_q=p["seq_len_q"])


def _run_static(p, d, params):
    rows = d["q"].shape[:-1]
    out = torch.full_like(d["q"], 11.0)
    lse = torch.full(rows, 13.0, dtype=torch.float32, device=DEV)
    pkb.paged_decode_run_static(params, d["q"], d["kv_cache"], None, d["kv_indptr"],
                                d["kv_indices"], d["seq_lens"], out, lse)
    return out, lse


def _run_workspace(p, d, params):
    rows = d["q"].shape[:-1]
    ws = torch.empty(pkb.paged_decode_workspace_size(params), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(d["q"])
    lse = torch.empty(rows, dtype=torch.float32, device=DEV)
    pkb.paged_decode_run(params, d["q"], d["kv_cache"], None, d["kv_indptr"], d["kv_indices"],
                         d["seq_lens"], out, lse, ws)
    return out, lse


def _oracle(p):
    return A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                          kv_cache=p["kv_cache"], bmm1_scale=p["sm_scale"],
                          mask_type=p["mask_type"], window_left=p["window_left"],
                          seq_len_q=p["seq_len_q"])


def test_static_scratch_decode_matches_oracle_and_workspace_decode():
    """Three calls in a row with different shapes, each checked against the oracle and the
    workspace route; the last has 16 heads x 8 queries = 128 rows per (request, KV head), so
    it runs the tensor-core route through the same fixed scratch."""
    cases = [
        (W.make_decode_problem(901, [3000, 17, 640, 129], Hq=32, Hkv=8, D=128, page_size=16), 128),
        (W.make_decode_problem(902, [50, 7000], Hq=8, Hkv=2, D=128, page_size=16), 0),
        (W.make_decode_problem(903, [900, 260, 1500], Hq=32, Hkv=2, D=128, page_size=32,
                               seq_len_q=8, mask_type="causal"), 0),
    ]
    for p, chunk in cases:
        d = to_dev(p)
        params = _params(p, d, chunk)
        out, lse = _run_static(p, d, params)
        rc, raw = pkb.paged_decode_static_status()
        assert rc == pkb.OK, (rc, raw)
        out_ref, lse_ref = _run_workspace(p, d, params)
        torch.cuda.synchronize()
        o_ref, l_ref = _oracle(p)
        check_out(out, o_ref)
        check_lse(lse, l_ref)
        check_out(out, out_ref.float().cpu().numpy().astype(np.float64))
        check_lse(lse, lse_ref.cpu().numpy().astype(np.float64))


def test_static_scratch_call_allocates_nothing():
    """Around a repeated call (the first one has looked up the array's address and loaded the
    kernels) the device's free memory does not move."""
    p = W.make_decode_problem(904, [700, 2100, 33], Hq=16, Hkv=4, D=128, page_size=16)
    d = to_dev(p)
    params = _params(p, d, 0)
    _run_static(p, d, params)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:-1], dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    pkb.paged_decode_run_static(params, d["q"], d["kv_cache"], None, d["kv_indptr"],
                                d["kv_indices"], d["seq_lens"], out, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    check_out(out, _oracle(p)[0])


def test_static_status_reports_a_page_outside_the_pool():
    """A page id >= num_pages breaks the contract: the copy of that page is skipped and the
    metadata bit is set; the next good call clears it again."""
    p = W.make_decode_problem(905, [300, 500], Hq=8, Hkv=2, D=128, page_size=16)
    d = to_dev(p)
    params = _params(p, d, 0)
    bad = d["kv_indices"].clone()
    bad[3] = p["num_pages"] + 5
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:-1], dtype=torch.float32, device=DEV)
    pkb.paged_decode_run_static(params, d["q"], d["kv_cache"], None, d["kv_indptr"], bad,
                                d["seq_lens"], out, lse)
    rc, raw = pkb.paged_decode_static_status()
    assert rc == pkb.ERR_METADATA, (rc, raw)
    out, lse = _run_static(p, d, params)
    rc, raw = pkb.paged_decode_static_status()
    assert rc == pkb.OK, (rc, raw)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)


def test_static_scratch_rejects_problems_over_its_size():
    params = pkb.DecodeParams(batch=4096, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                              page_size=16, num_pages=1 << 20, combined_cache=1,
                              max_seq_len=65536, mask_type=0, window_left=-1, bmm1_scale=0.0,
                              bmm2_scale=1.0, split_chunk=128)
    assert pkb.paged_decode_workspace_size(params) > (32 << 20)
    rc = pkb.lib().paged_decode_run_static(params, None, None, None, None, None, None, None,
                                           None, None, None)
    assert rc == pkb.ERR_WORKSPACE
