"""The decode entry point that allocates nothing (scratch in a fixed array inside the
library), for callers that cannot allocate device memory when they call in.  Its results
must match the regular workspace-based decode on consecutive calls, so that leftovers of one
call in the shared scratch never leak into the next.  Collected last on purpose."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, to_dev

pytestmark = pytest.mark.gpu


def _decode_both(p, split_chunk):
    d = to_dev(p)
    B, Hq, _ = p["q"].shape
    params = pkb.decode_params(d["q"], d["kv_cache"], p["max_seq_len"], bmm1_scale=p["sm_scale"],
                               split_chunk=split_chunk)
    ws = torch.empty(pkb.paged_decode_workspace_size(params), dtype=torch.uint8, device=DEV)
    out_ref = torch.empty_like(d["q"])
    lse_ref = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    pkb.paged_decode_run(params, d["q"], d["kv_cache"], None, d["kv_indptr"], d["kv_indices"],
                         d["seq_lens"], out_ref, lse_ref, ws)
    out = torch.full_like(d["q"], 11.0)
    lse = torch.full((B, Hq), 13.0, dtype=torch.float32, device=DEV)
    pkb.paged_decode_run_static(params, d["q"], d["kv_cache"], None, d["kv_indptr"],
                                d["kv_indices"], d["seq_lens"], out, lse)
    torch.cuda.synchronize()
    return out, lse, out_ref, lse_ref


def test_static_scratch_decode_matches_workspace_decode_twice():
    # two calls in a row with different shapes: the second must not see the first's scratch
    cases = [W.make_decode_problem(901, [3000, 17, 640, 129], Hq=32, Hkv=8, D=128, page_size=16),
             W.make_decode_problem(902, [50, 7000], Hq=8, Hkv=2, D=128, page_size=16)]
    for p, chunk in zip(cases, (128, 0)):
        out, lse, out_ref, lse_ref = _decode_both(p, chunk)
        check_out(out, out_ref.float().cpu().numpy().astype(np.float64))
        check_lse(lse, lse_ref.cpu().numpy().astype(np.float64))


def test_static_scratch_rejects_problems_over_its_size():
    params = pkb.DecodeParams(batch=4096, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                              page_size=16, num_pages=1 << 20, combined_cache=1,
                              max_seq_len=65536, mask_type=0, window_left=-1, bmm1_scale=0.0,
                              bmm2_scale=1.0, split_chunk=128)
    assert pkb.paged_decode_workspace_size(params) > (32 << 20)
    rc = pkb.lib().paged_decode_run_static(params, None, None, None, None, None, None, None,
                                           None, None, None)
    assert rc == pkb.ERR_WORKSPACE
