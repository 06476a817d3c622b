"""GPU parity of the packed-Q paged prefill path (device planner + tcgen05 kernel) against the
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


def _run(p):
    d = to_dev(p)
    T, Hq, D = p["q"].shape
    B = p["seq_lens_kv"].numel()
    out = torch.full_like(d["q"], 5.0)
    lse = torch.full((T, Hq), 9.0, dtype=torch.float32, device=DEV)
    params = pkb.prefill_params(d["q"], d["k_cache"], d["block_tables"], B,
                                mask_type=p["mask_type"], window_left=p["window_left"],
                                sm_scale=p["sm_scale"], output_scale=p["output_scale"])
    ws = torch.empty(pkb.paged_prefill_workspace_size(params), dtype=torch.uint8, device=DEV)
    pkb.paged_prefill_run(params, d["q"], d["k_cache"], d["v_cache"], d["qo_indptr"],
                          d["block_tables"], d["seq_lens_kv"], out, lse, ws)
    torch.cuda.synchronize()
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.OK, (rc, raw)
    return out, lse, ws, params


def _oracle(p, rows=None):
    return A.batch_prefill(p["q"], p["k_cache"], p["v_cache"], p["qo_indptr"], p["block_tables"],
                           p["seq_lens_kv"], mask_type=p["mask_type"],
                           window_left=p["window_left"], sm_scale=p["sm_scale"],
                           output_scale=p["output_scale"], rows=rows)


def _check_plan(p, ws, params):
    lay = pkb.plan_layout(params)
    n = int(read_ws(ws, lay.count_offset, 1)[0])
    recs = read_ws(ws, lay.tiles_offset, 8 * n).numpy().reshape(-1, 8)
    ref = PL.plan_prefill_tiles(params.num_kv_heads, p["qo_indptr"], p["seq_lens_kv"],
                                lay.tile_tokens, p["mask_type"], p["window_left"])
    assert np.array_equal(recs, ref)


CASES = [
    # (q_lens, prefix, Hq, Hkv, ps, mask, window, oscale)
    ([1, 70, 130, 5], [0, 10, 300, 0], 8, 2, 16, "causal", -1, 1.0),
    ([64, 200], [100, 0], 32, 8, 32, "causal", 63, 1.0),
    ([33, 129], [7, 130], 4, 4, 64, "dense", -1, 0.7),
    ([300], [260], 16, 2, 128, "causal", 0, 1.0),
    ([257, 31, 96], [0, 400, 1], 8, 1, 32, "causal", 200, 2.0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_matches_oracle(case):
    q_lens, prefix, Hq, Hkv, ps, mask, win, osc = CASES[case]
    p = W.make_prefill_problem(300 + case, q_lens, prefix, Hq=Hq, Hkv=Hkv, D=128, page_size=ps,
                               mask_type=mask, window_left=win, output_scale=osc)
    out, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


@pytest.mark.slow
@pytest.mark.parametrize("window", [-1, 1023])
def test_prefill_b16_workload_sampled(window):
    """The 16-request workload in its bench launch configuration.  Compared rows: every row
    of the shortest request, of the last 16 work tiles in launch order (the tail of the
    persistent grid) and of each request's last tile (a ragged second sub-tile), the first
    and last row of every request, and random rows."""
    p = W.prefill_b16(window_left=window)
    out, lse, ws, params = _run(p)
    _check_plan(p, ws, params)
    lay = pkb.plan_layout(params)
    n = int(read_ws(ws, lay.count_offset, 1)[0])
    recs = read_ws(ws, lay.tiles_offset, 8 * n).numpy().reshape(-1, 8)
    qo = p["qo_indptr"].numpy()
    nq = qo[1:] - qo[:-1]
    rows = set()
    b_min = int(np.argmin(nq))
    rows |= set(range(int(qo[b_min]), int(qo[b_min + 1])))
    for b, g, tok0, ntok, kv0, kv1, row0, _ in recs[-16:]:
        rows |= set(range(int(row0), int(row0) + int(ntok)))
    for b in range(len(nq)):
        last = recs[(recs[:, 0] == b) & (recs[:, 2] + recs[:, 3] == nq[b])]
        assert len(last) > 0
        row0, ntok = int(last[0, 6]), int(last[0, 3])
        rows |= set(range(row0, row0 + ntok))
        rows |= {int(qo[b]), int(qo[b + 1]) - 1}
    rng = np.random.default_rng(7)
    rows |= set(rng.integers(0, int(qo[-1]), 40).tolist())
    rows = sorted(rows)
    o_ref, l_ref = _oracle(p, rows=rows)
    check_out(out[rows], o_ref[rows])
    check_lse(lse[rows], l_ref[rows])
