"""GPU parity of the packed-Q prefill path with head dimension 256 (the prefill planner with
128 / G tokens per tile + the D = 256 tensor-core kernel) against the float64 oracle,
through the C ABI."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from oracle import planner as PL
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, read_ws, to_dev

pytestmark = pytest.mark.gpu

D = 256


def _run(p, out_dtype=torch.bfloat16):
    d = to_dev(p)
    T, Hq, _ = p["q"].shape
    B = p["seq_lens_kv"].numel()
    out = torch.full(p["q"].shape, 5.0, dtype=out_dtype, device=DEV)
    lse = torch.full((T, Hq), 9.0, dtype=torch.float32, device=DEV)
    params = pkb.prefill_params(d["q"], d["k_cache"], d["block_tables"], B,
                                mask_type=p["mask_type"], window_left=p["window_left"],
                                sm_scale=p["sm_scale"], output_scale=p["output_scale"],
                                out_dtype=out_dtype)
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
    G = params.num_qo_heads // params.num_kv_heads
    assert lay.tile_tokens == 128 // G                   # one 128-row sub-tile per tile
    n = int(read_ws(ws, lay.count_offset, 1)[0])
    recs = read_ws(ws, lay.tiles_offset, 8 * n).numpy().reshape(-1, 8)
    ref = PL.plan_prefill_tiles(params.num_kv_heads, p["qo_indptr"], p["seq_lens_kv"],
                                lay.tile_tokens, p["mask_type"], p["window_left"])
    assert np.array_equal(recs, ref)


CASES = [
    # (q_lens, prefixes, Hq, Hkv, page size, mask, window, output scale)
    ([200, 56, 300], [100, 0, 640], 8, 2, 32, "causal", -1, 1.0),
    ([128, 1, 77], [0, 500, 33], 4, 4, 16, "dense", -1, 0.5),
    ([333, 64], [900, 0], 16, 2, 64, "causal", 200, 1.0),     # G = 8: 16 tokens per tile
    ([500], [1100], 12, 2, 128, "causal", 37, 1.25),          # G = 6: 126 live rows of 128
    ([40, 90], [0, 7], 24, 2, 16, "dense", -1, 1.0),          # G = 12: 120 live rows
    ([1, 2, 3], [0, 0, 0], 2, 1, 32, "causal", 0, 1.0),       # tiny, window 0
    ([150, 70], [213, 30], 8, 2, 16, "causal", -1, 1.0),      # 8 K and 2 V page pieces
    ([260, 45], [0, 700], 4, 2, 128, "causal", 100, 1.0),     # one page per KV tile, window
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill256_matches_oracle(case):
    q_lens, prefix, Hq, Hkv, ps, mask, win, oscale = CASES[case]
    p = W.make_prefill_problem(600 + case, q_lens, prefix, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                               mask_type=mask, window_left=win, output_scale=oscale)
    out, lse, ws, params = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    _check_plan(p, ws, params)


def test_prefill256_output_types():
    p = W.make_prefill_problem(610, [150, 260], [60, 300], Hq=8, Hkv=2, D=D, page_size=32,
                               mask_type="causal", window_left=120)
    o_ref, l_ref = _oracle(p)
    outs = {}
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        out, lse, _, _ = _run(p, dt)
        check_out(out, o_ref)
        check_lse(lse, l_ref)
        outs[dt] = out
    assert torch.equal(outs[torch.float32].to(torch.bfloat16), outs[torch.bfloat16])


def test_prefill256_more_queries_than_keys_gives_empty_rows():
    """Causal with more queries than keys is outside the contract; queries before the first
    key see nothing and get 0 / -inf, the rest are exact."""
    p = W.make_prefill_problem(611, [40], [0], Hq=4, Hkv=1, D=D, page_size=16,
                               mask_type="causal")
    p["seq_lens_kv"] = torch.tensor([25], dtype=torch.int32)
    out, lse, _, _ = _run(p)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)
    assert torch.all(out[:15].float() == 0) and torch.all(torch.isneginf(lse[:15]))


@pytest.mark.slow
def test_prefill256_b16_sampled():
    rng = np.random.default_rng(7)
    q_lens = rng.integers(128, 2048, size=16, endpoint=True)
    prefix = rng.integers(0, 2048, size=16, endpoint=True)
    p = W.make_prefill_problem(612, q_lens, prefix, Hq=16, Hkv=4, D=D, page_size=32,
                               mask_type="causal")
    out, lse, _, _ = _run(p)
    T = p["q"].shape[0]
    rows = sorted(set([0, 1, T - 1] + list(rng.integers(0, T, 60))))
    o_ref, l_ref = _oracle(p, rows=rows)
    check_out(out, o_ref, rows=rows)
    check_lse(lse[rows], l_ref[rows])


@pytest.mark.slow
def test_prefill_b16_d256_workload_sampled():
    """The bench workload at its full size: 40 random rows plus every request's first and last
    row against the oracle, and the whole plan bit for bit."""
    p = W.prefill_b16_d256()
    out, lse, ws, params = _run(p)
    qo = p["qo_indptr"].numpy()
    rng = np.random.default_rng(8)
    rows = set(rng.integers(0, int(qo[-1]), 40).tolist())
    for b in range(len(qo) - 1):
        rows |= {int(qo[b]), int(qo[b + 1]) - 1}
    rows = sorted(rows)
    o_ref, l_ref = _oracle(p, rows=rows)
    check_out(out[rows], o_ref[rows])
    check_lse(lse[rows], l_ref[rows])
    _check_plan(p, ws, params)
