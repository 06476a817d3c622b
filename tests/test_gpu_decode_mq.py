"""GPU parity of multi-query decode (prims_ts_batch_decode_with_kv_cache with seq_len_q > 1 or
packed qo_indptr) against the float64 oracle, through the C ABI.

Units of at most 64 rows (G x queries) run on the split-KV decode kernel in 1, 2 or 4
row blocks; larger units take the tensor-core tile route.  Both plans are compared bit for
bit with the planner oracle."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from oracle import planner as PL
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, read_ws, to_dev

pytestmark = pytest.mark.gpu


def _run(p, split_chunk=0, max_seq_len_q=None):
    d = to_dev(p)
    cache = d["kv_cache"] if "kv_cache" in d else (d["k_cache"], d["v_cache"])
    qo = d.get("qo_indptr")
    lse = torch.full(tuple(p["q"].shape[:-1]), 7.0, dtype=torch.float32, device=DEV)
    out = torch.full_like(d["q"], 3.0)
    params = pkb.decode_params(d["q"], cache, p["max_seq_len"], bmm1_scale=p["sm_scale"],
                               bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                               window_left=p["window_left"], split_chunk=split_chunk,
                               seq_len_q=p["seq_len_q"], qo_indptr=qo,
                               max_seq_len_q=max_seq_len_q or p["max_seq_len_q"])
    ws = torch.empty(pkb.paged_decode_workspace_size(params), dtype=torch.uint8, device=DEV)
    k, v = (cache, None) if not isinstance(cache, tuple) else cache
    pkb.paged_decode_run(params, d["q"], k, v, d["kv_indptr"], d["kv_indices"], d["seq_lens"],
                         out, lse, ws, qo_indptr=qo)
    torch.cuda.synchronize()
    return out, lse, ws, params


def _oracle(p):
    return A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                          kv_cache=p.get("kv_cache"), k_cache=p.get("k_cache"),
                          v_cache=p.get("v_cache"), bmm1_scale=p["sm_scale"],
                          bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                          window_left=p["window_left"], seq_len_q=p["seq_len_q"],
                          qo_indptr=p["qo_indptr"])


def _qo(p):
    q_lens = np.asarray(p["q_lens"], np.int64)
    return np.concatenate([[0], np.cumsum(q_lens)])


def _check_plan(p, ws, params):
    lay = pkb.plan_layout(params)
    lens = [int(x) for x in p["seq_lens"]]
    Hkv = params.num_kv_heads
    if lay.split_chunk:                              # split-KV route
        B = len(lens)
        off = read_ws(ws, lay.split_offset_offset, B + 1).numpy()
        off_ref, items_ref = PL.plan_decode(lens, Hkv, lay.split_chunk, p["window_left"],
                                            q_lens=p["q_lens"])
        assert np.array_equal(off, off_ref)
        items = read_ws(ws, lay.items_offset, 4 * Hkv * int(off[-1])).numpy().reshape(-1, 4)
        assert np.array_equal(items, items_ref)
        order = read_ws(ws, lay.order_offset, len(items_ref)).numpy()
        assert np.array_equal(order, PL.decode_work_order(items_ref, lay.split_chunk))
    else:                                            # tile route
        n = int(read_ws(ws, lay.count_offset, 1)[0])
        recs = read_ws(ws, lay.tiles_offset, 8 * n).numpy().reshape(-1, 8)
        ref = PL.plan_prefill_tiles(Hkv, _qo(p), lens, lay.tile_tokens, p["mask_type"],
                                    p["window_left"])
        assert np.array_equal(recs, ref)


CASES = [
    # (lens, Hq, Hkv, ps, combined, mask, window, bmm2, chunk, seq_len_q, q_lens)
    ([1500, 40, 700], 16, 4, 16, True, "causal", -1, 1.0, 256, 4, None),        # 16 rows
    ([300, 2000], 4, 2, 32, False, "dense", -1, 0.5, 0, 3, None),              # 6 rows
    ([900, 64, 3100], 24, 3, 16, True, "causal", 150, 1.0, 384, 3, None),      # 24 rows
    ([1200, 333], 8, 2, 64, False, "causal", -1, 1.0, 128, 16, None),          # 64 rows
    ([800, 50, 1000], 16, 1, 128, True, "causal", 40, 2.0, 256, 3, None),      # 48 rows
    ([1000, 2, 517, 64], 16, 4, 16, False, "causal", 100, 1.0, 256, 1, [1, 3, 8, 5]),  # packed
    ([2100, 700], 8, 8, 8, True, "dense", -1, 1.0, 0, 1, [7, 2]),               # packed, 7 rows
    ([2000, 900], 32, 4, 16, True, "causal", -1, 1.0, 0, 16, None),            # tiled: 128 rows
    ([1300, 5, 800], 16, 4, 32, False, "causal", 64, 1.0, 0, 1, [20, 4, 17]),  # tiled: 80 rows
    ([777, 1500], 8, 2, 24, True, "causal", -1, 1.0, 256, 4, None),           # page size 24
    ([1000, 130], 8, 2, 48, False, "dense", -1, 1.0, 128, 1, None),           # page size 48
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_multi_query_decode_matches_oracle(case):
    lens, Hq, Hkv, ps, comb, mask, win, s2, chunk, sq, q_lens = CASES[case]
    p = W.make_decode_problem(300 + case, lens, Hq=Hq, Hkv=Hkv, D=128, page_size=ps,
                              combined=comb, mask_type=mask, window_left=win, bmm2_scale=s2,
                              seq_len_q=sq, q_lens=q_lens)
    out, lse, ws, params = _run(p, chunk)
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.OK, (rc, raw)
    o_ref, l_ref = _oracle(p)
    check_out(out.reshape(-1, Hq, 128), o_ref.reshape(-1, Hq, 128))
    check_lse(lse.reshape(-1, Hq), l_ref.reshape(-1, Hq))
    _check_plan(p, ws, params)


def test_packed_bound_larger_than_every_request():
    """max_seq_len_q above every request's count: the rows past a request's queries are
    computed but never written."""
    p = W.make_decode_problem(320, [600, 90, 1200], Hq=8, Hkv=2, D=128, page_size=16,
                              q_lens=[2, 1, 3], mask_type="causal")
    out, lse, ws, _ = _run(p, 256, max_seq_len_q=6)
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.OK, (rc, raw)
    o_ref, l_ref = _oracle(p)
    check_out(out, o_ref)
    check_lse(lse, l_ref)


def test_packed_offsets_over_the_bound_are_reported():
    """A request with more queries than max_seq_len_q breaks the packed contract: the plan
    reports it and no row outside the output is written."""
    p = W.make_decode_problem(321, [400, 300], Hq=4, Hkv=1, D=128, page_size=16,
                              q_lens=[5, 3], mask_type="causal")
    out, lse, ws, _ = _run(p, 128, max_seq_len_q=4)
    rc, _ = pkb.paged_attn_workspace_status(ws)
    assert rc == pkb.ERR_METADATA
    # request 1 stays within its bound and its rows are right
    o_ref, l_ref = _oracle(p)
    check_out(out[5:], o_ref[5:])
    check_lse(lse[5:], l_ref[5:])


def test_fixed_form_equals_packed_form():
    p = W.make_decode_problem(322, [1700, 300, 45], Hq=16, Hkv=4, D=128, page_size=16,
                              seq_len_q=3, mask_type="causal", window_left=200)
    o_fix, l_fix, _, _ = _run(p, 256)
    packed = dict(p, q=p["q"].reshape(9, 16, 128), seq_len_q=1, max_seq_len_q=3,
                  qo_indptr=torch.tensor([0, 3, 6, 9], dtype=torch.int32), q_lens=[3, 3, 3])
    o_pk, l_pk, _, _ = _run(packed, 256)
    assert torch.equal(o_fix.reshape(9, 16, 128), o_pk)
    assert torch.equal(l_fix.reshape(9, 16), l_pk)


@pytest.mark.slow
def test_decode_b64_sq4_workload_sampled():
    """The four-query bench workload at its full size (B=64, SQ=4, causal): the plan and the
    claim order bit for bit, and the output and LSE of the shortest, the longest and a few
    random requests against the oracle."""
    p = W.decode_b64_sq4()
    out, lse, ws, params = _run(p)
    _check_plan(p, ws, params)
    lens = p["seq_lens"].numpy()
    reqs = {int(np.argmin(lens)), int(np.argmax(lens)), 0, int(lens.size) - 1}
    reqs |= set(np.random.default_rng(9).integers(0, lens.size, 2).tolist())
    reqs = sorted(reqs)
    o_ref, l_ref = A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                                  kv_cache=p.get("kv_cache"), k_cache=p.get("k_cache"),
                                  v_cache=p.get("v_cache"), bmm1_scale=p["sm_scale"],
                                  bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                                  window_left=p["window_left"], seq_len_q=p["seq_len_q"],
                                  qo_indptr=p["qo_indptr"], rows=reqs)
    check_out(out[reqs].reshape(-1, out.shape[-2], out.shape[-1]),
              o_ref[reqs].reshape(-1, o_ref.shape[-2], o_ref.shape[-1]))
    check_lse(lse[reqs].reshape(-1, lse.shape[-1]), l_ref[reqs].reshape(-1, l_ref.shape[-1]))
