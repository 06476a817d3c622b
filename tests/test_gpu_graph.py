"""The run entry points do no device-to-host synchronisation and read every piece of metadata
on the device, so a launch can be captured once in a CUDA graph and replayed after the caller
rewrites the metadata in place (new lengths, page tables and query rows within the same
static bounds).  Each replay is checked against the float64 oracle."""
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out

pytestmark = pytest.mark.gpu


def _pad_rows(t, n, fill=0):
    """t with its first dimension padded to n rows of `fill`."""
    out = torch.full((n,) + tuple(t.shape[1:]), fill, dtype=t.dtype)
    out[: t.shape[0]] = t
    return out


def test_decode_graph_replay_with_new_metadata():
    Hq, Hkv, D, ps, max_len = 16, 4, 128, 16, 3000
    probs = [W.make_decode_problem(130, [2900, 17, 1200, 640], Hq=Hq, Hkv=Hkv, D=D, page_size=ps),
             W.make_decode_problem(131, [5, 2999, 300, 2048], Hq=Hq, Hkv=Hkv, D=D, page_size=ps)]
    P = max(p["kv_cache"].shape[0] for p in probs)
    NI = max(p["kv_indices"].numel() for p in probs)
    B = 4
    # device buffers sized for both problems; the graph captures their addresses
    q = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
    cache = torch.empty((P,) + tuple(probs[0]["kv_cache"].shape[1:]), dtype=torch.bfloat16,
                        device=DEV)
    indptr = torch.empty(B + 1, dtype=torch.int32, device=DEV)
    indices = torch.empty(NI, dtype=torch.int32, device=DEV)
    lens = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=DEV)
    params = pkb.decode_params(q, cache, max_len, split_chunk=256)
    ws = torch.zeros(pkb.paged_decode_workspace_size(params), dtype=torch.uint8, device=DEV)

    def stage(p):
        q.copy_(p["q"])
        cache.copy_(_pad_rows(p["kv_cache"], P))
        indptr.copy_(p["kv_indptr"])
        indices.copy_(_pad_rows(p["kv_indices"], NI))
        lens.copy_(p["seq_lens"])

    def run():
        pkb.paged_decode_run(params, q, cache, None, indptr, indices, lens, out, lse, ws)

    stage(probs[0])
    run()                                       # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for p in probs:
        stage(p)
        out.fill_(3.0)
        g.replay()
        torch.cuda.synchronize()
        rc, raw = pkb.paged_attn_workspace_status(ws)
        assert rc == pkb.OK, (rc, raw)
        o_ref, l_ref = A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                                      kv_cache=p["kv_cache"], bmm1_scale=p["sm_scale"],
                                      bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                                      window_left=p["window_left"])
        check_out(out, o_ref)
        check_lse(lse, l_ref)


def test_prefill_graph_replay_with_new_metadata():
    Hq, Hkv, D, ps = 8, 2, 128, 32
    probs = [W.make_prefill_problem(140, [200, 56, 300], [100, 0, 640], Hq=Hq, Hkv=Hkv, D=D,
                                    page_size=ps),
             W.make_prefill_problem(141, [1, 400, 155], [900, 33, 0], Hq=Hq, Hkv=Hkv, D=D,
                                    page_size=ps)]
    T = probs[0]["q"].shape[0]
    assert all(p["q"].shape[0] == T for p in probs)
    P = max(p["k_cache"].shape[0] for p in probs)
    C = max(p["block_tables"].shape[1] for p in probs)
    B = 3
    q = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=DEV)
    kc = torch.empty((P,) + tuple(probs[0]["k_cache"].shape[1:]), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    qo = torch.empty(B + 1, dtype=torch.int32, device=DEV)
    bt = torch.empty((B, C), dtype=torch.int32, device=DEV)
    lens = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=DEV)
    params = pkb.prefill_params(q, kc, bt, B, mask_type="causal", window_left=-1,
                                sm_scale=probs[0]["sm_scale"])
    ws = torch.zeros(pkb.paged_prefill_workspace_size(params), dtype=torch.uint8, device=DEV)

    def stage(p):
        q.copy_(p["q"])
        kc.copy_(_pad_rows(p["k_cache"], P))
        vc.copy_(_pad_rows(p["v_cache"], P))
        qo.copy_(p["qo_indptr"])
        t = torch.zeros((B, C), dtype=torch.int32)
        t[:, : p["block_tables"].shape[1]] = p["block_tables"]
        bt.copy_(t)
        lens.copy_(p["seq_lens_kv"])

    def run():
        pkb.paged_prefill_run(params, q, kc, vc, qo, bt, lens, out, lse, ws)

    stage(probs[0])
    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for p in probs:
        stage(p)
        out.fill_(5.0)
        g.replay()
        torch.cuda.synchronize()
        rc, raw = pkb.paged_attn_workspace_status(ws)
        assert rc == pkb.OK, (rc, raw)
        o_ref, l_ref = A.batch_prefill(p["q"], p["k_cache"], p["v_cache"], p["qo_indptr"],
                                       p["block_tables"], p["seq_lens_kv"],
                                       mask_type=p["mask_type"], window_left=p["window_left"],
                                       sm_scale=p["sm_scale"], output_scale=p["output_scale"])
        check_out(out, o_ref)
        check_lse(lse, l_ref)
