"""Output element types ([PRE] and [DEC] out_dtype): bf16, fp16 and fp32 outputs of the prefill
and decode paths against the float64 oracle, and the fp32 output rounded to bf16 equal, bit
for bit, to the bf16 output of the same launch configuration."""
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_lse, check_out, to_dev

pytestmark = pytest.mark.gpu


def _prefill(p, dtype):
    d = to_dev(p)
    out, lse = pkb.batch_prefill_with_paged_kv_cache(
        d["q"], d["k_cache"], d["v_cache"], d["qo_indptr"], d["block_tables"], d["seq_lens_kv"],
        page_size=p["page_size"], mask_type=p["mask_type"], window_left=p["window_left"],
        sm_scale=p["sm_scale"], output_scale=p["output_scale"], out_dtype=dtype,
        lse=torch.empty(p["q"].shape[:2], dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    assert out.dtype == dtype
    return out, lse


def _decode(p, dtype, split_chunk=0):
    d = to_dev(p)
    lse = torch.empty(tuple(p["q"].shape[:-1]), dtype=torch.float32, device=DEV)
    out, lse = pkb.batch_decode_with_paged_kv_cache(
        d["q"], d["kv_cache"], None, d["kv_indptr"], d["kv_indices"], d["seq_lens"],
        p["max_seq_len"], seq_len_q=p["seq_len_q"], qo_indptr=d["qo_indptr"],
        max_seq_len_q=p["max_seq_len_q"] if p["qo_indptr"] is not None else None,
        bmm1_scale=p["sm_scale"], bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
        window_left=p["window_left"], out_dtype=dtype, lse=lse, split_chunk=split_chunk)
    torch.cuda.synchronize()
    assert out.dtype == dtype
    return out, lse


def _check_all(run, ref):
    o_ref, l_ref = ref
    outs = {}
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        o, l = run(dt)
        check_out(o.reshape(-1, o.shape[-2], o.shape[-1]),
                  o_ref.reshape(-1, o.shape[-2], o.shape[-1]))
        check_lse(l.reshape(-1, l.shape[-1]), l_ref.reshape(-1, l.shape[-1]))
        outs[dt] = o
    assert torch.equal(outs[torch.float32].to(torch.bfloat16), outs[torch.bfloat16])


def test_prefill_output_types():
    p = W.make_prefill_problem(500, [300, 77, 129], [100, 0, 700], Hq=16, Hkv=4, D=128,
                               page_size=32, mask_type="causal", window_left=250,
                               output_scale=0.75)
    ref = A.batch_prefill(p["q"], p["k_cache"], p["v_cache"], p["qo_indptr"], p["block_tables"],
                          p["seq_lens_kv"], mask_type="causal", window_left=250,
                          sm_scale=p["sm_scale"], output_scale=0.75)
    _check_all(lambda dt: _prefill(p, dt), ref)


def _decode_ref(p):
    return A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                          kv_cache=p["kv_cache"], bmm1_scale=p["sm_scale"],
                          bmm2_scale=p["bmm2_scale"], mask_type=p["mask_type"],
                          window_left=p["window_left"], seq_len_q=p["seq_len_q"],
                          qo_indptr=p["qo_indptr"])


@pytest.mark.parametrize("kw", [
    dict(seq_lens=[2000, 40, 900], Hq=16, Hkv=4, mask_type="dense", bmm2_scale=1.5),
    dict(seq_lens=[1500, 333], Hq=16, Hkv=4, mask_type="causal", seq_len_q=3),
    dict(seq_lens=[1200, 90], Hq=32, Hkv=2, mask_type="causal", q_lens=[9, 5]),  # tile route
])
def test_decode_output_types(kw):
    kw = dict(kw)
    lens = kw.pop("seq_lens")
    p = W.make_decode_problem(501, lens, D=128, page_size=16, **kw)
    _check_all(lambda dt: _decode(p, dt, split_chunk=256), _decode_ref(p))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_prefill_output_at_16_byte_offset(D, dt):
    """An output that is 16- but not 32-byte aligned takes the 16-byte store path of the
    epilogue; it must hold exactly what the aligned output holds."""
    p = W.make_prefill_problem(502, [200, 65], [50, 300], Hq=8, Hkv=2, D=D, page_size=32,
                               mask_type="causal")
    aligned, _ = _prefill(p, dt)
    n = aligned.numel()
    shift = 16 // aligned.element_size()
    buf = torch.full((n + shift,), 7.0, dtype=dt, device=DEV)
    view = buf[shift:].view(aligned.shape)
    assert view.data_ptr() % 32 == 16
    d = to_dev(p)
    pkb.batch_prefill_with_paged_kv_cache(
        d["q"], d["k_cache"], d["v_cache"], d["qo_indptr"], d["block_tables"], d["seq_lens_kv"],
        page_size=p["page_size"], mask_type=p["mask_type"], window_left=p["window_left"],
        sm_scale=p["sm_scale"], output_scale=p["output_scale"], out=view)
    torch.cuda.synchronize()
    assert torch.equal(view, aligned)
    assert torch.all(buf[:shift] == 7.0)
