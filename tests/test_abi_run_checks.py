"""CPU checks of the run entry points' host-side argument checks: a null or misaligned pointer,
invalid static parameters or a workspace that is too small return their status code before
anything is enqueued.  Every call here fails one of those checks, so the placeholder device
addresses below are never used by the library (no copy, memset or launch is issued)."""
import ctypes as C

import pytest

import paged_kv_block_gb300 as pkb
from paged_kv_block_gb300 import build as B

A16 = 0x7F0000100000          # 16-byte aligned placeholder address, never dereferenced
MIS8 = A16 + 8                # 8 bytes off a 16-byte boundary
MIS2 = A16 + 2                # 2 bytes off a 4-byte boundary


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pkb.lib()


def _pp(**kw):
    p = pkb.PrefillParams(batch=3, total_q=100, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                          page_size=32, num_pages=10, max_pages_per_request=4, mask_type=1,
                          window_left=-1, sm_scale=0.0, output_scale=1.0)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _prefill(lib, p, q=A16, k=A16, v=A16, out=A16, ws=A16, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = pkb.paged_prefill_workspace_size(p)
    return lib.paged_prefill_run(C.byref(p), q, k, v, A16, A16, A16, out, None, ws, ws_bytes,
                                 None)


def test_prefill_argument_checks(lib):
    p = _pp()
    assert _prefill(lib, p, q=None) == pkb.ERR_INVALID_ARGUMENT
    assert _prefill(lib, p, q=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _prefill(lib, p, v=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _prefill(lib, p, out=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _prefill(lib, p, ws=None) == pkb.ERR_WORKSPACE
    assert _prefill(lib, p, ws_bytes=16) == pkb.ERR_WORKSPACE
    assert _prefill(lib, _pp(out_dtype=7), ws_bytes=16) == pkb.ERR_INVALID_ARGUMENT
    assert _prefill(lib, _pp(head_dim=64), ws_bytes=16) == pkb.ERR_INVALID_ARGUMENT


def _dp(**kw):
    p = pkb.DecodeParams(batch=4, num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                         num_pages=64, combined_cache=1, max_seq_len=1024, mask_type=0,
                         window_left=-1, bmm1_scale=0.0, bmm2_scale=1.0, split_chunk=0)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _decode(lib, p, query=A16, k=A16, v=None, qo=None, out=A16, ws=A16, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = pkb.paged_decode_workspace_size(p)
    return lib.paged_decode_run(C.byref(p), query, k, v, A16, A16, A16, qo, out, None, ws,
                                ws_bytes, None)


def test_decode_argument_checks(lib):
    p = _dp()
    assert _decode(lib, p, query=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _decode(lib, p, out=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _decode(lib, p, qo=A16) == pkb.ERR_INVALID_ARGUMENT      # qo_indptr without the packed form
    assert _decode(lib, _dp(combined_cache=0)) == pkb.ERR_INVALID_ARGUMENT   # V pool missing
    assert _decode(lib, p, ws=None) == pkb.ERR_WORKSPACE
    assert _decode(lib, p, ws_bytes=16) == pkb.ERR_WORKSPACE
    packed = _dp(max_seq_len_q=4, total_q=10)
    assert _decode(lib, packed) == pkb.ERR_INVALID_ARGUMENT          # packed form without qo_indptr
    assert _decode(lib, packed, qo=A16, ws_bytes=16) == pkb.ERR_WORKSPACE
    assert _decode(lib, _dp(out_dtype=5), ws_bytes=16) == pkb.ERR_INVALID_ARGUMENT


def _sp(**kw):
    p = pkb.SageParams(batch=1, num_heads=2, q_len=128, kv_len=256, head_dim=128, capacity=4,
                       block_sparse_num=4, uniform_block_count=1, block_sizes_rank=0,
                       softmax_scale=0.0)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _sage(lib, p, q=A16, k=A16, v=A16, out=A16, ws=A16, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = pkb.paged_sage_workspace_size(p)
    return lib.paged_sage_run(C.byref(p), q, k, v, A16, A16, A16, A16, None, None, out, ws,
                              ws_bytes, None)


def test_sage_argument_checks_come_before_any_work(lib):
    p = _sp()
    assert _sage(lib, p, out=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _sage(lib, p, q=None) == pkb.ERR_INVALID_ARGUMENT
    assert _sage(lib, p, q=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert _sage(lib, p, v=MIS2) == pkb.ERR_INVALID_ARGUMENT       # FP8 V needs 4-byte alignment
    assert _sage(lib, p, v=A16 + 4, ws_bytes=16) == pkb.ERR_WORKSPACE
    assert _sage(lib, p, ws=None) == pkb.ERR_WORKSPACE
    assert _sage(lib, _sp(head_dim=64), ws_bytes=16) == pkb.ERR_INVALID_ARGUMENT
    assert _sage(lib, _sp(block_sizes_rank=2)) == pkb.ERR_INVALID_ARGUMENT   # block_sizes missing


def test_sparse_run_argument_checks(lib):
    p = pkb.AttnParams(form=0, batch=2, q_len=128, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                       page_size=16, num_pages=64, combined_cache=0, q_block_size=64,
                       kv_block_size=64, max_seq_len_kv=256, mask_type=1, has_valid_bits=0,
                       sm_scale=0.0)
    m = pkb.AttnMeta()
    n = pkb.paged_attn_workspace_size(p)

    def run(q=A16, k=A16, v=A16, out=A16, ws=A16, ws_bytes=n):
        return lib.paged_attn_run(C.byref(p), C.byref(m), q, k, v, out, None, None, ws,
                                  ws_bytes, None)

    assert run(q=None) == pkb.ERR_INVALID_ARGUMENT
    assert run(ws=None) == pkb.ERR_WORKSPACE
    assert run(ws_bytes=16) == pkb.ERR_WORKSPACE
    # block-sparse: the output must start on a 16-byte boundary as well
    m.kv_indptr_dev = m.block_indptr_dev = m.seq_lens_kv_dev = A16
    assert run(out=MIS8) == pkb.ERR_INVALID_ARGUMENT
    assert run(k=MIS8) == pkb.ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("form", [1, 2])
def test_bitmap_run_argument_checks(lib, form):
    """The bitmap and indexed forms refuse a missing V, missing bounds, unaligned tensors
    (out_fp32 included) and an unsupported head size or group before any work."""
    def params(**kw):
        p = pkb.AttnParams(form=form, batch=1, q_len=64, num_qo_heads=24, num_kv_heads=2,
                           head_dim=256, num_blocks=16, block_size=4, max_blocks_per_query=16,
                           sm_scale=0.0, index_width=8)
        for k, v in kw.items():
            setattr(p, k, v)
        return p

    m = pkb.AttnMeta(lo_dev=A16, hi_dev=A16, block_first_dev=A16, block_last_dev=A16,
                     sel_blocks_dev=A16, sel_indices_dev=A16, blk_base_dev=A16, tok_base_dev=A16)

    def run(p, q=A16, k=A16, v=A16, out=A16, out32=None, meta=m):
        n = pkb.paged_attn_workspace_size(p)
        return lib.paged_attn_run(C.byref(p), C.byref(meta), q, k, v, out, out32, None, A16,
                                  max(n, 16), None)

    p = params()
    assert run(p, v=None) == pkb.ERR_INVALID_ARGUMENT
    for bad in (dict(q=MIS8), dict(k=MIS8), dict(v=MIS8), dict(out=MIS8), dict(out32=MIS8)):
        assert run(p, **bad) == pkb.ERR_INVALID_ARGUMENT, bad
    no_hi = pkb.AttnMeta(lo_dev=A16, block_first_dev=A16, block_last_dev=A16,
                         sel_blocks_dev=A16, sel_indices_dev=A16)
    assert run(p, meta=no_hi) == pkb.ERR_INVALID_ARGUMENT
    assert run(params(head_dim=128)) == pkb.ERR_INVALID_ARGUMENT        # D = 256 only
    assert run(params(num_qo_heads=40, num_kv_heads=2)) == pkb.ERR_UNSUPPORTED   # G = 20 > 16
