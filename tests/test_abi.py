"""CPU checks of the C ABI: the library builds and loads, exports every declared entry point,
sizes workspaces from static arguments only, and validates metadata on the host.  Nothing
here launches device work."""
import os
import re

import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from paged_kv_block_gb300 import build as B
from paged_kv_block_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pkb.lib()


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(paged_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    assert pkb.paged_attn_strerror(0) == "ok"
    assert "workspace" in pkb.paged_attn_strerror(pkb.ERR_WORKSPACE)


def _bsr_params(**over):
    kw = dict(form=pkb.FORM_BSR, batch=2, q_len=128, num_qo_heads=8, num_kv_heads=2,
              head_dim=128, page_size=16, num_pages=64, combined_cache=0, q_block_size=64,
              kv_block_size=64, max_seq_len_kv=256, mask_type=1, has_valid_bits=0,
              num_blocks=0, block_size=0, max_blocks_per_query=0, sm_scale=0.0)
    kw.update(over)
    return pkb.AttnParams(**kw)


def test_workspace_sizes_from_static_arguments(lib):
    p = _bsr_params()
    n = pkb.paged_attn_workspace_size(p)
    assert n > 0
    lay = pkb.plan_layout(p)
    # two requests x two KV heads x two q-blocks, one 64-token CTA tile each
    assert lay.tiles_capacity == 8 and lay.tile_tokens == 64
    assert lay.tiles_offset + 32 * lay.tiles_capacity <= n
    for bad in (dict(head_dim=64), dict(kv_block_size=48), dict(q_block_size=1, num_qo_heads=2,
                                                                num_kv_heads=2),
                dict(page_size=12), dict(num_qo_heads=7), dict(mask_type=3)):
        assert pkb.paged_attn_workspace_size(_bsr_params(**bad)) == 0, bad
    dp = pkb.DecodeParams(batch=64, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                          num_pages=100, combined_cache=1, max_seq_len=8192, mask_type=0,
                          window_left=-1, bmm1_scale=0.0, bmm2_scale=1.0, split_chunk=512)
    assert pkb.paged_decode_workspace_size(dp) > 64 * 8 * 16 * 4 * 128 * 4
    assert pkb.paged_decode_split_chunk(dp) == 512
    dp.window_left = 5       # a window needs the causal mask
    assert pkb.paged_decode_workspace_size(dp) == 0
    pp = pkb.PrefillParams(batch=3, total_q=100, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=32, num_pages=10, max_pages_per_request=4, mask_type=1,
                           window_left=-1, sm_scale=0.0, output_scale=1.0)
    assert pkb.paged_prefill_workspace_size(pp) > 0
    pp.page_size = 8         # the prefill page sizes are 16, 32, 64 and 128
    assert pkb.paged_prefill_workspace_size(pp) == 0


def test_validate_bsr_accepts_good_and_rejects_bad_metadata(lib):
    p = W.tiny_bsr()
    params = _bsr_params()
    args = [p["kv_indptr"], p["kv_indices"], p["block_indptr"], p["block_indices"],
            p["seq_lens_kv"]]
    pkb.paged_attn_validate_bsr(params, *args)

    def expect_bad(i, tensor):
        a = list(args)
        a[i] = tensor
        with pytest.raises(pkb.PagedAttnError) as e:
            pkb.paged_attn_validate_bsr(params, *a)
        assert e.value.code == pkb.ERR_METADATA

    bad = p["kv_indices"].clone()
    bad[3] = 64                                   # page id outside the pool
    expect_bad(1, bad)
    bad = p["kv_indptr"].clone()
    bad[1] = 10                                   # request 0 owns too few pages
    expect_bad(0, bad)
    bad = p["block_indices"].clone()
    if bad.numel() > 1:
        bad[1] = bad[0]                           # duplicate block in a row (or across rows)
        row_ptr = p["block_indptr"].flatten()
        if int(row_ptr[1]) - int(row_ptr[0]) >= 2:
            expect_bad(3, bad)
    bad = p["block_indices"].clone()
    bad[0] = 4                                    # block id past max_seq_len_kv / kv_block_size
    expect_bad(3, bad)
    bad = p["seq_lens_kv"].clone()
    bad[0] = 300                                  # longer than max_seq_len_kv
    expect_bad(4, bad)


def test_binding_refuses_host_tensors(lib):
    p = W.tiny_bsr()
    with pytest.raises(ValueError):
        pkb.bsr_meta(p["kv_indptr"], p["kv_indices"], p["block_indptr"], p["block_indices"],
                     p["seq_lens_kv"])
