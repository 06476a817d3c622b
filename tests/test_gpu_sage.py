"""GPU parity of the prequantized block-sparse attention (int8 Q/K, FP8 E4M3 V, fp32 scales;
exact bf16 copies + the block-sparse tensor-core kernel with scales) against the float64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import paged_kv_block_gb300 as pkb
from oracle import attention as A
from paged_kv_block_gb300 import workloads as W
from tests.gpu_util import DEV, check_out

pytestmark = pytest.mark.gpu


def _run(p, idx=None, nums=None, uniform_flag=False, expect=pkb.OK):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    idx = d["q2k_block_index"] if idx is None else idx.to(DEV)
    nums = d["q2k_block_nums"] if nums is None else nums.to(DEV)
    out = torch.full(p["q_int8"].shape, 3.0, dtype=torch.bfloat16, device=DEV)
    params = pkb.sage_params(d["q_int8"], d["k_int8"], idx, p["block_sparse_num"],
                             block_sizes=d["block_sizes"], softmax_scale=p["softmax_scale"],
                             uniform_block_count=uniform_flag)
    ws = torch.zeros(pkb.paged_sage_workspace_size(params), dtype=torch.uint8, device=DEV)
    pkb.paged_sage_run(params, d["q_int8"], d["k_int8"], d["v_fp8"], d["q_scale"], d["k_scale"],
                       d["v_scale"], idx, nums, d["block_sizes"], out, ws)
    torch.cuda.synchronize()
    rc, raw = pkb.paged_attn_workspace_status(ws)
    assert rc == expect, (rc, raw)
    return out


def _oracle(p, idx=None, nums=None):
    return A.sage_block_sparse_attention(
        p["q_int8"], p["k_int8"], p["v_fp8"], p["q_scale"], p["k_scale"], p["v_scale"],
        p["q2k_block_index"] if idx is None else idx, p["block_sparse_num"], p["block_sizes"],
        p["q2k_block_nums"] if nums is None else nums, p["softmax_scale"])


def _flat(x):
    """[B, H, S, D] as [B * H * S, 1, D] rows (a tensor stays a tensor)."""
    return x.reshape(-1, 1, x.shape[-1])


CASES = [
    dict(B=2, H=4, Sq=300, Sk=1000, capacity=6, sizes="bhnb", empty_rows=0.2),
    dict(B=1, H=2, Sq=128, Sk=640, uniform=3, sizes="none"),
    dict(B=3, H=1, Sq=64, Sk=64, capacity=1, sizes="nb"),
    dict(B=2, H=2, Sq=1, Sk=130, capacity=3, sizes="bnb"),
    dict(B=1, H=8, Sq=200, Sk=2048, capacity=12, sizes="none"),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_sage_matches_oracle(case):
    p = W.make_sage_problem(700 + case, **CASES[case])
    out = _run(p, uniform_flag=CASES[case].get("uniform") is not None)
    check_out(_flat(out), _flat(_oracle(p)))


def test_sage_uniform_count_without_per_row_counts():
    p = W.make_sage_problem(710, B=1, H=3, Sq=190, Sk=700, uniform=4, sizes="bhnb")
    out = _run(p)                                  # counts NULL: block_sparse_num applies
    check_out(_flat(out), _flat(_oracle(p)))


def test_sage_out_of_range_ids_and_counts_are_reported():
    p = W.make_sage_problem(711, B=1, H=2, Sq=128, Sk=500, capacity=4, sizes="none")
    idx = p["q2k_block_index"].clone()
    nums = p["q2k_block_nums"].clone()
    idx[0, 0, 0, 0] = 99                           # past NB = 8: dropped
    nums[0, 1, 1] = 4                              # the whole row, valid ids
    out = _run(p, idx=idx, nums=nums, expect=pkb.ERR_METADATA)
    check_out(_flat(out), _flat(_oracle(p, idx=idx, nums=nums)))


def test_sage_rows_without_blocks_are_exactly_zero():
    p = W.make_sage_problem(712, B=1, H=2, Sq=150, Sk=300, capacity=2, sizes="none")
    nums = torch.zeros_like(p["q2k_block_nums"])
    out = _run(p, nums=nums)
    assert torch.all(out.float() == 0)


def test_sage_no_keys_gives_zeros():
    p = W.make_sage_problem(713, B=1, H=1, Sq=70, Sk=64, capacity=1, sizes="none")
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    params = pkb.sage_params(d["q_int8"], d["k_int8"][:, :, :0], d["q2k_block_index"], 0)
    ws = torch.zeros(pkb.paged_sage_workspace_size(params), dtype=torch.uint8, device=DEV)
    out = torch.full(p["q_int8"].shape, 3.0, dtype=torch.bfloat16, device=DEV)
    pkb.paged_sage_run(params, d["q_int8"], d["k_int8"], d["v_fp8"], d["q_scale"], d["k_scale"],
                       d["v_scale"], d["q2k_block_index"], None, None, out, ws)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0)


@pytest.mark.slow
def test_sage_b2h16_workload_sampled():
    """The bench workload at its full size (B=2, H=16, Sq=Sk=4096, 16 blocks per query block):
    four (b, h) slices against the oracle, which treats every (b, h) independently."""
    p = W.sage_b2h16()
    out = _run(p, uniform_flag=True)
    for b, h in ((0, 0), (0, 9), (1, 7), (1, 15)):
        sub = {k: (v[b:b + 1, h:h + 1] if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
        check_out(_flat(out[b:b + 1, h:h + 1]), _flat(_oracle(sub)))
