"""Helpers shared by the GPU parity tests (tolerances from the parity contract)."""
import numpy as np
import torch

OUT_MAX_ABS = 2e-2     # bf16 output, max |gpu - oracle|
OUT_MEAN_ABS = 2e-3    # bf16 output, mean |gpu - oracle|
LSE_ABS = 1e-3         # fp32 LSE, max |gpu - oracle|

DEV = torch.device("cuda:0")


def to_dev(prob):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in prob.items()}


def check_out(out, ref, rows=None, max_abs=OUT_MAX_ABS, mean_abs=OUT_MEAN_ABS):
    """out: GPU tensor; ref: float64 array (NaN marks rows the oracle did not compute)."""
    o = out.float().cpu().numpy().astype(np.float64)
    r = np.asarray(ref)
    if rows is not None:
        o, r = o[rows], r[rows]
    mask = ~np.isnan(r)
    assert mask.any()
    assert np.all(np.isfinite(o[mask])), "non-finite output"
    d = np.abs(o[mask] - r[mask])
    assert d.max() <= max_abs, f"max abs err {d.max()}"
    assert d.mean() <= mean_abs, f"mean abs err {d.mean()}"
    return d.max(), d.mean()


def check_lse(lse, ref, tol=LSE_ABS):
    l = lse.float().cpu().numpy().astype(np.float64)
    r = np.asarray(ref)
    mask = ~np.isnan(r)
    ninf_r = np.isneginf(r) & mask
    assert np.array_equal(np.isneginf(l) & mask, ninf_r), "-inf rows differ"
    fin = mask & ~ninf_r
    if fin.any():
        d = np.abs(l[fin] - r[fin])
        assert np.all(np.isfinite(l[fin]))
        assert d.max() <= tol, f"lse max abs err {d.max()}"
        return d.max()
    return 0.0


def read_ws(workspace, offset, count, dtype=torch.int32):
    """Copy `count` elements of `dtype` at byte `offset` of a workspace back to the host."""
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return workspace[offset:offset + nbytes].cpu().view(dtype).clone()
