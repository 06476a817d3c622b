"""Python binding of libpagedattn, the GB300 paged-KV attention forward library.

Argument marshalling only: every step of the computation (planning included) runs in the
library's CUDA kernels.  The low-level functions carry the C ABI's names
(``paged_attn_plan``, ``paged_attn_run``, ``paged_prefill_run``, ``paged_decode_run``, ...)
and take torch tensors; the convenience functions below them follow the argument names of
the FlashInfer pages (block_sparse_attention_with_paged_kv_cache,
batch_prefill_with_paged_kv_cache, prims_ts_batch_decode_with_kv_cache, qsa_forward).

The library must be built first (``paged_kv_block_gb300.build.build()``); importing works
without it, but any call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedattn.so")

FORM_BSR, FORM_BITMAP, FORM_INDEXED = 0, 1, 2
MASK = {"dense": 0, "causal": 1}
DTYPE = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}

OK = 0
ERR_INVALID_ARGUMENT = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5
ERR_METADATA = -6
ERR_CAPACITY = -7


class AttnParams(C.Structure):
    _fields_ = [("form", C.c_int), ("batch", C.c_int), ("q_len", C.c_int),
                ("num_qo_heads", C.c_int), ("num_kv_heads", C.c_int), ("head_dim", C.c_int),
                ("page_size", C.c_int), ("num_pages", C.c_int), ("combined_cache", C.c_int),
                ("q_block_size", C.c_int), ("kv_block_size", C.c_int),
                ("max_seq_len_kv", C.c_int), ("mask_type", C.c_int), ("has_valid_bits", C.c_int),
                ("num_blocks", C.c_int), ("block_size", C.c_int),
                ("max_blocks_per_query", C.c_int), ("sm_scale", C.c_float),
                ("index_width", C.c_int)]


class AttnMeta(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "kv_indptr_dev", "kv_indices_dev", "block_indptr_dev", "block_indices_dev",
        "seq_lens_kv_dev", "kv_valid_bits_dev", "sel_blocks_dev", "lo_dev", "hi_dev",
        "blk_base_dev", "tok_base_dev", "block_first_dev", "block_last_dev",
        "sel_indices_dev")]


class PrefillParams(C.Structure):
    _fields_ = [("batch", C.c_int), ("total_q", C.c_int), ("num_qo_heads", C.c_int),
                ("num_kv_heads", C.c_int), ("head_dim", C.c_int), ("page_size", C.c_int),
                ("num_pages", C.c_int), ("max_pages_per_request", C.c_int),
                ("mask_type", C.c_int), ("window_left", C.c_int), ("sm_scale", C.c_float),
                ("output_scale", C.c_float), ("out_dtype", C.c_int)]


class DecodeParams(C.Structure):
    _fields_ = [("batch", C.c_int), ("num_qo_heads", C.c_int), ("num_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("page_size", C.c_int), ("num_pages", C.c_int),
                ("combined_cache", C.c_int), ("max_seq_len", C.c_int), ("mask_type", C.c_int),
                ("window_left", C.c_int), ("bmm1_scale", C.c_float), ("bmm2_scale", C.c_float),
                ("split_chunk", C.c_int), ("seq_len_q", C.c_int), ("max_seq_len_q", C.c_int),
                ("total_q", C.c_int), ("out_dtype", C.c_int)]


class SageParams(C.Structure):
    _fields_ = [("batch", C.c_int), ("num_heads", C.c_int), ("q_len", C.c_int),
                ("kv_len", C.c_int), ("head_dim", C.c_int), ("capacity", C.c_int),
                ("block_sparse_num", C.c_int), ("uniform_block_count", C.c_int),
                ("block_sizes_rank", C.c_int), ("softmax_scale", C.c_float)]


class PlanLayout(C.Structure):
    _fields_ = [("status_offset", C.c_size_t), ("tiles_offset", C.c_size_t),
                ("tiles_capacity", C.c_int64), ("count_offset", C.c_size_t),
                ("indptr_offset", C.c_size_t), ("indices_offset", C.c_size_t),
                ("indices_capacity", C.c_int64), ("split_offset_offset", C.c_size_t),
                ("items_offset", C.c_size_t), ("items_capacity", C.c_int64),
                ("split_chunk", C.c_int), ("tile_tokens", C.c_int),
                ("order_offset", C.c_size_t)]


_LIB = None
_EXPORTS = {
    "paged_attn_workspace_size": (C.c_size_t, [C.POINTER(AttnParams)]),
    "paged_attn_validate_bsr": (C.c_int, [C.POINTER(AttnParams), C.c_void_p, C.c_void_p,
                                          C.c_int64, C.c_void_p, C.c_void_p, C.c_int64,
                                          C.c_void_p, C.POINTER(C.c_int64)]),
    "paged_attn_plan": (C.c_int, [C.POINTER(AttnParams), C.POINTER(AttnMeta), C.c_void_p,
                                  C.c_size_t, C.c_void_p]),
    "paged_attn_run": (C.c_int, [C.POINTER(AttnParams), C.POINTER(AttnMeta), C.c_void_p,
                                 C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                 C.c_void_p, C.c_size_t, C.c_void_p]),
    "paged_prefill_workspace_size": (C.c_size_t, [C.POINTER(PrefillParams)]),
    "paged_prefill_run": (C.c_int, [C.POINTER(PrefillParams)] + [C.c_void_p] * 9
                          + [C.c_size_t, C.c_void_p]),
    "paged_decode_workspace_size": (C.c_size_t, [C.POINTER(DecodeParams)]),
    "paged_decode_split_chunk": (C.c_int, [C.POINTER(DecodeParams)]),
    "paged_decode_run": (C.c_int, [C.POINTER(DecodeParams)] + [C.c_void_p] * 10
                         + [C.c_size_t, C.c_void_p]),
    "paged_attn_plan_layout_of": (C.c_int, [C.POINTER(AttnParams), C.POINTER(PlanLayout)]),
    "paged_prefill_plan_layout_of": (C.c_int, [C.POINTER(PrefillParams), C.POINTER(PlanLayout)]),
    "paged_decode_plan_layout_of": (C.c_int, [C.POINTER(DecodeParams), C.POINTER(PlanLayout)]),
    "paged_decode_run_static": (C.c_int, [C.POINTER(DecodeParams)] + [C.c_void_p] * 10),
    "paged_decode_static_status": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32)]),
    "paged_attn_workspace_status": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(C.c_uint32)]),
    "paged_sage_workspace_size": (C.c_size_t, [C.POINTER(SageParams)]),
    "paged_sage_run": (C.c_int, [C.POINTER(SageParams)] + [C.c_void_p] * 11
                       + [C.c_size_t, C.c_void_p]),
    "paged_attn_strerror": (C.c_char_p, [C.c_int]),
    "paged_attn_kernel_timer": (C.c_int, [C.c_int]),
    "paged_attn_kernel_timer_read": (C.c_int, [C.POINTER(C.c_double), C.POINTER(C.c_int64)]),
    "paged_attn_launch_count": (C.c_int64, []),
    "paged_attn_l2_read_probe": (C.c_int, [C.c_void_p, C.c_size_t, C.c_int, C.c_void_p,
                                           C.c_void_p]),
}


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "paged_kv_block_gb300.build.build()")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _EXPORTS.items():
            f = getattr(h, name)
            f.restype, f.argtypes = res, args
        _LIB = h
    return _LIB


class PagedAttnError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {paged_attn_strerror(code)} ({code})")


def _check(code, what):
    if code != OK:
        raise PagedAttnError(code, what)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return C.c_void_p(t.data_ptr())


def _dev(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------------------
# C ABI, one function per entry point
# ---------------------------------------------------------------------------------------

def paged_attn_strerror(code: int) -> str:
    return lib().paged_attn_strerror(int(code)).decode()


def paged_attn_workspace_size(params: AttnParams) -> int:
    return int(lib().paged_attn_workspace_size(C.byref(params)))


def paged_attn_validate_bsr(params, kv_indptr, kv_indices, block_indptr, block_indices,
                            seq_lens_kv) -> None:
    """Host-side metadata validation (host int32 tensors).  Raises PagedAttnError."""
    ts = [t.detach().to("cpu", torch.int32).contiguous() for t in
          (kv_indptr, kv_indices, block_indptr, block_indices, seq_lens_kv)]
    bad = C.c_int64(-1)
    rc = lib().paged_attn_validate_bsr(C.byref(params), _ptr(ts[0]), _ptr(ts[1]), ts[1].numel(),
                                       _ptr(ts[2]), _ptr(ts[3]), ts[3].numel(), _ptr(ts[4]),
                                       C.byref(bad))
    if rc != OK:
        raise PagedAttnError(rc, f"paged_attn_validate_bsr (item {bad.value})")


def paged_attn_plan(params: AttnParams, meta: AttnMeta, workspace, stream=None) -> None:
    _check(lib().paged_attn_plan(C.byref(params), C.byref(meta), _dev(workspace, "workspace"),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "paged_attn_plan")


def paged_attn_run(params: AttnParams, meta: AttnMeta, q, k, v, out, out_fp32, lse, workspace,
                   stream=None) -> None:
    _check(lib().paged_attn_run(C.byref(params), C.byref(meta), _dev(q, "q"), _dev(k, "k"),
                                _dev(v, "v"), _dev(out, "out"), _dev(out_fp32, "out_fp32"),
                                _dev(lse, "lse"), _dev(workspace, "workspace"),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "paged_attn_run")


def paged_prefill_workspace_size(params: PrefillParams) -> int:
    return int(lib().paged_prefill_workspace_size(C.byref(params)))


def paged_prefill_run(params: PrefillParams, q, k_cache, v_cache, qo_indptr, block_tables,
                      seq_lens_kv, out, lse, workspace, stream=None) -> None:
    _check(lib().paged_prefill_run(C.byref(params), _dev(q, "q"), _dev(k_cache, "k_cache"),
                                   _dev(v_cache, "v_cache"), _dev(qo_indptr, "qo_indptr"),
                                   _dev(block_tables, "block_tables"),
                                   _dev(seq_lens_kv, "seq_lens_kv"), _dev(out, "out"),
                                   _dev(lse, "lse"), _dev(workspace, "workspace"),
                                   workspace.numel() * workspace.element_size(),
                                   _stream(stream)),
           "paged_prefill_run")


def paged_decode_workspace_size(params: DecodeParams) -> int:
    return int(lib().paged_decode_workspace_size(C.byref(params)))


def paged_decode_split_chunk(params: DecodeParams) -> int:
    return int(lib().paged_decode_split_chunk(C.byref(params)))


def paged_decode_run(params: DecodeParams, query, k, v, kv_indptr, kv_indices, seq_lens, out,
                     lse, workspace, stream=None, qo_indptr=None) -> None:
    """qo_indptr: packed query offsets (params.max_seq_len_q > 0), else None."""
    _check(lib().paged_decode_run(C.byref(params), _dev(query, "query"), _dev(k, "k"),
                                  _dev(v, "v"), _dev(kv_indptr, "kv_indptr"),
                                  _dev(kv_indices, "kv_indices"), _dev(seq_lens, "seq_lens"),
                                  _dev(qo_indptr, "qo_indptr"),
                                  _dev(out, "out"), _dev(lse, "lse"),
                                  _dev(workspace, "workspace"),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "paged_decode_run")


def plan_layout(params) -> PlanLayout:
    """Where the plan of `params` (any of the three parameter structs) sits in the
    workspace."""
    o = PlanLayout()
    fn = {AttnParams: lib().paged_attn_plan_layout_of,
          PrefillParams: lib().paged_prefill_plan_layout_of,
          DecodeParams: lib().paged_decode_plan_layout_of}[type(params)]
    _check(fn(C.byref(params), C.byref(o)), "plan_layout")
    return o


def paged_decode_run_static(params: DecodeParams, query, k, v, kv_indptr, kv_indices, seq_lens,
                            out, lse, stream=None, qo_indptr=None) -> None:
    """paged_decode_run for callers that cannot allocate: the scratch is a fixed array
    inside the library (see the C header for its size and the sharing rules)."""
    _check(lib().paged_decode_run_static(C.byref(params), _dev(query, "query"), _dev(k, "k"),
                                         _dev(v, "v"), _dev(kv_indptr, "kv_indptr"),
                                         _dev(kv_indices, "kv_indices"),
                                         _dev(seq_lens, "seq_lens"),
                                         _dev(qo_indptr, "qo_indptr"), _dev(out, "out"),
                                         _dev(lse, "lse"), _stream(stream)),
           "paged_decode_run_static")


def paged_decode_static_status(stream=None):
    """(status code, raw word) of the last paged_decode_run_static call on the current
    device; synchronises the stream."""
    raw = C.c_uint32(0)
    rc = lib().paged_decode_static_status(_stream(stream), C.byref(raw))
    return rc, raw.value


def paged_attn_workspace_status(workspace, stream=None):
    """(status code, raw word) of the device status word; synchronises the stream."""
    raw = C.c_uint32(0)
    rc = lib().paged_attn_workspace_status(_dev(workspace, "workspace"), _stream(stream),
                                           C.byref(raw))
    return rc, raw.value


def paged_attn_kernel_timer(enable: bool) -> None:
    _check(lib().paged_attn_kernel_timer(int(bool(enable))), "paged_attn_kernel_timer")


def paged_attn_kernel_timer_read():
    """(total milliseconds, launches) of the main kernels bracketed since enabling."""
    ms, n = C.c_double(0.0), C.c_int64(0)
    _check(lib().paged_attn_kernel_timer_read(C.byref(ms), C.byref(n)),
           "paged_attn_kernel_timer_read")
    return ms.value, n.value


def paged_attn_l2_read_probe(buf, reps, sink, stream=None) -> None:
    """Enqueue the L2 read-rate probe over the bytes of `buf` (a device tensor)."""
    _check(lib().paged_attn_l2_read_probe(_dev(buf, "buf"), buf.numel() * buf.element_size(),
                                          int(reps), _dev(sink, "sink"), _stream(stream)),
           "paged_attn_l2_read_probe")


def paged_attn_launch_count() -> int:
    return int(lib().paged_attn_launch_count())


def _workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------------------
# Convenience forms with the pages' argument names
# ---------------------------------------------------------------------------------------

def _pools(paged_kv_cache):
    """(k_arg, v_arg, combined, Hkv, page_size, num_pages, D) of a combined cache tensor
    [P, 2, Hkv, ps, D] or a (K, V) tuple of [P, Hkv, ps, D] pools."""
    if isinstance(paged_kv_cache, (tuple, list)):
        k, v = paged_kv_cache
        P, Hkv, ps, D = k.shape
        return k, v, 0, Hkv, ps, P, D
    P, two, Hkv, ps, D = paged_kv_cache.shape
    assert two == 2
    return paged_kv_cache, None, 1, Hkv, ps, P, D


def bsr_params(q, paged_kv_cache, q_block_size, kv_block_size, max_seq_len_kv, *,
               has_valid_bits=False, mask_type="dense", sm_scale=None) -> AttnParams:
    B, Sq, Hq, D = q.shape
    _, _, combined, Hkv, ps, P, _ = _pools(paged_kv_cache)
    return AttnParams(form=FORM_BSR, batch=B, q_len=Sq, num_qo_heads=Hq, num_kv_heads=Hkv,
                      head_dim=D, page_size=ps, num_pages=P, combined_cache=combined,
                      q_block_size=q_block_size, kv_block_size=kv_block_size,
                      max_seq_len_kv=int(max_seq_len_kv), mask_type=MASK[mask_type],
                      has_valid_bits=int(bool(has_valid_bits)), num_blocks=0, block_size=0,
                      max_blocks_per_query=0, sm_scale=float(sm_scale or 0.0))


def bsr_meta(paged_kv_indptr, paged_kv_indices, block_indptr, block_indices, seq_lens_kv,
             kv_valid_bits=None) -> AttnMeta:
    m = AttnMeta()
    m.kv_indptr_dev = _dev(paged_kv_indptr, "paged_kv_indptr")
    m.kv_indices_dev = _dev(paged_kv_indices, "paged_kv_indices")
    m.block_indptr_dev = _dev(block_indptr, "block_indptr")
    m.block_indices_dev = _dev(block_indices, "block_indices")
    m.seq_lens_kv_dev = _dev(seq_lens_kv, "seq_lens_kv")
    m.kv_valid_bits_dev = _dev(kv_valid_bits, "kv_valid_bits")
    return m


def block_sparse_attention_with_paged_kv_cache(q, paged_kv_cache, paged_kv_indptr,
                                               paged_kv_indices, block_indptr, block_indices,
                                               q_block_size, kv_block_size, *, max_seq_len_kv,
                                               seq_lens_kv, kv_valid_bits=None,
                                               mask_type="dense", sm_scale=None, out=None,
                                               lse=None, workspace=None, stream=None):
    """Plan + run one block-sparse launch; returns (out, lse)."""
    params = bsr_params(q, paged_kv_cache, q_block_size, kv_block_size, max_seq_len_kv,
                        has_valid_bits=kv_valid_bits is not None, mask_type=mask_type,
                        sm_scale=sm_scale)
    meta = bsr_meta(paged_kv_indptr, paged_kv_indices, block_indptr, block_indices,
                    seq_lens_kv, kv_valid_bits)
    k, v, *_ = _pools(paged_kv_cache)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = _workspace(paged_attn_workspace_size(params), q.device)
    paged_attn_plan(params, meta, workspace, stream)
    paged_attn_run(params, meta, q, k, v, out, None, lse, workspace, stream)
    return out, lse


def _out_dtype(out_dtype, out, q):
    """[PRE]/[DEC] out_dtype: the given dtype, else out's dtype when out is given, else the
    query's dtype."""
    dt = out_dtype if out_dtype is not None else (out.dtype if out is not None else q.dtype)
    if dt not in DTYPE:
        raise ValueError(f"unsupported output dtype {dt}")
    if out is not None and out.dtype != dt:
        raise ValueError("out does not have out_dtype")
    return dt


def prefill_params(q, k_cache, block_tables, batch, *, mask_type="dense", window_left=-1,
                   sm_scale=None, output_scale=1.0, out_dtype=torch.bfloat16) -> PrefillParams:
    total_q, Hq, D = q.shape
    P, Hkv, ps, _ = k_cache.shape
    return PrefillParams(batch=batch, total_q=total_q, num_qo_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, page_size=ps, num_pages=P,
                         max_pages_per_request=block_tables.shape[1],
                         mask_type=MASK[mask_type], window_left=int(window_left),
                         sm_scale=float(sm_scale or 0.0), output_scale=float(output_scale),
                         out_dtype=DTYPE[out_dtype])


def batch_prefill_with_paged_kv_cache(q, k_cache, v_cache, qo_indptr, block_tables, seq_lens_kv,
                                      *, page_size=32, kv_layout="HND", mask_type="dense",
                                      window_left=-1, sm_scale=None, output_scale=1.0,
                                      out_dtype=None, out=None, lse=None, workspace=None,
                                      stream=None):
    """Plan + run one packed-Q prefill launch; returns (out, lse)."""
    out_dtype = _out_dtype(out_dtype, out, q)
    if kv_layout != "HND":
        raise ValueError("only the HND layout is supported")
    if k_cache.shape[2] != page_size:
        raise ValueError("page_size does not match the pools")
    params = prefill_params(q, k_cache, block_tables, seq_lens_kv.numel(), mask_type=mask_type,
                            window_left=window_left, sm_scale=sm_scale,
                            output_scale=output_scale, out_dtype=out_dtype)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = _workspace(paged_prefill_workspace_size(params), q.device)
    paged_prefill_run(params, q, k_cache, v_cache, qo_indptr, block_tables, seq_lens_kv, out, lse,
                      workspace, stream)
    return out, lse


def decode_params(query, kv_cache, max_seq_len, *, bmm1_scale=None, bmm2_scale=1.0,
                  mask_type="dense", window_left=-1, split_chunk=0, seq_len_q=1,
                  qo_indptr=None, max_seq_len_q=None, out_dtype=torch.bfloat16) -> DecodeParams:
    """Static arguments of a decode call.  query is [B, Hq, D] (one query per request),
    [B, SQ, Hq, D] (seq_len_q = SQ > 1) or packed [total_q, Hq, D] with qo_indptr, whose
    static bound max_seq_len_q is then required."""
    _, _, combined, Hkv, ps, P, _ = _pools(kv_cache)
    sq, max_sq, total_q = 1, 0, 0
    if qo_indptr is not None:
        if max_seq_len_q is None:
            raise ValueError("the packed form needs max_seq_len_q")
        total_q, Hq, D = query.shape
        B = qo_indptr.numel() - 1
        max_sq = int(max_seq_len_q)
    elif seq_len_q > 1:
        B, sq, Hq, D = query.shape
        if sq != seq_len_q:
            raise ValueError("query.shape[1] must equal seq_len_q")
    else:
        B, Hq, D = query.shape
    return DecodeParams(batch=B, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=ps,
                        num_pages=P, combined_cache=combined, max_seq_len=int(max_seq_len),
                        mask_type=MASK[mask_type], window_left=int(window_left),
                        bmm1_scale=float(bmm1_scale or 0.0), bmm2_scale=float(bmm2_scale),
                        split_chunk=int(split_chunk), seq_len_q=int(sq), max_seq_len_q=max_sq,
                        total_q=int(total_q), out_dtype=DTYPE[out_dtype])


def batch_decode_with_paged_kv_cache(query, kv_cache, workspace_buffer, paged_kv_indptr,
                                     paged_kv_indices, seq_lens, max_seq_len, *, seq_len_q=1,
                                     qo_indptr=None, max_seq_len_q=None, bmm1_scale=None,
                                     bmm2_scale=1.0, out=None, out_dtype=None, lse=None,
                                     mask_type="dense", window_left=-1, kv_layout="HND",
                                     split_chunk=0, stream=None):
    """Decode with split-KV over a CSR page table; returns (out, lse).  One query per
    request ([B, Hq, D]), seq_len_q fixed queries ([B, SQ, Hq, D]) or packed queries
    ([total_q, Hq, D] with qo_indptr and its bound max_seq_len_q)."""
    if kv_layout != "HND":
        raise ValueError("only the HND layout is supported")
    out_dtype = _out_dtype(out_dtype, out, query)
    params = decode_params(query, kv_cache, max_seq_len, bmm1_scale=bmm1_scale,
                           bmm2_scale=bmm2_scale, mask_type=mask_type, window_left=window_left,
                           split_chunk=split_chunk, seq_len_q=seq_len_q, qo_indptr=qo_indptr,
                           max_seq_len_q=max_seq_len_q, out_dtype=out_dtype)
    k, v, *_ = _pools(kv_cache)
    if out is None:
        out = torch.empty(query.shape, dtype=out_dtype, device=query.device)
    if workspace_buffer is None:
        workspace_buffer = _workspace(paged_decode_workspace_size(params), query.device)
    paged_decode_run(params, query, k, v, paged_kv_indptr, paged_kv_indices, seq_lens, out, lse,
                     workspace_buffer, stream, qo_indptr=qo_indptr)
    return out, lse


def qsa_params(q, k, num_blocks, *, scale=0.0625, block_size=4,
               max_blocks_per_query=0) -> AttnParams:
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    return AttnParams(form=FORM_BITMAP, batch=1, q_len=T, num_qo_heads=Hq, num_kv_heads=Hkv,
                      head_dim=D, page_size=0, num_pages=0, combined_cache=0, q_block_size=0,
                      kv_block_size=0, max_seq_len_kv=0, mask_type=0, has_valid_bits=0,
                      num_blocks=int(num_blocks), block_size=int(block_size),
                      max_blocks_per_query=int(max_blocks_per_query), sm_scale=float(scale))


def qsa_meta(sel_blocks, lo, hi, blk_base, tok_base, block_first, block_last) -> AttnMeta:
    m = AttnMeta()
    m.sel_blocks_dev = _dev(sel_blocks, "sel_blocks")
    m.lo_dev, m.hi_dev = _dev(lo, "lo"), _dev(hi, "hi")
    m.blk_base_dev, m.tok_base_dev = _dev(blk_base, "blk_base"), _dev(tok_base, "tok_base")
    m.block_first_dev = _dev(block_first, "block_first")
    m.block_last_dev = _dev(block_last, "block_last")
    return m


def qsa_forward(q, k, v, sel_blocks, lo, hi, blk_base, tok_base, block_first, block_last,
                scale=0.0625, block_size=4, *, max_blocks_per_query=0, workspace=None,
                stream=None):
    """Per-query bitmap sparse attention; returns (out bf16, out_fp32, lse [Hq, T])."""
    if not math.isfinite(scale):
        raise ValueError("scale must be finite")
    T, Hq, D = q.shape
    params = qsa_params(q, k, sel_blocks.shape[1], scale=scale, block_size=block_size,
                        max_blocks_per_query=max_blocks_per_query)
    meta = qsa_meta(sel_blocks, lo, hi, blk_base, tok_base, block_first, block_last)
    out = torch.empty_like(q)
    out_fp32 = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(paged_attn_workspace_size(params), q.device)
    paged_attn_plan(params, meta, workspace, stream)
    paged_attn_run(params, meta, q, k, v, out, out_fp32, lse, workspace, stream)
    return out, out_fp32, lse


def qsa_indexed_params(q, k, num_blocks, index_width, *, scale=0.0625, block_size=4,
                       max_blocks_per_query=0) -> AttnParams:
    p = qsa_params(q, k, num_blocks, scale=scale, block_size=block_size,
                   max_blocks_per_query=max_blocks_per_query)
    p.form = FORM_INDEXED
    p.index_width = int(index_width)
    return p


def qsa_indexed_meta(sel_indices, lo, hi, block_first, block_last) -> AttnMeta:
    m = AttnMeta()
    m.sel_indices_dev = _dev(sel_indices, "sel_indices")
    m.lo_dev, m.hi_dev = _dev(lo, "lo"), _dev(hi, "hi")
    m.block_first_dev = _dev(block_first, "block_first")
    m.block_last_dev = _dev(block_last, "block_last")
    return m


def qsa_indexed_forward(q, k, v, sel_indices, lo, hi, block_first, block_last, scale=0.0625,
                        block_size=4, *, max_blocks_per_query=0, workspace=None, stream=None):
    """Per-query block sparse attention from index rows sel_indices [T, K] int32 (each query
    token's selected global block ids; negative entries unused): the indexed entry point the
    [QSA] notes recommend when the indices already exist.  Returns (out bf16, out_fp32,
    lse [Hq, T])."""
    if not math.isfinite(scale):
        raise ValueError("scale must be finite")
    T, Hq, D = q.shape
    params = qsa_indexed_params(q, k, block_first.numel(), sel_indices.shape[1], scale=scale,
                                block_size=block_size, max_blocks_per_query=max_blocks_per_query)
    meta = qsa_indexed_meta(sel_indices, lo, hi, block_first, block_last)
    out = torch.empty_like(q)
    out_fp32 = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(paged_attn_workspace_size(params), q.device)
    paged_attn_plan(params, meta, workspace, stream)
    paged_attn_run(params, meta, q, k, v, out, out_fp32, lse, workspace, stream)
    return out, out_fp32, lse


def sage_params(q_int8, k_int8, q2k_block_index, block_sparse_num, *, block_sizes=None,
                softmax_scale=None, uniform_block_count=False) -> SageParams:
    B, H, Sq, D = q_int8.shape
    Sk = k_int8.shape[2]
    return SageParams(batch=B, num_heads=H, q_len=Sq, kv_len=Sk, head_dim=D,
                      capacity=q2k_block_index.shape[-1], block_sparse_num=int(block_sparse_num),
                      uniform_block_count=int(bool(uniform_block_count)),
                      block_sizes_rank=0 if block_sizes is None else block_sizes.dim(),
                      softmax_scale=float(softmax_scale or 0.0))


def paged_sage_workspace_size(params: SageParams) -> int:
    return int(lib().paged_sage_workspace_size(C.byref(params)))


def paged_sage_run(params: SageParams, q_int8, k_int8, v_fp8, q_scale, k_scale, v_scale,
                   q2k_block_index, q2k_block_nums, block_sizes, out, workspace,
                   stream=None) -> None:
    _check(lib().paged_sage_run(C.byref(params), _dev(q_int8, "q_int8"), _dev(k_int8, "k_int8"),
                                _dev(v_fp8, "v_fp8"), _dev(q_scale, "q_scale"),
                                _dev(k_scale, "k_scale"), _dev(v_scale, "v_scale"),
                                _dev(q2k_block_index, "q2k_block_index"),
                                _dev(q2k_block_nums, "q2k_block_nums"),
                                _dev(block_sizes, "block_sizes"), _dev(out, "out"),
                                _dev(workspace, "workspace"),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "paged_sage_run")


def bsa_sage_fwd(q_int8, k_int8, v_fp8, q_scale, k_scale, v_scale, q2k_block_index,
                 block_sparse_num, block_sizes=None, q2k_block_nums=None, softmax_scale=None, *,
                 out=None, uniform_block_count=False, contiguous_block_indices=False,
                 workspace=None, stream=None):
    """Prequantized block-sparse attention with the arguments of
    bsa_attn_sm120_blk64_sage_fwd: int8 Q/K [B, H, S, 128], FP8 E4M3 V [B, H, 128,
    ceil(Sk / 64) * 64] (uint8 or float8_e4m3fn storage), fp32 scales; returns out bf16
    [B, H, Sq, 128].  contiguous_block_indices is a hint that changes nothing here."""
    if softmax_scale is not None and not (softmax_scale > 0 and math.isfinite(softmax_scale)):
        raise ValueError("softmax_scale must be positive and finite")
    if contiguous_block_indices and not uniform_block_count:
        raise ValueError("contiguous_block_indices requires uniform_block_count")
    params = sage_params(q_int8, k_int8, q2k_block_index, block_sparse_num,
                         block_sizes=block_sizes, softmax_scale=softmax_scale,
                         uniform_block_count=uniform_block_count)
    if out is None:
        out = torch.empty(q_int8.shape, dtype=torch.bfloat16, device=q_int8.device)
    if workspace is None:
        workspace = _workspace(paged_sage_workspace_size(params), q_int8.device)
    v = v_fp8.view(torch.uint8) if v_fp8.dtype != torch.uint8 else v_fp8
    paged_sage_run(params, q_int8, k_int8, v, q_scale, k_scale, v_scale, q2k_block_index,
                   q2k_block_nums, block_sizes, out, workspace, stream)
    return out
