#!/usr/bin/env python
"""Benchmark of the paged-KV attention forward library on one GB300.

Headline (one JSON line): the paged decode workload (B=64, Hq=32, Hkv=8, D=128, lens
U[512, 8192], combined cache, page 16, split-KV), as KV GB/s over the live K/V bytes.  A step
is one call of paged_decode_run: device planner, split-KV partial kernel and merge.  The
other named workloads (block-sparse, packed prefill, bitmap) are measured in the same run and
reported under "per_config" as tensor TFLOPS over visible (selected, unmasked, valid) pairs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-extra] [--skip-cpu]

Under torchrun each rank runs the same workload on its own GPU (replicas: the path has no
exchange step), the timed region is bracketed by a barrier and synchronisation on both
sides, and the slowest rank's time is reported.  --impl reference times the float64 CPU
oracle on a bounded sample of the workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import paged_kv_block_gb300 as pkb  # noqa: E402
from paged_kv_block_gb300 import workloads as W  # noqa: E402

METRIC = "sparse/prefill attn TFLOPS & decode KV GB/s; % of tensor/HBM roofline, 1 GB300"
HEADLINE = "decode_b64"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------------------
# environment
# ----------------------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            self.path = f"/tmp/pkb_clocks_{os.getpid()}.csv"
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "decode_split_kernel": ["paged_kv_block_gb300/csrc/decode.cu",
                            "paged_kv_block_gb300/csrc/common.cuh"],
    "qsa_kernel": ["paged_kv_block_gb300/csrc/qsa.cu", "paged_kv_block_gb300/csrc/common.cuh"],
    "attn_tc_kernel": ["paged_kv_block_gb300/csrc/attn_tc.cu",
                       "paged_kv_block_gb300/csrc/common.cuh"],
    "attn256_kernel": ["paged_kv_block_gb300/csrc/attn256.cu",
                       "paged_kv_block_gb300/csrc/common.cuh"],
}


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel's
    source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------------------
# work accounting (independent of the checker package)
# ----------------------------------------------------------------------------------------

def decode_kv_bytes(p):
    Hkv = p["kv_cache"].shape[2]
    D = p["kv_cache"].shape[-1]
    return int(p["seq_lens"].to(torch.int64).sum()) * Hkv * D * 2 * 2


def bsr_pairs(p):
    q = p["q"]
    B, Sq, Hq, _ = q.shape
    Hkv = (p["k_cache"] if "k_cache" in p else p["kv_cache"][:, 0]).shape[1]
    G = Hq // Hkv
    qbs, kvbs = p["q_block_size"], p["kv_block_size"]
    nqb = -(-Sq // qbs)
    bptr = p["block_indptr"].numpy().astype(np.int64)
    bidx = p["block_indices"].numpy().astype(np.int64)
    lens = p["seq_lens_kv"].numpy().astype(np.int64)
    words = p["kv_valid_bits"].numpy().view(np.uint32) if p["kv_valid_bits"] is not None else None
    total = 0
    for b in range(B):
        L = int(lens[b])
        live = np.ones(L, bool)
        if words is not None:
            j = np.arange(L)
            live = ((words[b][j >> 5] >> (j & 31).astype(np.uint32)) & 1).astype(bool)
        for g in range(Hkv):
            for r in range(nqb):
                blocks = bidx[bptr[b, g, r]:bptr[b, g, r + 1]]
                keys = (blocks[:, None] * kvbs + np.arange(kvbs)[None, :]).ravel()
                keys = keys[keys < L]
                keys = np.sort(keys[live[keys]])
                rows = np.arange(r * qbs, min((r + 1) * qbs, Sq))
                if p["mask_type"] == "causal":
                    total += int(np.searchsorted(keys, L - Sq + rows, side="right").sum())
                else:
                    total += keys.size * rows.size
    return total * G


def prefill_pairs(p):
    qo = p["qo_indptr"].numpy().astype(np.int64)
    lens = p["seq_lens_kv"].numpy().astype(np.int64)
    Hq = p["q"].shape[1]
    w = p["window_left"]
    total = 0
    for b in range(lens.size):
        nq, L = int(qo[b + 1] - qo[b]), int(lens[b])
        if p["mask_type"] != "causal":
            total += nq * L
            continue
        pos = L - nq + np.arange(nq)
        hi = np.minimum(pos + 1, L)
        lo = np.maximum(pos - w, 0) if w >= 0 else np.zeros_like(pos)
        total += int(np.maximum(hi - lo, 0).sum())
    return total * Hq


def qsa_pairs(p):
    sel = p["sel_blocks"].numpy()
    t, g = np.nonzero(sel)
    lo, hi = p["lo"].numpy()[t].astype(np.int64), p["hi"].numpy()[t].astype(np.int64)
    first = p["block_first"].numpy()[g].astype(np.int64)
    last = p["block_last"].numpy()[g].astype(np.int64)
    return int(np.maximum(np.minimum(last, hi) - np.maximum(first, lo) + 1, 0).sum()) * \
        p["q"].shape[1]


def qsa_indexed_pairs(p):
    idx = p["sel_indices"].numpy()
    NB = p["block_first"].numel()
    t, c = np.nonzero((idx >= 0) & (idx < NB))
    g = idx[t, c].astype(np.int64)
    lo, hi = p["lo"].numpy()[t].astype(np.int64), p["hi"].numpy()[t].astype(np.int64)
    first = p["block_first"].numpy()[g].astype(np.int64)
    last = p["block_last"].numpy()[g].astype(np.int64)
    return int(np.maximum(np.minimum(last, hi) - np.maximum(first, lo) + 1, 0).sum()) * \
        p["q"].shape[1]


def sage_pairs(p):
    """Visible (query, head, key) triples of the prequantized form."""
    B, H, Sq, _ = p["q_int8"].shape
    Sk = p["k_int8"].shape[2]
    idx = p["q2k_block_index"].numpy()
    nums = p["q2k_block_nums"].numpy() if p["q2k_block_nums"] is not None else None
    bs = p["block_sizes"]
    total = 0
    for b in range(B):
        for h in range(H):
            for r in range(-(-Sq // 64)):
                n = int(nums[b, h, r]) if nums is not None else p["block_sparse_num"]
                rows = min(64, Sq - 64 * r)
                for c in idx[b, h, r, :n]:
                    c = int(c)
                    size = min(64, Sk - 64 * c)
                    if bs is not None:
                        size = min(size, int(bs.reshape(-1)[c] if bs.dim() == 1 else
                                              (bs[b, c] if bs.dim() == 2 else bs[b, h, c])))
                    total += rows * max(size, 0)
    return total


# Block-granular counts: the (row, head, key) triples of every selected block (or, for dense
# prefill, of every 128-key tile a work tile visits) taken whole, before the length, validity,
# causal and window masks cut it.  A secondary figure beside the visible-pair count: the
# tensor cores do at least this much work, and visible / block-granular is the share of it that
# counts toward the headline TFLOPS.

def bsr_block_pairs(p):
    q = p["q"]
    B, Sq, Hq, _ = q.shape
    Hkv = (p["k_cache"] if "k_cache" in p else p["kv_cache"][:, 0]).shape[1]
    qbs, kvbs = p["q_block_size"], p["kv_block_size"]
    nqb = -(-Sq // qbs)
    bptr = p["block_indptr"].numpy().astype(np.int64).reshape(B, Hkv, nqb + 1)
    rows = np.minimum(qbs, Sq - qbs * np.arange(nqb))
    nblk = bptr[:, :, 1:] - bptr[:, :, :-1]
    return int((nblk * rows[None, None, :]).sum()) * kvbs * (Hq // Hkv)


def prefill_tile_pairs(p):
    """Work tiles of 2 x (128 // G) tokens (one sub-tile of 128 // G for D = 256) against the
    128-key KV tiles that meet their causal / window span, 128 keys each."""
    qo = p["qo_indptr"].numpy().astype(np.int64)
    lens = p["seq_lens_kv"].numpy().astype(np.int64)
    Hq, D = p["q"].shape[1], p["q"].shape[2]
    G = Hq // p["k_cache"].shape[1]
    T = (128 // G) * (1 if D == 256 else 2)
    causal, w = p["mask_type"] == "causal", p["window_left"]
    total = 0
    for b in range(lens.size):
        nq, L = int(qo[b + 1] - qo[b]), int(lens[b])
        for tok0 in range(0, nq, T):
            ntok = min(T, nq - tok0)
            p0 = L - nq + tok0
            hi = min(L, p0 + ntok) if causal else L
            lo = max(0, p0 - w) if (causal and w >= 0) else 0
            if hi > lo:
                total += (-(-hi // 128) - lo // 128) * 128 * ntok
    return total * Hq


def _qsa_block_pairs(t, g, p):
    lo, hi = p["lo"].numpy()[t].astype(np.int64), p["hi"].numpy()[t].astype(np.int64)
    first = p["block_first"].numpy()[g].astype(np.int64)
    last = p["block_last"].numpy()[g].astype(np.int64)
    meets = np.maximum(first, lo) <= np.minimum(last, hi)
    return int((last - first + 1)[meets].sum()) * p["q"].shape[1]


def qsa_block_pairs(p):
    t, g = np.nonzero(p["sel_blocks"].numpy())
    return _qsa_block_pairs(t, g, p)


def qsa_indexed_block_pairs(p):
    idx = p["sel_indices"].numpy()
    t, c = np.nonzero((idx >= 0) & (idx < p["block_first"].numel()))
    return _qsa_block_pairs(t, idx[t, c].astype(np.int64), p)


def sage_block_pairs(p):
    B, H, Sq, _ = p["q_int8"].shape
    nqb = -(-Sq // 64)
    rows = np.minimum(64, Sq - 64 * np.arange(nqb))
    if p["q2k_block_nums"] is not None:
        n = p["q2k_block_nums"].numpy().astype(np.int64).reshape(B, H, nqb)
    else:
        n = np.full((B, H, nqb), p["block_sparse_num"], np.int64)
    return int((n * rows[None, None, :]).sum()) * 64


BLOCK_COUNTERS = {"bsr": bsr_block_pairs, "prefill": prefill_tile_pairs,
                  "qsa": qsa_block_pairs, "qsa_indexed": qsa_indexed_block_pairs,
                  "sage": sage_block_pairs}


# ----------------------------------------------------------------------------------------
# one workload on the GPU
# ----------------------------------------------------------------------------------------

def block_granular(p, kernel_ms):
    """The labelled secondary figure: block-granular triples and the kernel's rate over them."""
    nb = BLOCK_COUNTERS[p["form"]](p)
    D = (p["q"] if "q" in p else p["q_int8"]).shape[-1]
    return {"pairs": nb, "tflops_kernel": 4 * D * nb / (kernel_ms * 1e-3) / 1e12,
            "what": "selected blocks (dense prefill: the 128-key tiles each work tile visits) "
                    "taken whole, before length, validity, causal and window masks"}


def main_kernel(p):
    """Name of the kernel that does the attention arithmetic of workload p."""
    if p["form"] == "decode":
        return "decode_split_kernel"
    if p["form"] in ("qsa", "qsa_indexed"):
        return "qsa_kernel"
    if p["form"] == "prefill" and p["q"].shape[-1] == 256:
        return "attn256_kernel"
    return "attn_tc_kernel"


def make_workload(name):
    if name == "decode_b64":
        return W.decode_b64()
    if name == "decode_b64_sq4":
        return W.decode_b64_sq4()
    if name == "tiny_bsr":
        return W.tiny_bsr()
    if name == "prefill_b16":
        return W.prefill_b16(window_left=-1)
    if name == "prefill_b16_w1023":
        return W.prefill_b16(window_left=1023)
    if name == "prefill_b16_d256":
        return W.prefill_b16_d256()
    if name == "long_bsr":
        return W.long_bsr()
    if name == "qsa_t32k":
        return W.qsa_t32k()
    if name == "qsa_t32k_indexed":
        return W.qsa_t32k_indexed()
    if name == "sage_b2h16":
        return W.sage_b2h16()
    raise ValueError(name)


def describe(name, p):
    if p["form"] == "sage":
        B, H, Sq, D = p["q_int8"].shape
        return {"workload": name, "batch": B, "num_heads": H, "q_len": Sq,
                "kv_len": int(p["k_int8"].shape[2]), "head_dim": D, "blocks_per_row":
                p["block_sparse_num"], "inputs": "int8 Q/K, FP8 E4M3 V, fp32 scales"}
    if p["form"] == "decode":
        d = {"workload": name, "batch": int(p["q"].shape[0]), "num_qo_heads": int(p["q"].shape[-2]),
             "num_kv_heads": int(p["kv_cache"].shape[2]), "head_dim": int(p["q"].shape[-1]),
             "page_size": int(p["page_size"]), "seq_lens": "U[512,8192]",
             "total_kv_tokens": int(p["seq_lens"].sum()), "cache": "combined [P,2,Hkv,ps,D]",
             "mask": p["mask_type"], "split_kv": True}
        if p["seq_len_q"] > 1:
            d["seq_len_q"] = int(p["seq_len_q"])
        return d
    if p["form"] == "bsr":
        return {"workload": name, "batch": int(p["q"].shape[0]), "q_len": int(p["q"].shape[1]),
                "num_qo_heads": int(p["q"].shape[2]), "page_size": int(p["page_size"]),
                "q_block_size": p["q_block_size"], "kv_block_size": p["kv_block_size"],
                "selected_blocks": int(p["block_indices"].numel()), "mask": p["mask_type"],
                "kv_valid_bits": p["kv_valid_bits"] is not None}
    if p["form"] == "prefill":
        return {"workload": name, "batch": int(p["seq_lens_kv"].numel()),
                "total_q": int(p["q"].shape[0]), "num_qo_heads": int(p["q"].shape[1]),
                "head_dim": int(p["q"].shape[2]),
                "page_size": int(p["page_size"]), "mask": p["mask_type"],
                "window_left": p["window_left"]}
    d = {"workload": name, "tokens": int(p["q"].shape[0]), "num_qo_heads": int(p["q"].shape[1]),
         "head_dim": int(p["q"].shape[2]), "num_blocks": int(p["block_first"].numel())}
    if p["form"] == "qsa_indexed":
        d["index_width"] = int(p["sel_indices"].shape[1])
    return d


class Runner:
    """Owns the device copies of one workload and runs one step through the C ABI."""

    def __init__(self, p, dev):
        self.p = p
        self.dev = dev
        self.d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
        d = self.d
        self.form = p["form"]
        if self.form == "decode":
            self.params = pkb.decode_params(d["q"], d["kv_cache"], p["max_seq_len"],
                                            bmm1_scale=p["sm_scale"], bmm2_scale=p["bmm2_scale"],
                                            mask_type=p["mask_type"],
                                            window_left=p["window_left"],
                                            seq_len_q=p["seq_len_q"], qo_indptr=d["qo_indptr"],
                                            max_seq_len_q=p["max_seq_len_q"])
            self.ws = torch.empty(pkb.paged_decode_workspace_size(self.params), dtype=torch.uint8,
                                  device=dev)
            self.out = torch.empty_like(d["q"])
            self.lse = torch.empty(d["q"].shape[:-1], dtype=torch.float32, device=dev)
        elif self.form == "bsr":
            cache = d["kv_cache"] if "kv_cache" in d else (d["k_cache"], d["v_cache"])
            self.k, self.v = (cache, None) if not isinstance(cache, tuple) else cache
            self.params = pkb.bsr_params(d["q"], cache, p["q_block_size"], p["kv_block_size"],
                                         p["max_seq_len_kv"],
                                         has_valid_bits=p["kv_valid_bits"] is not None,
                                         mask_type=p["mask_type"], sm_scale=p["sm_scale"])
            self.meta = pkb.bsr_meta(d["kv_indptr"], d["kv_indices"], d["block_indptr"],
                                     d["block_indices"], d["seq_lens_kv"], d["kv_valid_bits"])
            self.ws = torch.empty(pkb.paged_attn_workspace_size(self.params), dtype=torch.uint8,
                                  device=dev)
            self.out = torch.empty_like(d["q"])
            self.lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
        elif self.form == "prefill":
            self.params = pkb.prefill_params(d["q"], d["k_cache"], d["block_tables"],
                                             d["seq_lens_kv"].numel(), mask_type=p["mask_type"],
                                             window_left=p["window_left"],
                                             sm_scale=p["sm_scale"],
                                             output_scale=p["output_scale"])
            self.ws = torch.empty(pkb.paged_prefill_workspace_size(self.params),
                                  dtype=torch.uint8, device=dev)
            self.out = torch.empty_like(d["q"])
            self.lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev)
        elif self.form == "sage":
            self.params = pkb.sage_params(d["q_int8"], d["k_int8"], d["q2k_block_index"],
                                          p["block_sparse_num"], block_sizes=d["block_sizes"],
                                          softmax_scale=p["softmax_scale"],
                                          uniform_block_count=p["q2k_block_nums"] is None)
            self.ws = torch.zeros(pkb.paged_sage_workspace_size(self.params), dtype=torch.uint8,
                                  device=dev)
            self.out = torch.empty(d["q_int8"].shape, dtype=torch.bfloat16, device=dev)
        else:
            if self.form == "qsa_indexed":
                self.params = pkb.qsa_indexed_params(d["q"], d["k"], d["block_first"].numel(),
                                                     d["sel_indices"].shape[1], scale=p["scale"])
                self.meta = pkb.qsa_indexed_meta(d["sel_indices"], d["lo"], d["hi"],
                                                 d["block_first"], d["block_last"])
            else:
                self.params = pkb.qsa_params(d["q"], d["k"], d["sel_blocks"].shape[1],
                                             scale=p["scale"])
                self.meta = pkb.qsa_meta(d["sel_blocks"], d["lo"], d["hi"], d["blk_base"],
                                         d["tok_base"], d["block_first"], d["block_last"])
            self.ws = torch.empty(pkb.paged_attn_workspace_size(self.params), dtype=torch.uint8,
                                  device=dev)
            self.out = torch.empty_like(d["q"])
            self.out32 = torch.empty(d["q"].shape, dtype=torch.float32, device=dev)
            self.lse = torch.empty(d["q"].shape[1], d["q"].shape[0], dtype=torch.float32,
                                   device=dev)

    def inputs(self):
        """The step's input tensors (device), in a fixed order."""
        names = {"decode": ["q", "kv_cache", "kv_indptr", "kv_indices", "seq_lens",
                            "qo_indptr"],
                 "bsr": ["q", "k_cache", "v_cache", "kv_cache", "kv_indptr", "kv_indices",
                         "block_indptr", "block_indices", "seq_lens_kv", "kv_valid_bits"],
                 "prefill": ["q", "k_cache", "v_cache", "qo_indptr", "block_tables",
                             "seq_lens_kv"],
                 "qsa": ["q", "k", "v", "sel_blocks", "lo", "hi", "blk_base", "tok_base",
                         "block_first", "block_last"],
                 "qsa_indexed": ["q", "k", "v", "sel_indices", "lo", "hi", "block_first",
                                 "block_last"],
                 "sage": ["q_int8", "k_int8", "v_fp8", "q_scale", "k_scale", "v_scale",
                          "q2k_block_index", "q2k_block_nums", "block_sizes"]}[self.form]
        return [(n, self.d[n]) for n in names if isinstance(self.d.get(n), torch.Tensor)]

    def step(self):
        d = self.d
        if self.form == "decode":
            pkb.paged_decode_run(self.params, d["q"], d["kv_cache"], None, d["kv_indptr"],
                                 d["kv_indices"], d["seq_lens"], self.out, self.lse, self.ws,
                                 qo_indptr=d["qo_indptr"])
        elif self.form == "bsr":
            pkb.paged_attn_plan(self.params, self.meta, self.ws)
            pkb.paged_attn_run(self.params, self.meta, d["q"], self.k, self.v, self.out, None,
                               self.lse, self.ws)
        elif self.form == "sage":
            pkb.paged_sage_run(self.params, d["q_int8"], d["k_int8"], d["v_fp8"], d["q_scale"],
                               d["k_scale"], d["v_scale"], d["q2k_block_index"],
                               d["q2k_block_nums"], d["block_sizes"], self.out, self.ws)
        elif self.form == "prefill":
            pkb.paged_prefill_run(self.params, d["q"], d["k_cache"], d["v_cache"],
                                  d["qo_indptr"], d["block_tables"], d["seq_lens_kv"], self.out,
                                  self.lse, self.ws)
        else:
            pkb.paged_attn_plan(self.params, self.meta, self.ws)
            pkb.paged_attn_run(self.params, self.meta, d["q"], d["k"], d["v"], self.out,
                               self.out32, self.lse, self.ws)

    def status(self):
        return pkb.paged_attn_workspace_status(self.ws)


def barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def max_over_ranks(x, dist_on, device):
    """The largest x over all ranks: the job's time is its slowest rank's."""
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if dist_on:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms_step, scale):
    """Whole-job throughput: the units every rank processed in a step (each rank runs the same
    workload) over the slowest rank's step time."""
    return units_per_rank * world / (ms_step * 1e-3) / scale


def time_steps(r, steps, warmup, dist_on):
    """(region ms, main-kernel ms per launch, kernel launches of this library in the region).

    The region is timed with the kernel timer off (its events would sit between the planner
    and the main kernel); the main kernel's own time comes from a second pass of `steps`
    steps with the timer on."""
    for _ in range(warmup):
        r.step()
    torch.cuda.synchronize()
    barrier(dist_on)
    torch.cuda.synchronize()
    n0 = pkb.paged_attn_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        r.step()
    e1.record()
    torch.cuda.synchronize()
    barrier(dist_on)
    torch.cuda.synchronize()
    n1 = pkb.paged_attn_launch_count()
    pkb.paged_attn_kernel_timer(True)
    for _ in range(steps):
        r.step()
    torch.cuda.synchronize()
    pkb.paged_attn_kernel_timer(False)
    kms, kn = pkb.paged_attn_kernel_timer_read()
    return e0.elapsed_time(e1), kms / max(kn, 1), n1 - n0


def time_e2e(r, steps):
    """Each step copies its inputs from pinned host memory, runs, and reads the output back."""
    host = [(n, t.cpu().pin_memory()) for n, t in r.inputs()]
    out_host = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for _, t in host)
    d2h = out_host.numel() * out_host.element_size()
    for _ in range(2):
        for n, t in host:
            r.d[n].copy_(t, non_blocking=True)
        r.step()
        out_host.copy_(r.out, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        for n, t in host:
            r.d[n].copy_(t, non_blocking=True)
        r.step()
        out_host.copy_(r.out, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ----------------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ----------------------------------------------------------------------------------------

def decode_subbatch(p, reqs):
    """The requests `reqs` of a decode workload with their pages copied to a compact pool."""
    indptr = p["kv_indptr"].numpy()
    idx = p["kv_indices"].numpy()
    pages, new_ptr = [], [0]
    for b in reqs:
        pg = idx[indptr[b]:indptr[b + 1]]
        pages.append(pg)
        new_ptr.append(new_ptr[-1] + pg.size)
    allp = np.concatenate(pages)
    return dict(p, q=p["q"][list(reqs)], kv_cache=p["kv_cache"][torch.from_numpy(allp).long()],
                kv_indptr=torch.tensor(new_ptr, dtype=torch.int32),
                kv_indices=torch.arange(allp.size, dtype=torch.int32),
                seq_lens=p["seq_lens"][list(reqs)])


def oracle_decode_seconds(p):
    from oracle import attention as A
    t0 = time.perf_counter()
    A.batch_decode(p["q"], p["kv_indptr"], p["kv_indices"], p["seq_lens"],
                   kv_cache=p["kv_cache"], bmm1_scale=p["sm_scale"], bmm2_scale=p["bmm2_scale"],
                   mask_type=p["mask_type"], window_left=p["window_left"],
                   seq_len_q=p.get("seq_len_q", 1))
    return time.perf_counter() - t0


def cpu_baseline_decode(p, budget_s=12.0):
    """Oracle over consecutive 8-request sub-batches, looping over the batch, until about
    budget_s seconds."""
    B = p["q"].shape[0]
    done_bytes, secs, subs, passes = 0, 0.0, 0, 0
    while secs < budget_s:
        for s in range(0, B, 8):
            sub = decode_subbatch(p, range(s, min(B, s + 8)))
            secs += oracle_decode_seconds(sub)
            done_bytes += decode_kv_bytes(sub)
            subs += 1
            if secs >= budget_s:
                break
        passes += 1
    return {"value": done_bytes / secs / 1e9, "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"float64 oracle on {subs} 8-request sub-batches of the {B}-request batch "
                      f"({passes} pass(es); {done_bytes / 1e9:.3f} GB of live K/V, {secs:.1f} s; "
                      "BLAS threads = all host cores, page gathers single-threaded)"}


# ----------------------------------------------------------------------------------------
# Oracle samples of the other workloads: seeded slices that are problems of their own, so
# that their work is counted exactly by the same counters as the full workload.
# ----------------------------------------------------------------------------------------

def bsr_qblock_slice(p, r0, r1):
    """Query blocks [r0, r1) of a block-sparse problem as a problem of its own.  The sampled
    queries keep their positions: the KV length of each request is cut to the key after the
    last sampled query's position (later keys are causally invisible to them), so the
    bottom-right alignment p = L - Sq + i still places query i of the slice at its original
    position."""
    qbs = p["q_block_size"]
    B, Sq = p["q"].shape[:2]
    bptr = p["block_indptr"].numpy().astype(np.int64)
    bidx = p["block_indices"].numpy().astype(np.int64)
    Hkv = bptr.shape[1]
    n = r1 - r0
    i0, i1 = r0 * qbs, min(r1 * qbs, Sq)
    lens = p["seq_lens_kv"].numpy().astype(np.int64)
    new_lens = np.maximum(lens - Sq + i1, 0) if p["mask_type"] == "causal" else lens
    ptr = np.zeros((B, Hkv, n + 1), dtype=np.int64)
    rows, off = [], 0
    for b in range(B):
        for g in range(Hkv):
            for k, r in enumerate(range(r0, r1)):
                ptr[b, g, k] = off
                rows.append(bidx[bptr[b, g, r]:bptr[b, g, r + 1]])
                off += rows[-1].size
            ptr[b, g, n] = off
    return dict(p, q=p["q"][:, i0:i1].contiguous(),
                block_indptr=torch.from_numpy(ptr.astype(np.int32)),
                block_indices=torch.from_numpy(np.concatenate(rows).astype(np.int32)),
                seq_lens_kv=torch.from_numpy(new_lens.astype(np.int32)),
                max_seq_len_kv=int(new_lens.max()))


def prefill_subbatch(p, reqs):
    """Requests `reqs` of a packed prefill problem with their pages copied to compact pools."""
    qo = p["qo_indptr"].numpy().astype(np.int64)
    tables = p["block_tables"].numpy()[list(reqs)]
    pages, inv = np.unique(tables, return_inverse=True)
    rows = np.concatenate([np.arange(qo[b], qo[b + 1]) for b in reqs])
    nq = [int(qo[b + 1] - qo[b]) for b in reqs]
    pg = torch.from_numpy(pages).long()
    return dict(p, q=p["q"][torch.from_numpy(rows)], k_cache=p["k_cache"][pg],
                v_cache=p["v_cache"][pg],
                qo_indptr=torch.tensor(np.concatenate([[0], np.cumsum(nq)]), dtype=torch.int32),
                block_tables=torch.from_numpy(inv.reshape(tables.shape).astype(np.int32)),
                seq_lens_kv=p["seq_lens_kv"][list(reqs)], num_pages=int(pages.size))


def qsa_last_sequence(p):
    """The last packed sequence of a bitmap (or indexed) problem, re-based to start at token 0
    and block 0 (sequences never share blocks or keys)."""
    tb = p["tok_base"].numpy() if "tok_base" in p else None
    lo = p["lo"].numpy().astype(np.int64)
    t0 = int(lo[-1])
    bs = p["block_size"]
    b0 = t0 // bs
    sub = dict(p, q=p["q"][t0:], k=p["k"][t0:], v=p["v"][t0:],
               lo=torch.from_numpy((lo[t0:] - t0).astype(np.int32)),
               hi=torch.from_numpy((p["hi"].numpy()[t0:].astype(np.int64) - t0).astype(np.int32)),
               block_first=p["block_first"][b0:] - t0, block_last=p["block_last"][b0:] - t0)
    if tb is not None:
        sub["tok_base"] = torch.from_numpy((tb[t0:] - t0).astype(np.int32))
        sub["blk_base"] = torch.from_numpy((p["blk_base"].numpy()[t0:] - b0).astype(np.int32))
    if "sel_blocks" in p:
        sub["sel_blocks"] = p["sel_blocks"][t0:, b0:].contiguous()
    else:
        idx = p["sel_indices"].numpy()[t0:].astype(np.int64)
        sub["sel_indices"] = torch.from_numpy(np.where(idx >= 0, idx - b0, idx).astype(np.int32))
    return sub


def qsa_rows(p, rows):
    """The query rows `rows` of a bitmap or indexed problem, for counting their pairs."""
    r = torch.as_tensor(rows, dtype=torch.long)
    sub = dict(p, q=p["q"][r], lo=p["lo"][r], hi=p["hi"][r])
    key = "sel_blocks" if "sel_blocks" in p else "sel_indices"
    sub[key] = p[key][r]
    return sub


def oracle_sample_rate(name, p):
    """Time the float64 oracle (as it stands) on a seeded slice of workload `p`; returns the
    cpu_baseline record in the workload's unit."""
    from oracle import attention as A
    rng = np.random.default_rng(77)
    cores = os.cpu_count()
    form = p["form"]
    if form == "decode":
        B = p["q"].shape[0]
        reqs = sorted(rng.choice(B, size=8, replace=False).tolist())
        sub = decode_subbatch(p, reqs)
        secs = oracle_decode_seconds(sub)
        nb = decode_kv_bytes(sub)
        return {"value": nb / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "seconds": secs, "sample": f"requests {reqs} of {B} ({nb / 1e9:.3f} GB K/V)"}
    t0 = time.perf_counter()
    if form == "bsr":
        Sq, qbs = p["q"].shape[1], p["q_block_size"]
        nqb = -(-Sq // qbs)
        if nqb <= 4:
            sub, what = p, "the whole workload"
        else:
            r1 = int(rng.integers(nqb // 2, nqb + 1))
            sub, what = bsr_qblock_slice(p, r1 - 4, r1), f"query blocks {r1 - 4}..{r1 - 1} of {nqb}"
        t0 = time.perf_counter()
        A.block_sparse_attention(
            sub["q"], sub["kv_indptr"], sub["kv_indices"], sub["block_indptr"],
            sub["block_indices"], sub["q_block_size"], sub["kv_block_size"], sub["seq_lens_kv"],
            kv_cache=sub.get("kv_cache"), k_cache=sub.get("k_cache"), v_cache=sub.get("v_cache"),
            kv_valid_bits=sub.get("kv_valid_bits"), mask_type=sub["mask_type"],
            sm_scale=sub["sm_scale"])
        pairs, D = bsr_pairs(sub), sub["q"].shape[-1]
    elif form == "prefill":
        B = p["seq_lens_kv"].numel()
        reqs = sorted(rng.choice(B, size=2, replace=False).tolist())
        sub, what = prefill_subbatch(p, reqs), f"requests {reqs} of {B}"
        t0 = time.perf_counter()
        A.batch_prefill(sub["q"], sub["k_cache"], sub["v_cache"], sub["qo_indptr"],
                        sub["block_tables"], sub["seq_lens_kv"], mask_type=sub["mask_type"],
                        window_left=sub["window_left"], sm_scale=sub["sm_scale"],
                        output_scale=sub["output_scale"])
        pairs, D = prefill_pairs(sub), sub["q"].shape[-1]
    elif form in ("qsa", "qsa_indexed"):
        seq = qsa_last_sequence(p)
        T = seq["q"].shape[0]
        rows = sorted(rng.choice(T, size=min(T, 384), replace=False).tolist())
        what = f"{len(rows)} random tokens of the last packed sequence ({T} tokens)"
        t0 = time.perf_counter()
        if form == "qsa":
            A.qsa_forward(seq["q"], seq["k"], seq["v"], seq["sel_blocks"], seq["lo"], seq["hi"],
                          seq["blk_base"], seq["tok_base"], seq["block_first"],
                          seq["block_last"], seq["scale"], seq["block_size"], rows=rows)
            pairs = qsa_pairs(qsa_rows(seq, rows))
        else:
            A.qsa_indexed_forward(seq["q"], seq["k"], seq["v"], seq["sel_indices"], seq["lo"],
                                  seq["hi"], seq["block_first"], seq["block_last"],
                                  seq["scale"], seq["block_size"], rows=rows)
            pairs = qsa_indexed_pairs(qsa_rows(seq, rows))
        D = seq["q"].shape[-1]
    elif form == "sage":
        B, H = p["q_int8"].shape[:2]
        b, h = int(rng.integers(0, B)), int(rng.integers(0, H))
        sl = lambda t: None if t is None else t[b:b + 1, h:h + 1]  # noqa: E731
        sub = dict(p, q_int8=sl(p["q_int8"]), k_int8=sl(p["k_int8"]), v_fp8=sl(p["v_fp8"]),
                   q_scale=sl(p["q_scale"]), k_scale=sl(p["k_scale"]), v_scale=sl(p["v_scale"]),
                   q2k_block_index=sl(p["q2k_block_index"]),
                   q2k_block_nums=sl(p["q2k_block_nums"]))
        if p["block_sizes"] is not None and p["block_sizes"].dim() > 1:
            sub["block_sizes"] = (p["block_sizes"][b:b + 1] if p["block_sizes"].dim() == 2
                                  else sl(p["block_sizes"]))
        what = f"(b, h) = ({b}, {h}) of ({B}, {H})"
        t0 = time.perf_counter()
        A.sage_block_sparse_attention(sub["q_int8"], sub["k_int8"], sub["v_fp8"], sub["q_scale"],
                                      sub["k_scale"], sub["v_scale"], sub["q2k_block_index"],
                                      sub["block_sparse_num"], sub["block_sizes"],
                                      sub["q2k_block_nums"], sub["softmax_scale"])
        pairs, D = sage_pairs(sub), sub["q_int8"].shape[-1]
    else:
        raise ValueError(form)
    secs = time.perf_counter() - t0
    flops = 4 * D * pairs
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": secs,
            "sample": f"{what}: {pairs} visible pairs, {flops / 1e9:.2f} GFLOP in {secs:.2f} s "
                      "(BLAS threads = all host cores)"}


def qsa_gathered_bytes(p):
    """K/V bytes the bitmap (or indexed) form gathers: every query token reads the K and V
    rows of each selected block that meets [lo, hi], for all KV heads."""
    first = p["block_first"].numpy().astype(np.int64)
    last = p["block_last"].numpy().astype(np.int64)
    lo, hi = p["lo"].numpy().astype(np.int64), p["hi"].numpy().astype(np.int64)
    if "sel_blocks" in p:
        t, g = np.nonzero(p["sel_blocks"].numpy())
    else:
        idx = p["sel_indices"].numpy()
        t, c = np.nonzero((idx >= 0) & (idx < first.size))
        g = idx[t, c].astype(np.int64)
    live = (np.minimum(last[g], hi[t]) >= np.maximum(first[g], lo[t]))
    Hkv, D = p["k"].shape[1], p["k"].shape[2]
    return int(live.sum()) * int(p["block_size"]) * Hkv * D * 2 * 2


def l2_read_gbs(dev, mib=24, reps=64):
    """The L2 read rate of this GPU: the library's probe over an L2-resident buffer, best of
    5 launches, timed with events on the current stream."""
    buf = torch.zeros(mib << 20, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        pkb.paged_attn_l2_read_probe(buf, reps, sink)
    best = float("inf")
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkb.paged_attn_l2_read_probe(buf, reps, sink)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return buf.numel() * reps / (best * 1e-3) / 1e9


# ----------------------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------------------

def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    p = make_workload(args.workload)
    if p["form"] != "decode":
        print(json.dumps({"impl": "reference", "unavailable":
                          "the reference arm is defined on the decode workload"}))
        return 0
    sub = decode_subbatch(p, range(0, 8))
    nbytes = decode_kv_bytes(sub)
    for _ in range(args.warmup):
        oracle_decode_seconds(sub)
    secs = [oracle_decode_seconds(sub) for _ in range(args.steps)]
    tot = sum(secs)
    v = nbytes * args.steps / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": describe(args.workload, p),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": "float64 oracle on requests 0..7 of the 64-request "
                                       f"decode batch per step ({nbytes / 1e9:.3f} GB K/V)"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-extra", action="store_true", help="skip the per_config workloads")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    dist_on = world > 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if dist_on:
        torch.distributed.init_process_group("nccl", device_id=dev)
    pk, pk_src = peaks()

    p = make_workload(args.workload)
    r = Runner(p, dev)
    sampler = ClockSampler(local)
    sampler.start()
    region_ms, kernel_ms, launches = time_steps(r, args.steps, args.warmup, dist_on)
    clocks = sampler.stop()
    rc, raw = r.status()
    if rc != pkb.OK:
        raise RuntimeError(f"device status {raw:#x}")
    region_ms = max_over_ranks(region_ms, dist_on, dev)
    ms_step = region_ms / args.steps

    if p["form"] == "decode":
        units = decode_kv_bytes(p)
        unit, scale = "GB/s", 1e9
        kernel, bound, peak = "decode_split_kernel", "hbm", pk["hbm_gbs"]
    else:
        nbytes = None
        units = {"bsr": bsr_pairs, "prefill": prefill_pairs, "qsa": qsa_pairs,
                 "qsa_indexed": qsa_indexed_pairs, "sage": sage_pairs}[p["form"]](p)
        units *= 4 * (p["q"] if "q" in p else p["q_int8"]).shape[-1]
        unit, scale = "TFLOP/s", 1e12
        kernel = main_kernel(p)
        bound, peak = "tensor", pk["bf16_tflops"]
    value = job_rate(units, world, ms_step, scale)
    achieved = units / (kernel_ms * 1e-3) / scale
    traffic = recorded_traffic(kernel, args.workload)
    e2e_ms, h2d, d2h = time_e2e(r, max(3, min(args.steps, 10)))
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16; see workloads.py)",
            "config": dict(describe(args.workload, p),
                           l2="inputs larger than L2" if p["form"] == "decode" else
                           "L2 not flushed between steps",
                           parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                         "unit": unit, "frac": achieved / peak, "traffic": traffic,
                         "kernel": kernel, "kernel_ms": kernel_ms,
                         "peak_source": f"{pk_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})"},
            "e2e": {"value": job_rate(units, world, e2e_ms, scale), "unit": unit,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            "gpu_launches": launches,
            "clocks": clocks}
    if p["form"] != "decode":
        line["block_granular"] = block_granular(p, kernel_ms)
    del r
    torch.cuda.empty_cache()

    # The oracle baselines run after every GPU timing: their BLAS threads would otherwise
    # compete with the launching thread of the latency-bound workloads.
    cpu_todo = []
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu_todo.append(None)                      # the headline workload
    l2_gbs = None
    if p["form"] in ("qsa", "qsa_indexed"):
        l2_gbs = l2_read_gbs(dev)
        gb = qsa_gathered_bytes(p)
        line["roofline_l2"] = {"bound": "l2", "achieved": gb / (kernel_ms * 1e-3) / 1e9,
                               "peak": l2_gbs, "unit": "GB/s",
                               "frac": gb / (kernel_ms * 1e-3) / 1e9 / l2_gbs,
                               "gathered_bytes": gb,
                               "peak_source": "measured in this run (paged_attn_l2_read_probe "
                                              "over a 24 MiB L2-resident buffer)"}
    if not args.no_extra and rank == 0:
        extra = {}
        for name in ("decode_b64_sq4", "tiny_bsr", "prefill_b16", "prefill_b16_w1023",
                     "prefill_b16_d256", "long_bsr", "qsa_t32k", "qsa_t32k_indexed",
                     "sage_b2h16"):
            if name == args.workload:
                continue
            try:
                q = make_workload(name)
                rr = Runner(q, dev)
                reg, kms, _ = time_steps(rr, max(3, min(args.steps, 20)), 3, False)
                rc, raw = rr.status()
                if rc != pkb.OK:
                    raise RuntimeError(f"device status {raw:#x}")
                steps = max(3, min(args.steps, 20))
                if q["form"] == "decode":
                    nb = decode_kv_bytes(q)
                    extra[name] = {"gbs_step": nb / (reg / steps * 1e-3) / 1e9,
                                   "gbs_kernel": nb / (kms * 1e-3) / 1e9,
                                   "frac_hbm_peak": nb / (kms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                   "ms_step": reg / steps, "ms_kernel": kms, "kv_bytes": nb,
                                   "kernel": main_kernel(q),
                                   "traffic": recorded_traffic(main_kernel(q), name)}
                    del rr
                    torch.cuda.empty_cache()
                    if not args.skip_cpu:
                        cpu_todo.append(name)
                    continue
                n = {"bsr": bsr_pairs, "prefill": prefill_pairs, "qsa": qsa_pairs,
                     "qsa_indexed": qsa_indexed_pairs, "sage": sage_pairs}[q["form"]](q)
                flops = 4 * (q["q"] if "q" in q else q["q_int8"]).shape[-1] * n
                tk = flops / (kms * 1e-3) / 1e12
                extra[name] = {"tflops_step": flops / (reg / steps * 1e-3) / 1e12,
                               "tflops_kernel": tk,
                               "frac_bf16_peak": tk / pk["bf16_tflops"],
                               "frac_bf16_sustained": tk / pk.get("bf16_tflops_sustained",
                                                                  pk["bf16_tflops"]),
                               "ms_step": reg / steps, "ms_kernel": kms,
                               "visible_pairs": n, "flops": flops,
                               "kernel": main_kernel(q),
                               "block_granular": block_granular(q, kms),
                               "traffic": recorded_traffic(main_kernel(q), name)}
                if q["form"] in ("qsa", "qsa_indexed"):
                    if l2_gbs is None:
                        l2_gbs = l2_read_gbs(dev)
                    gb = qsa_gathered_bytes(q)
                    extra[name]["l2_gather"] = {
                        "bound": "l2", "achieved": gb / (kms * 1e-3) / 1e9, "peak": l2_gbs,
                        "unit": "GB/s", "frac": gb / (kms * 1e-3) / 1e9 / l2_gbs,
                        "gathered_bytes": gb,
                        "peak_source": "measured in this run (paged_attn_l2_read_probe over "
                                       "a 24 MiB L2-resident buffer)"}
                del rr
                torch.cuda.empty_cache()
            except pkb.PagedAttnError as e:
                extra[name] = {"unavailable": str(e)}
                continue
            if not args.skip_cpu:
                cpu_todo.append(name)
        line["per_config"] = extra
    for name in cpu_todo:
        if name is None:
            line["cpu_baseline"] = (cpu_baseline_decode(p) if p["form"] == "decode" else
                                    oracle_sample_rate(args.workload, p))
        else:
            line["per_config"][name]["cpu_baseline"] = oracle_sample_rate(name,
                                                                         make_workload(name))
    if rank == 0:
        print(json.dumps(line))
    if dist_on:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
