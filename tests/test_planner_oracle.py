"""Pins of the planner oracle (CPU): brute-force coverage checks and invariants."""
import numpy as np
import torch

from oracle import planner as PL
from paged_kv_block_gb300 import workloads as W
from tests import bruteforce as BF


def _check_order(recs, natural_key):
    cost = recs[:, 5] - recs[:, 4]
    assert np.all(np.diff(cost) <= 0)
    for c in np.unique(cost):
        sub = recs[cost == c]
        keys = [natural_key(r) for r in sub]
        assert keys == sorted(keys)


def test_bsr_tiles_cover_every_row_once():
    B, Sq, Hq, Hkv, qbs = 2, 50, 8, 2, 12
    p = W.make_bsr_problem(1, B=B, Sq=Sq, Hq=Hq, Hkv=Hkv, D=8, seq_lens=[70, 55], page_size=4,
                           qbs=qbs, kvbs=4, policy="random", p=0.4)
    tt = 5
    recs = PL.plan_bsr_tiles(B, Sq, Hq, Hkv, qbs, p["block_indptr"], tt)
    assert len(recs) == PL.bsr_tile_capacity(B, Sq, Hkv, qbs, tt)
    seen = np.zeros((B, Hkv, Sq), int)
    bptr = p["block_indptr"].numpy()
    for b, g, tok0, ntok, kb, ke, qrow, z in recs:
        assert 1 <= ntok <= tt and z == 0 and qrow == b * Sq + tok0
        r = tok0 // qbs
        assert (tok0 + ntok - 1) // qbs == r                      # never crosses a q-block
        assert (kb, ke) == (bptr[b, g, r], bptr[b, g, r + 1])
        seen[b, g, tok0:tok0 + ntok] += 1
    assert np.all(seen == 1)
    _check_order(recs, lambda r: (r[0], r[1], r[2]))


def test_prefill_tiles_hold_exactly_the_visible_key_span():
    for mask, w in (("causal", -1), ("causal", 37), ("dense", -1), ("causal", 0)):
        p = W.make_prefill_problem(2, q_lens=[130, 7, 300], prefix_lens=[0, 250, 90], Hq=4,
                                   Hkv=2, D=8, page_size=16, mask_type=mask, window_left=w)
        tt = 32
        recs = PL.plan_prefill_tiles(2, p["qo_indptr"], p["seq_lens_kv"], tt, mask, w)
        qo = p["qo_indptr"].numpy()
        seen = {}
        for b, g, tok0, ntok, kb, ke, qrow, _ in recs:
            assert qrow == qo[b] + tok0
            vis = set()
            for i in range(tok0, tok0 + ntok):
                vis.update(BF.prefill_visible(p, b, i))
                seen[(b, g, i)] = seen.get((b, g, i), 0) + 1
            if not vis:
                assert kb == ke == 0
                continue
            assert kb == min(vis) // 128 and ke == max(vis) // 128 + 1
        assert all(v == 1 for v in seen.values())
        assert len(seen) == 2 * int(qo[-1])
        _check_order(recs, lambda r: (r[0], r[1], r[2]))


def test_decode_splits_partition_the_visible_keys():
    lens = [1, 127, 128, 129, 1000, 5]
    for w in (-1, 0, 200):
        for chunk in (128, 256, 1024):
            off, items = PL.plan_decode(lens, 3, chunk, w)
            assert off[0] == 0 and np.all(np.diff(off) >= 1)
            assert len(items) == 3 * off[-1]
            for b, L in enumerate(lens):
                n = off[b + 1] - off[b]
                lo = max(0, L - 1 - w) if w >= 0 else 0
                for g in range(3):
                    rows = items[3 * off[b] + g * n: 3 * off[b] + (g + 1) * n]
                    assert np.all(rows[:, 0] == b) and np.all(rows[:, 1] == g)
                    assert rows[0, 2] == lo and rows[-1, 3] == L
                    assert np.all(rows[1:, 2] == rows[:-1, 3])
                    assert np.all(rows[:, 3] - rows[:, 2] <= chunk)
                    assert np.all(rows[1:, 2] % chunk == 0)


def test_multi_query_decode_splits_cover_the_visible_union():
    """With nq queries per request the splits of (b, g) tile exactly the keys that at least
    one query of b sees (the brute-force visibility rule), cut at chunk multiples."""
    lens, q_lens = [1, 6, 130, 300, 1000, 2], [1, 6, 3, 8, 16, 2]
    for mask, w in (("dense", -1), ("causal", -1), ("causal", 0), ("causal", 100)):
        prob = dict(q_lens=q_lens, seq_lens=lens, mask_type=mask, window_left=w)
        for chunk in (128, 256):
            off, items = PL.plan_decode(lens, 2, chunk, w, q_lens=q_lens)
            for b, L in enumerate(lens):
                seen = sorted(set(j for i in range(q_lens[b])
                                  for j in BF.decode_visible(prob, b, i)))
                n = off[b + 1] - off[b]
                for g in range(2):
                    rows = items[2 * off[b] + g * n: 2 * off[b] + (g + 1) * n]
                    assert rows[0, 2] == seen[0] and rows[-1, 3] == seen[-1] + 1
                    assert seen == list(range(seen[0], seen[-1] + 1))
                    assert np.all(rows[1:, 2] == rows[:-1, 3])
                    assert np.all(rows[1:, 2] % chunk == 0)
                    assert np.all(rows[:, 3] - rows[:, 2] <= chunk)


def test_decode_work_order_is_a_stable_size_class_sort():
    lens = [1, 700, 129, 4000, 333, 2049]
    chunk = 512
    _, items = PL.plan_decode(lens, 2, chunk)
    order = PL.decode_work_order(items, chunk)
    assert sorted(order.tolist()) == list(range(len(items)))
    size = items[order, 3] - items[order, 2]
    cls = np.minimum(7, 8 * size // chunk)
    assert np.all(np.diff(cls) <= 0)                       # larger classes first
    for c in np.unique(cls):
        assert np.all(np.diff(order[cls == c]) > 0)       # list order inside a class
    assert size[0] == chunk and size[-1] == min(items[:, 3] - items[:, 2])


def test_indexed_csr_keeps_caller_order_and_drops_what_cannot_be_seen():
    p = W.make_qsa_indexed_problem(5, [16, 24], Hq=2, Hkv=1, D=8, block_size=4, n_near=2,
                                   n_random=3, extra_cols=4, junk=0.5)
    idx = p["sel_indices"].numpy().copy()
    NB = p["block_first"].numel()
    idx[3, 0] = NB + 5                           # out of range: dropped
    indptr, indices = PL.plan_indexed(idx, p["lo"], p["hi"], p["block_first"], p["block_last"])
    for t in range(idx.shape[0]):
        row = indices[indptr[t]:indptr[t + 1]].tolist()
        seen = BF.qsa_indexed_visible(dict(p, sel_indices=idx), t)
        # exactly the listed blocks that hold a visible key, in the order listed
        want = [int(g) for g in idx[t] if 0 <= g < NB and any(4 * g <= j <= 4 * g + 3 for j in seen)]
        assert row == want


def test_decode_chunk_formula():
    # floor(64 * 8 * 64 / (16 * 152)) = 13 tiles of 128 keys
    assert PL.decode_split_chunk(64, 8, 8192, 152) == 1664
    assert PL.decode_split_chunk(1, 1, 100, 152) == 128
    assert PL.decode_split_chunk(4096, 8, 1000, 148) == 128 * 8
    assert PL.decode_split_chunk(4096, 8, 1 << 20, 148) % 128 == 0


def test_bitmap_csr_matches_bruteforce():
    p = W.make_qsa_problem(3, [16, 24, 8], Hq=2, Hkv=1, D=8, block_size=4, n_near=2,
                           n_random=3)
    p["lo"] = p["lo"] + torch.tensor([(t % 3) for t in range(48)], dtype=torch.int32)
    indptr, indices = PL.plan_bitmap(p["sel_blocks"], p["lo"], p["hi"], p["block_first"],
                                     p["block_last"])
    first = p["block_first"].numpy()
    for t in range(48):
        got = indices[indptr[t]:indptr[t + 1]].tolist()
        js = BF.qsa_visible(p, t)
        blocks = sorted(set(int(np.searchsorted(first, j, side="right") - 1) for j in js))
        assert got == blocks
