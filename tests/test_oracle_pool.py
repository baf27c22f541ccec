"""Pins of the oracle's hierarchical sparse indexer ("DeepSeek's Attention and KV Cache",
"The hierarchical indexer"; "From First Principles: DeepSeek-V4.1-Flash Inference", "The
Hierarchical Sparse Indexer").

The pool is pinned by what characterises it, not by retyping it: its size from the
printed figures; the kept blocks dominate every other block under (block maximum desc,
block index asc), checked pair by pair against maxima computed here; exactly the visible
positions of the kept blocks are listed, ascending; a row of at most 2,048 blocks gives
every visible position; and, from the mathematics, the Full layer's own top-512 lies in
its pool, so a Reindex over the pool with the Full layer's scores selects the same 512
entries.  Index scores at listed positions equal the range scores already pinned."""
import json
import os

import numpy as np
import pytest

import synth

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hier_pool.json")))


def test_pool_size_from_the_pages(orc):
    assert G["block_positions"] * G["blocks_kept"] == G["pool_positions"] == 16384
    assert (orc.POOL_BLOCK, orc.POOL_BLOCKS, orc.POOL) == (8, 2048, 16384)


def _block_max(s, nv, block):
    nb = (nv + block - 1) // block
    return np.array([max(float(v) for v in s[j * block:min(nv, (j + 1) * block)]) for j in range(nb)])


def _check_pool(orc, s, nv, block, keep):
    pool, n = orc.block_pool(s, nv, block, keep)
    assert pool.size == block * keep and (pool[n:] == -1).all()
    listed = pool[:n]
    assert (np.diff(listed) > 0).all() and (listed >= 0).all() and (listed < nv).all()
    bm = _block_max(s, nv, block) + 0.0          # -0 -> +0
    nb = bm.size
    kept = sorted(set(int(p) // block for p in listed))
    assert len(kept) == min(keep, nb)
    # exactly the visible positions of the kept blocks
    want = [p for j in kept for p in range(j * block, min(nv, (j + 1) * block))]
    assert listed.tolist() == want
    # dominance: every kept block beats every dropped block under (max desc, index asc)
    dropped = sorted(set(range(nb)) - set(kept))
    for j in kept:
        for i in dropped:
            assert bm[j] > bm[i] or (bm[j] == bm[i] and j < i), (j, i, bm[j], bm[i])
    return pool, n


@pytest.mark.parametrize("nv,block,keep", [(11, 2, 3), (50, 8, 3), (1000, 8, 40), (997, 8, 124), (64, 8, 8),
                                           (65, 8, 8), (5, 8, 3), (0, 8, 3)])
def test_pool_characterisation_random_and_ties(orc, nv, block, keep):
    rng = np.random.default_rng(nv + block + keep)
    s = rng.standard_normal(max(nv, 1)).astype(np.float32)
    s[rng.integers(max(nv, 1), size=max(nv, 1) // 3)] = 0.5          # many equal maxima
    if nv > 4:
        s[1], s[3] = -0.0, 0.0
    _check_pool(orc, s, nv, block, keep)
    t = np.round(s * 2).astype(np.float32) / 2                       # heavy ties
    _check_pool(orc, t, nv, block, keep)


def test_short_rows_list_every_visible_position(orc):
    s = synth.normal_f32(801, (16384 + 5,))
    for nv in (1, 7, 8, 9, 1000, 16384):
        pool, n = orc.block_pool(s, nv)
        assert n == nv and pool[:n].tolist() == list(range(nv))


def test_full_topk_lies_in_its_pool_and_reindex_reproduces_it(orc):
    for seed, nv in ((802, 40000), (803, 16385), (804, 131072)):
        s = synth.normal_f32(seed, (nv,))
        pool, n = orc.block_pool(s, nv)
        assert 16384 - 7 <= n <= 16384                               # 2,048 blocks, the last may be partial
        top = orc.topk(s, 512)
        assert set(top.tolist()) <= set(pool[:n].tolist())
        again = orc.pool_topk(s[pool[:n]], pool, n, 512)
        assert np.array_equal(again, top)


def test_pool_topk_short_pool_pads(orc):
    s = synth.normal_f32(805, (300,))
    pool, n = orc.block_pool(s, 300)
    out = orc.pool_topk(s[pool[:n]], pool, n, 512)
    assert out[:300].tolist() == list(range(300)) and (out[300:] == -1).all()


@pytest.mark.parametrize("mx", [False, True])
def test_index_score_at_equals_range_scores(orc, mx):
    keys = synth.normal_bf16(806, (400, 128))
    if mx:
        pages = orc.alloc_idx_mx_pages(4)
        orc.pack_idx_mx(keys, np.zeros(400, np.int32), np.arange(400, dtype=np.int64), pages, max_pages=4)
        rng_fn = orc.index_score_mx
    else:
        kv, pages = orc.alloc_pages(4)
        orc.pack_kv(synth.normal_bf16(807, (400, 512)), keys, np.zeros(400, np.int32),
                    np.arange(400, dtype=np.int64), kv, pages, None, 4)
        rng_fn = orc.index_score
    q = synth.normal_bf16(808, (64, 128))
    w = synth.normal_f32(809, (64,))
    I_all, M_all = rng_fn(q, w, pages, 0, 0, 400, None, 4)
    pos = np.array([0, 7, 8, 129, 255, 256, 399], np.int32)
    I, M = orc.index_score_at(q, w, pages, 0, pos, mx=mx, max_pages=4)
    assert np.array_equal(I, I_all[pos]) and np.array_equal(M, M_all[pos])
