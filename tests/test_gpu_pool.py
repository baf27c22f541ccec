"""Parity of the hierarchical sparse indexer ("DeepSeek's Attention and KV Cache", "The
hierarchical indexer"; "From First Principles: DeepSeek-V4.1-Flash Inference", "The
Hierarchical Sparse Indexer").

A Full step that publishes its pool: the pool equals the oracle's pool of the GPU's own
score row, bit-exact (block maxima, top 2,048 blocks, ascending positions).  A Reindex
step over that pool with a fresh indexer query: pool-slot scores within 1e-3 * M of the
oracle at the listed positions, the top-512 bit-exact against the oracle's selection on
the GPU's slot scores, attention within 2e-2.  With the Full layer's own query, the
pool-restricted Reindex reproduces the Full layer's selection and output exactly (the
Full top-512 lies in its pool).  A malformed pool sets the error word."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


def _setup(orc, csa2, B, T, seed, mx, block_table=None):
    max_pages = (T + 127) // 128
    cache = Cache(B, max_pages, mx=mx, block_table=block_table)
    bt = cache.bt_np
    lat, key, req_e, pos_e = fill_cache(cache, [T] * B, seed)
    if mx:
        ix_h = orc.alloc_idx_mx_pages(cache.n_pages)
        orc.pack_idx_mx(key, req_e, pos_e, ix_h, bt, max_pages)
        kv_h, _ = orc.alloc_pages(cache.n_pages)
        orc.pack_kv(lat, key, req_e, pos_e, kv_h, np.zeros(cache.n_pages * orc.IDX_PAGE_BYTES, np.uint8), bt,
                    max_pages)
    else:
        kv_h, ix_h = orc.alloc_pages(cache.n_pages)
        orc.pack_kv(lat, key, req_e, pos_e, kv_h, ix_h, bt, max_pages)
    window = synth.normal_bf16(seed + 16, (B * 128, 512))
    common = dict(n_q=B, t_max=T, req=dev(np.arange(B, dtype=np.int32)), n_visible=dev(np.full(B, T, np.int32)),
                  window=dev_bf16(window), win_start=dev(np.arange(B, dtype=np.int64) * 128),
                  win_len=dev(np.full(B, 128, np.int32)), cache=cache.c)
    return cache, kv_h, ix_h, window, max_pages, common


def _outs(B, ld):
    return dict(topk_idx=torch.full((B, 512), -9, dtype=torch.int32, device="cuda"),
                out=torch.zeros((B, 64, 512), dtype=torch.bfloat16, device="cuda"),
                lse=torch.zeros((B, 64), dtype=torch.float32, device="cuda"),
                scores=torch.full((B, ld), float("nan"), device="cuda"), ld=ld)


@pytest.mark.parametrize("B,T,mx", [(3, 40000, False), (2, 20003, True), (2, 9001, False), (1, 16390, False)])
def test_pool_full_then_reindex(orc, csa2, B, T, mx):
    seed = 900 + T % 97
    cache, kv_h, ix_h, window, mp, common = _setup(orc, csa2, B, T, seed, mx)
    score = orc.index_score_mx if mx else orc.index_score
    q = synth.normal_bf16(seed + 1, (B, 64, 512))
    qi_full = synth.normal_bf16(seed + 2, (B, 64, 128))
    w_full = synth.normal_f32(seed + 3, (B, 64))
    ws = csa2.alloc_workspace(B, 64, T, False, pool=True)
    pool = torch.full((B, 16384), -7, dtype=torch.int32, device="cuda")
    ldf = ((T + 3) // 4) * 4
    full = _outs(B, ldf)
    csa2.sparse_attn_full(csa2.make_step(**common, q=dev_bf16(q), q_idx=dev_bf16(qi_full), w=dev(w_full),
                                         pool=pool, **full), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    S = full["scores"].cpu().numpy()
    P = pool.cpu().numpy()
    for b in range(B):
        ref, n = orc.block_pool(S[b, :T], T)
        assert np.array_equal(P[b], ref), b
        assert np.array_equal(full["topk_idx"][b].cpu().numpy(), orc.topk(S[b, :T], 512))
    # Reindex over the pool with a fresh indexer query
    qi = synth.normal_bf16(seed + 4, (B, 64, 128))
    w = synth.normal_f32(seed + 5, (B, 64))
    re = _outs(B, 16384)
    csa2.sparse_attn_reindex(csa2.make_step(**common, q=dev_bf16(q), q_idx=dev_bf16(qi), w=dev(w), pool=pool, **re),
                             ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    G = re["scores"].cpu().numpy()
    idx = re["topk_idx"].cpu().numpy()
    O = re["out"].float().cpu().numpy()
    for b in range(B):
        _, n = orc.block_pool(S[b, :T], T)
        I, M = orc.index_score_at(qi[b], w[b], ix_h, b, P[b, :n], mx=mx, max_pages=mp)
        assert (np.abs(G[b, :n] - I) <= 1e-3 * M).all(), b
        assert np.isnan(G[b, n:]).all()
        assert np.array_equal(idx[b], orc.pool_topk(G[b, :n], P[b], n, 512)), b
        Oref, _ = orc.attention(q[b], idx[b], kv_h, b, window[128 * b:128 * b + 128], 128, None, None, mp)
        assert np.abs(O[b] - Oref).max() <= 2e-2
    # with the Full layer's own query the pool-restricted Reindex reproduces Full exactly
    same = _outs(B, 16384)
    csa2.sparse_attn_reindex(csa2.make_step(**common, q=dev_bf16(q), q_idx=dev_bf16(qi_full), w=dev(w_full),
                                            pool=pool, **same), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    assert torch.equal(same["topk_idx"], full["topk_idx"])
    assert torch.equal(same["out"], full["out"]) and torch.equal(same["lse"], full["lse"])


def test_pool_scores_in_workspace_and_malformed_pool(orc, csa2):
    B, T = 2, 30000
    cache, kv_h, ix_h, window, mp, common = _setup(orc, csa2, B, T, 950, False)
    q = dev_bf16(synth.normal_bf16(951, (B, 64, 512)))
    qi = dev_bf16(synth.normal_bf16(952, (B, 64, 128)))
    w = dev(synth.normal_f32(953, (B, 64)))
    ws = csa2.alloc_workspace(B, 64, T, True, pool=True)
    pool = torch.full((B, 16384), -7, dtype=torch.int32, device="cuda")
    a = _outs(B, 4)
    a.pop("scores")
    a["ld"] = 0
    csa2.sparse_attn_full(csa2.make_step(**common, q=q, q_idx=qi, w=w, pool=pool, **a), ws)
    b = _outs(B, 4)
    b.pop("scores")
    b["ld"] = 0
    csa2.sparse_attn_reindex(csa2.make_step(**common, q=q, q_idx=qi, w=w, pool=pool, **b), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    assert torch.equal(a["topk_idx"], b["topk_idx"]) and torch.equal(a["out"], b["out"])
    # a pool whose blocks do not start on a multiple of 8 is reported (info 6)
    bad = pool.clone()
    bad[0, :8] = torch.arange(3, 11, dtype=torch.int32, device="cuda")
    c = _outs(B, 4)
    c.pop("scores")
    c["ld"] = 0
    csa2.sparse_attn_reindex(csa2.make_step(**common, q=q, q_idx=qi, w=w, pool=bad, **c), ws)
    assert csa2.check(ws) == (csa2.ERR_DEVICE, 6)


@pytest.mark.parametrize("mx", [False, True])
def test_pool_over_a_block_table(orc, csa2, mx):
    """Paged cache with a permuted block table: the gather resolves every pooled block's
    page through it."""
    B, T = 2, 24000
    mp = (T + 127) // 128
    perm = np.random.default_rng(960 + mx).permutation(B * mp).astype(np.int32).reshape(B, mp)
    cache, kv_h, ix_h, window, mp, common = _setup(orc, csa2, B, T, 961, mx, block_table=perm)
    bt = cache.bt_np
    q = synth.normal_bf16(962, (B, 64, 512))
    qi = synth.normal_bf16(963, (B, 64, 128))
    w = synth.normal_f32(964, (B, 64))
    ws = csa2.alloc_workspace(B, 64, T, False, pool=True)
    pool = torch.full((B, 16384), -7, dtype=torch.int32, device="cuda")
    full = _outs(B, ((T + 3) // 4) * 4)
    csa2.sparse_attn_full(csa2.make_step(**common, q=dev_bf16(q), q_idx=dev_bf16(qi), w=dev(w), pool=pool, **full),
                          ws)
    qi2 = synth.normal_bf16(965, (B, 64, 128))
    w2 = synth.normal_f32(966, (B, 64))
    re = _outs(B, 16384)
    csa2.sparse_attn_reindex(csa2.make_step(**common, q=dev_bf16(q), q_idx=dev_bf16(qi2), w=dev(w2), pool=pool,
                                            **re), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    S, P = full["scores"].cpu().numpy(), pool.cpu().numpy()
    G, idx = re["scores"].cpu().numpy(), re["topk_idx"].cpu().numpy()
    O = re["out"].float().cpu().numpy()
    for b in range(B):
        ref, n = orc.block_pool(S[b, :T], T)
        assert np.array_equal(P[b], ref)
        I, M = orc.index_score_at(qi2[b], w2[b], ix_h, b, P[b, :n], mx=mx, block_table=bt, max_pages=mp)
        assert (np.abs(G[b, :n] - I) <= 1e-3 * M).all()
        assert np.array_equal(idx[b], orc.pool_topk(G[b, :n], P[b], n, 512))
        Oref, _ = orc.attention(q[b], idx[b], kv_h, b, window[128 * b:128 * b + 128], 128, None, bt, mp)
        assert np.abs(O[b] - Oref).max() <= 2e-2
