"""Parity of the MXFP4 indexer key ("DeepSeek's Attention and KV Cache": "A Precision
Primer", MX formats and E8M0, and "DeepSeek-V4", the indexer in four bits; "From First
Principles: DeepSeek-V4.1-Flash Inference", "What's in a cell": 64 B of nibbles plus four
E8M0 scales, 68 B).

The packed pages are bit-exact against the oracle (random, block table, outliers and edge
blocks); index scores are within 1e-3 * M (M = sum_j |w_j| ReLU(...); products of MXFP4
values are exact in fp32, so only the accumulation order differs); a Full-mode step over
an MXFP4 cache selects the oracle's top-512 of the GPU's own scores bit-exact and
attends within 2e-2."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


def _oracle_pages(orc, cache, lat, key, req, pos):
    kv, _ = orc.alloc_pages(cache.n_pages)
    ix_unused = np.zeros(cache.n_pages * orc.IDX_PAGE_BYTES, np.uint8)
    orc.pack_kv(lat, key, req, pos, kv, ix_unused, cache.bt_np, cache.max_pages)
    ix = orc.alloc_idx_mx_pages(cache.n_pages)
    orc.pack_idx_mx(key, req, pos, ix, cache.bt_np, cache.max_pages)
    return kv, ix


def _assert_pages(orc, cache, lat, key, req, pos):
    kv_h, ix_h = _oracle_pages(orc, cache, lat, key, req, pos)
    kv_g, ix_g = cache.host()
    assert ix_g.size == cache.n_pages * 8704
    bad = np.nonzero(kv_g != kv_h)[0]
    assert bad.size == 0, f"main-KV bytes differ at {bad[:8]}"
    bad = np.nonzero(ix_g != ix_h)[0]
    assert bad.size == 0, f"MXFP4 indexer bytes differ at {bad[:8]}: gpu {ix_g[bad[:8]]} oracle {ix_h[bad[:8]]}"
    return kv_h, ix_h


def test_pack_mx_random_block_table_outliers(orc, csa2):
    cache = Cache(n_req=3, max_pages=3, mx=True)
    _assert_pages(orc, cache, *fill_cache(cache, [300, 130, 1], seed=501))
    bt = np.array([[4, 1], [0, 3]], np.int32)
    cache = Cache(n_req=2, max_pages=2, block_table=bt, n_pages=5, mx=True)
    _assert_pages(orc, cache, *fill_cache(cache, [256, 200], seed=502, outlier_frac=0.05))


def _edge_keys():
    f = np.float32
    rng = np.random.default_rng(503)
    blocks = [
        np.zeros(32, f), -np.zeros(32, f),
        np.full(32, 2.0 ** -130, f) * np.array([1, -1] * 16, f),           # subnormal amax: e clamps to -127
        np.array([6.0] + [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4 + [-5.0, -0.25, -3.5], f),  # scale 1, ties
        np.array([3.0] + [1.0] * 31, f),                                    # amax = 6 * 2^-1 exactly
        np.array([3.015625] + [0.1] * 31, f),                               # 3 + delta: scale 1, max -> 3
        np.array([6.0 * 2 ** 100] + [2.0 ** 98] * 31, f),                   # large exponents
        np.array([3.3e38] + [-1e38] * 31, f),                               # near the bf16 maximum
        (rng.standard_normal(32) * 2.0 ** -100).astype(f),
        (rng.standard_normal(32) * 1e4).astype(f),
    ]
    rows = []
    for i in range(0, len(blocks), 4):
        grp = blocks[i:i + 4] + [rng.standard_normal(32).astype(f)] * (4 - len(blocks[i:i + 4]))
        rows.append(np.concatenate(grp))
    # every bf16 value with |x| <= 6 as an element of a block whose scale is 1
    vals = synth.bf16_to_f32(np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16))
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 6.0)]
    vals = np.concatenate([vals, np.zeros((-vals.size) % 31, np.float32)]).reshape(-1, 31)
    blk = np.concatenate([np.full((vals.shape[0], 1), 6.0, np.float32), vals], axis=1)
    blk = np.concatenate([blk, np.tile(blk[:1], ((-blk.shape[0]) % 4, 1))]).reshape(-1, 128)
    return synth.bf16_bits(np.concatenate([np.stack(rows), blk]).astype(np.float32))


def test_pack_mx_edge_blocks_and_every_bf16_element(orc, csa2):
    key = _edge_keys()
    n = key.shape[0]
    max_pages = (n + 127) // 128
    cache = Cache(n_req=1, max_pages=max_pages, mx=True)
    lat = synth.normal_bf16(504, (n, 512))
    req, pos = np.zeros(n, np.int32), np.arange(n, dtype=np.int64)
    cache.pack(lat, key, req, pos)
    _assert_pages(orc, cache, lat, key, req, pos)


def _index_run(orc, csa2, n_entries, heads_I, group, seed, qscale=1.0, outliers=0.0):
    n_req = len(n_entries)
    max_pages = (max(n_entries) + 127) // 128
    cache = Cache(n_req, max_pages, mx=True)
    lat, key, req_e, pos_e = fill_cache(cache, n_entries, seed, outliers)
    _, ix_h = _oracle_pages(orc, cache, lat, key, req_e, pos_e)
    req_q = np.repeat(np.arange(n_req), group).astype(np.int32)
    nvis = np.array([max(0, n_entries[r] - i) for r in range(n_req) for i in range(group)], np.int32)
    n_q = req_q.size
    q_idx = synth.normal_bf16(seed + 7, (n_q, heads_I, 128), scale=qscale)
    w = synth.normal_f32(seed + 8, (n_q, heads_I))
    t_max = int(max(n_entries))
    ld = ((t_max + 3) // 4) * 4 + 4
    scores = torch.full((n_q, ld), float("nan"), device="cuda")
    ws = csa2.alloc_workspace(n_q, heads_I, t_max, False)
    csa2.index_score(dev_bf16(q_idx), dev(w), heads_I, dev(req_q), dev(nvis), n_q, group, t_max, cache.c, scores,
                     ld, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    g = scores.cpu().numpy()
    for q in range(n_q):
        nv = int(nvis[q])
        I, M = orc.index_score_mx(q_idx[q], w[q], ix_h, int(req_q[q]), 0, nv, None, max_pages)
        err = np.abs(g[q, :nv].astype(np.float64) - I)
        bad = np.nonzero(err > 1e-3 * M)[0]
        assert bad.size == 0, (q, bad[:5], g[q, bad[:5]], I[bad[:5]], M[bad[:5]])
        assert np.isnan(g[q, nv:]).all(), "entries beyond the visible prefix must not be written"


@pytest.mark.parametrize("heads_I,group", [(64, 1), (32, 1), (64, 2), (32, 2)])
def test_index_mx_ragged(orc, csa2, heads_I, group):
    _index_run(orc, csa2, [1000, 333, 129], heads_I, group, seed=510 + heads_I + group)


def test_index_mx_outliers_peaky(orc, csa2):
    _index_run(orc, csa2, [5, 128, 700], 64, 1, seed=520, qscale=8.0, outliers=0.02)


def test_index_mx_many_tiles_per_cta(orc, csa2):
    """40 requests of 2,000-12,000 MXFP4 entries: about 14 tiles per persistent CTA across
    group boundaries, so the accumulator rotation and the per-issuer scale slots turn over."""
    rng = np.random.default_rng(530)
    _index_run(orc, csa2, [int(x) for x in rng.integers(2000, 12001, size=40)], 64, 1, seed=531)


def test_full_mode_over_mx_cache(orc, csa2):
    B, T = 3, 1100
    max_pages = (T + 127) // 128
    cache = Cache(B, max_pages, mx=True)
    lat, key, req_e, pos_e = fill_cache(cache, [T - 1] * B, seed=530)
    new_lat, new_key = synth.normal_bf16(531, (B, 512)), synth.normal_bf16(532, (B, 128))
    new_req, new_pos = np.arange(B, dtype=np.int32), np.full(B, T - 1, np.int64)
    kv_h, ix_h = _oracle_pages(orc, cache, np.concatenate([lat, new_lat]), np.concatenate([key, new_key]),
                               np.concatenate([req_e, new_req]), np.concatenate([pos_e, new_pos]))
    q = synth.normal_bf16(533, (B, 64, 512))
    q_idx = synth.normal_bf16(534, (B, 64, 128))
    w = synth.normal_f32(535, (B, 64))
    window = synth.normal_bf16(536, (B * 128, 512))
    ld = ((T + 3) // 4) * 4
    topk_idx = torch.full((B, 512), -9, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, 64, 512), dtype=torch.bfloat16, device="cuda")
    scores = torch.full((B, ld), float("nan"), device="cuda")
    step = csa2.make_step(n_q=B, t_max=T, q=dev_bf16(q), req=dev(np.arange(B, dtype=np.int32)),
                          n_visible=dev(np.full(B, T, np.int32)), window=dev_bf16(window),
                          win_start=dev(np.arange(B, dtype=np.int64) * 128), win_len=dev(np.full(B, 128, np.int32)),
                          cache=cache.c, q_idx=dev_bf16(q_idx), w=dev(w), n_new=B, new_latent=dev_bf16(new_lat),
                          new_idx_key=dev_bf16(new_key), new_req=dev(new_req), new_pos=dev(new_pos),
                          topk_idx=topk_idx, out=out, scores=scores, ld=ld)
    ws = csa2.alloc_workspace(B, 64, T, False)
    csa2.sparse_attn_full(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    kv_g, ix_g = cache.host()
    assert np.array_equal(kv_g, kv_h) and np.array_equal(ix_g, ix_h)
    S, idx, O = scores.cpu().numpy(), topk_idx.cpu().numpy(), out.float().cpu().numpy()
    for b in range(B):
        I, M = orc.index_score_mx(q_idx[b], w[b], ix_h, b, 0, T, None, max_pages)
        assert (np.abs(S[b, :T] - I) <= 1e-3 * M).all()
        assert np.array_equal(idx[b], orc.topk(S[b, :T], 512))
        Oref, _ = orc.attention(q[b], idx[b], kv_h, b, window[128 * b:128 * b + 128], 128, None, None, max_pages)
        assert np.abs(O[b] - Oref).max() <= 2e-2
