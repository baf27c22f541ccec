"""The three CSA2 modes end to end ("DeepSeek-V4.1-Flash and the 890-byte KV cache",
section 2: Full computes its own KV, indexer scores and top-512; Reindex reuses a
preceding layer's caches but rescored with its own indexer query; Reuse inherits both
cache and indices and only attends).

Full mode is checked stage by stage against the oracle: the packed bytes bit-exact, the
scores within 1e-3 * M, the top-512 bit-exact on the GPU's own scores, and the attention
within 2e-2 on the GPU-selected indices.  Mode identities are checked bit-exact."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


def _setup(orc, csa2, B, T, seed, heads_I=64):
    max_pages = (T + 127) // 128
    cache = Cache(B, max_pages)
    # entries 0..T-2 already cached; the step packs entry T-1 of every request
    lat, key, req_e, pos_e = fill_cache(cache, [T - 1] * B, seed)
    new_lat = synth.normal_bf16(seed + 11, (B, 512))
    new_key = synth.normal_bf16(seed + 12, (B, 128))
    new_req = np.arange(B, dtype=np.int32)
    new_pos = np.full(B, T - 1, np.int64)
    kv_h, ix_h = orc.alloc_pages(cache.n_pages)
    orc.pack_kv(np.concatenate([lat, new_lat]), np.concatenate([key, new_key]), np.concatenate([req_e, new_req]),
                np.concatenate([pos_e, new_pos]), kv_h, ix_h, None, max_pages)
    q = synth.normal_bf16(seed + 13, (B, 64, 512))
    q_idx = synth.normal_bf16(seed + 14, (B, heads_I, 128))
    w = synth.normal_f32(seed + 15, (B, heads_I))
    window = synth.normal_bf16(seed + 16, (B * 128, 512))
    d = dict(
        host=dict(kv=kv_h, ix=ix_h, q=q, q_idx=q_idx, w=w, window=window, max_pages=max_pages),
        cache=cache,
        args=dict(n_q=B, t_max=T, q=dev_bf16(q), req=dev(np.arange(B, dtype=np.int32)),
                  n_visible=dev(np.full(B, T, np.int32)), window=dev_bf16(window),
                  win_start=dev(np.arange(B, dtype=np.int64) * 128), win_len=dev(np.full(B, 128, np.int32)),
                  cache=cache.c, q_idx=dev_bf16(q_idx), w=dev(w), heads_I=heads_I),
        new=dict(n_new=B, new_latent=dev_bf16(new_lat), new_idx_key=dev_bf16(new_key), new_req=dev(new_req),
                 new_pos=dev(new_pos)),
    )
    return d


def _outputs(B, T):
    ld = ((T + 3) // 4) * 4
    return dict(topk_idx=torch.full((B, 512), -9, dtype=torch.int32, device="cuda"),
                out=torch.zeros((B, 64, 512), dtype=torch.bfloat16, device="cuda"),
                lse=torch.zeros((B, 64), dtype=torch.float32, device="cuda"),
                scores=torch.full((B, ld), float("nan"), device="cuda"), ld=ld)


@pytest.mark.parametrize("B,T", [(2, 2000), (3, 777)])
def test_full_mode_stage_by_stage(orc, csa2, B, T):
    d = _setup(orc, csa2, B, T, seed=60 + T)
    o = _outputs(B, T)
    step = csa2.make_step(**d["args"], **d["new"], **o)
    ws = csa2.alloc_workspace(B, 64, T, False)
    csa2.sparse_attn_full(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    h = d["host"]
    kv_g, ix_g = d["cache"].host()
    assert np.array_equal(kv_g, h["kv"]) and np.array_equal(ix_g, h["ix"])
    S = o["scores"].cpu().numpy()
    idx = o["topk_idx"].cpu().numpy()
    O = o["out"].float().cpu().numpy()
    for b in range(B):
        I, M = orc.index_score(h["q_idx"][b], h["w"][b], h["ix"], b, 0, T, None, h["max_pages"])
        assert (np.abs(S[b, :T] - I) <= 1e-3 * M).all()
        assert np.array_equal(idx[b], orc.topk(S[b, :T], 512))
        Oref, _ = orc.attention(h["q"][b], idx[b], h["kv"], b, h["window"][128 * b:128 * b + 128], 128, None, None,
                                h["max_pages"])
        assert np.abs(O[b] - Oref).max() <= 2e-2


def test_mode_identities(orc, csa2):
    B, T = 2, 1500
    d = _setup(orc, csa2, B, T, seed=70)
    ws = csa2.alloc_workspace(B, 64, T, True)
    full = _outputs(B, T)
    csa2.sparse_attn_full(csa2.make_step(**d["args"], **d["new"], **full), ws)
    # Reuse with Full's indices gives Full's output exactly
    reuse = _outputs(B, T)
    reuse["topk_idx"].copy_(full["topk_idx"])
    csa2.sparse_attn_reuse(csa2.make_step(**d["args"], **reuse), ws)
    # Reindex on the same (already packed) cache with the same indexer query selects the same entries
    reidx = _outputs(B, T)
    csa2.sparse_attn_reindex(csa2.make_step(**d["args"], **reidx), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    assert torch.equal(reuse["out"], full["out"]) and torch.equal(reuse["lse"], full["lse"])
    assert torch.equal(reidx["topk_idx"], full["topk_idx"])
    assert torch.equal(reidx["scores"], full["scores"])
    assert torch.equal(reidx["out"], full["out"])
    # scores kept in the workspace (scores=NULL) select the same entries
    nos = _outputs(B, T)
    nos.pop("scores")
    nos["ld"] = 0
    csa2.sparse_attn_reindex(csa2.make_step(**d["args"], **nos), ws)
    assert torch.equal(nos["topk_idx"], full["topk_idx"])
