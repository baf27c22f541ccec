"""Full-size parity of two further rows on sampled requests, in the benchmark's launch
configuration (64 requests x 131,072 entries, Full mode):

* MXFP4 68-byte indexer keys ("DeepSeek's Attention and KV Cache", "A Precision Primer",
  MX formats and E8M0; "DeepSeek-V4", the indexer in four bits): the pages of three
  page-aligned windows bit-exact, their scores within 1e-3 * M, the top-512 bit-exact on
  the GPU's row, attention within 2e-2;
* the hierarchical sparse indexer ("The hierarchical indexer"; "From First Principles:
  DeepSeek-V4.1-Flash Inference", "The Hierarchical Sparse Indexer"): the published pool
  bit-exact against the oracle's pool of the GPU's score row, then a Reindex over the
  pool with a fresh indexer query: slot scores within 1e-3 * M at all 16,384 listed
  positions, its top-512 bit-exact on the GPU's slot scores, attention within 2e-2."""
import numpy as np
import pytest
import torch

import synth
from helpers import host_bits
from test_gpu_fullsize import PAGE, TOL, DeviceCache, attn_excess, oracle_request

pytestmark = pytest.mark.gpu
B, T = 64, 131072


class MxDeviceCache(DeviceCache):
    """DeviceCache with MXFP4 indexer pages (8,704 bytes)."""

    def __init__(self, csa2, n_req, max_pages, seed):
        self.csa2, self.n_req, self.max_pages, self.seed, self.frac = csa2, n_req, max_pages, seed, 0.0
        n_pages = n_req * max_pages
        self.kv = torch.zeros(n_pages * csa2.KV_PAGE_BYTES, dtype=torch.uint8, device="cuda")
        self.idx = torch.zeros(n_pages * csa2.IDX_MX_PAGE_BYTES, dtype=torch.uint8, device="cuda")
        self.c = csa2.make_cache(self.kv, self.idx, max_pages, idx_format=csa2.IDX_MXFP4)
        self.ws = csa2.alloc_workspace(1, 64, 0, False)

    def pages(self, r):
        kvp, ixp = self.csa2.KV_PAGE_BYTES, self.csa2.IDX_MX_PAGE_BYTES
        m = self.max_pages
        return (self.kv[r * m * kvp:(r + 1) * m * kvp].cpu().numpy(),
                self.idx[r * m * ixp:(r + 1) * m * ixp].cpu().numpy())


def _mx_oracle_request(orc, dc, r, n_cached, positions, new_lat, new_key, new_pos):
    pos = np.unique(np.asarray(positions, np.int64))
    pos_c = pos[pos < n_cached]
    lat, key = dc.draws(r, n_cached)
    ix = torch.from_numpy(pos_c).cuda()
    lat_h = np.concatenate([host_bits(lat[ix]), new_lat])
    key_h = np.concatenate([host_bits(key[ix]), new_key])
    p_all = np.concatenate([pos_c, np.asarray(new_pos, np.int64)])
    del lat, key
    kv_h, _ = orc.alloc_pages(dc.max_pages)
    orc.pack_kv(lat_h, key_h, np.zeros(len(p_all), np.int32), p_all, kv_h,
                np.zeros(dc.max_pages * orc.IDX_PAGE_BYTES, np.uint8), None, dc.max_pages)
    ix_h = orc.alloc_idx_mx_pages(dc.max_pages)
    orc.pack_idx_mx(key_h, np.zeros(len(p_all), np.int32), p_all, ix_h, None, dc.max_pages)
    return kv_h, ix_h


def _step_inputs(csa2, seed):
    new_lat = synth.torch_normal_bf16(seed + 500, (B, 512), "cuda")
    new_key = synth.torch_normal_bf16(seed + 501, (B, 128), "cuda")
    rows = synth.torch_normal_bf16(seed + 502, (B * 128, 512), "cuda")
    ar = torch.arange(B, dtype=torch.int32, device="cuda")
    common = dict(n_q=B, t_max=T, req=ar, n_visible=torch.full((B,), T, dtype=torch.int32, device="cuda"),
                  window=rows, win_start=ar.to(torch.int64) * 128,
                  win_len=torch.full((B,), 128, dtype=torch.int32, device="cuda"))
    new = dict(n_new=B, new_latent=new_lat, new_idx_key=new_key, new_req=ar,
               new_pos=torch.full((B,), T - 1, dtype=torch.int64, device="cuda"))
    return new_lat, new_key, rows, common, new


def _outs(ld):
    return dict(topk_idx=torch.empty((B, 512), dtype=torch.int32, device="cuda"),
                out=torch.empty((B, 64, 512), dtype=torch.bfloat16, device="cuda"),
                lse=torch.empty((B, 64), dtype=torch.float32, device="cuda"),
                scores=torch.empty((B, ld), dtype=torch.float32, device="cuda"), ld=ld)


def test_mxfp4_full_decode_64x131072(orc, csa2):
    mp = T // PAGE
    dc = MxDeviceCache(csa2, B, mp, 560000)
    dc.fill(T - 1)
    new_lat, new_key, rows, common, new = _step_inputs(csa2, 560000)
    q = synth.torch_normal_bf16(560601, (B, 64, 512), "cuda")
    q_idx = synth.torch_normal_bf16(560602, (B, 64, 128), "cuda")
    w = synth.torch_normal_f32(560603, (B, 64), "cuda")
    o = _outs(T)
    ws = csa2.alloc_workspace(B, 64, T, False)
    csa2.sparse_attn_full(csa2.make_step(q=q, q_idx=q_idx, w=w, heads_I=64, cache=dc.c, **common, **new, **o), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    qh, qih, wh = host_bits(q), host_bits(q_idx), w.cpu().numpy()
    nl, nk, rw = host_bits(new_lat), host_bits(new_key), host_bits(rows)
    idx, O, L = o["topk_idx"].cpu().numpy(), o["out"].float().cpu().numpy(), o["lse"].cpu().numpy()
    windows = [(0, 4096), (T // 2, T // 2 + 4096), (T - 4096, T)]
    ixp = csa2.IDX_MX_PAGE_BYTES
    for r in (0, 41):
        sel = idx[r]
        win_pos = np.concatenate([np.arange(s0, s1) for s0, s1 in windows])
        kv_h, ix_h = _mx_oracle_request(orc, dc, r, T - 1, np.concatenate([win_pos, sel[sel >= 0]]),
                                        nl[r:r + 1], nk[r:r + 1], [T - 1])
        kv_g, ix_g = dc.pages(r)
        S_row = o["scores"][r].cpu().numpy()
        for s0, s1 in windows:
            p0, p1 = s0 // PAGE, (s1 + PAGE - 1) // PAGE
            assert np.array_equal(ix_g[p0 * ixp:p1 * ixp], ix_h[p0 * ixp:p1 * ixp]), (r, s0)
            I, M = orc.index_score_mx(qih[r], wh[r], ix_h, 0, s0, s1, None, mp)
            assert (np.abs(S_row[s0:s1] - I) <= 1e-3 * M).all(), (r, s0)
        assert np.array_equal(sel, orc.topk(S_row, 512)), r
        Oref, lref = orc.attention(qh[r], sel, kv_h, 0, rw[128 * r:128 * r + 128], 128, None, None, mp)
        assert attn_excess(O[r], Oref) <= TOL, r
        assert np.abs(L[r] - lref).max() <= 1e-2, r


def test_pool_full_decode_then_reindex_64x131072(orc, csa2):
    mp = T // PAGE
    dc = DeviceCache(csa2, B, mp, 570000)
    dc.fill(T - 1)
    new_lat, new_key, rows, common, new = _step_inputs(csa2, 570000)
    q = synth.torch_normal_bf16(570601, (B, 64, 512), "cuda")
    pool = torch.empty((B, 16384), dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(B, 64, T, False, pool=True)
    full = _outs(T)
    csa2.sparse_attn_full(csa2.make_step(q=q, q_idx=synth.torch_normal_bf16(570602, (B, 64, 128), "cuda"),
                                         w=synth.torch_normal_f32(570603, (B, 64), "cuda"), heads_I=64, cache=dc.c,
                                         pool=pool, **common, **new, **full), ws)
    q_idx = synth.torch_normal_bf16(570604, (B, 64, 128), "cuda")
    w = synth.torch_normal_f32(570605, (B, 64), "cuda")
    re = _outs(16384)
    csa2.sparse_attn_reindex(csa2.make_step(q=q, q_idx=q_idx, w=w, heads_I=64, cache=dc.c, pool=pool, **common,
                                            **re), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    P = pool.cpu().numpy()
    qh, qih, wh = host_bits(q), host_bits(q_idx), w.cpu().numpy()
    nl, nk, rw = host_bits(new_lat), host_bits(new_key), host_bits(rows)
    G, idx = re["scores"].cpu().numpy(), re["topk_idx"].cpu().numpy()
    O, L = re["out"].float().cpu().numpy(), re["lse"].cpu().numpy()
    for r in (7, 60):
        ref, n = orc.block_pool(full["scores"][r].cpu().numpy(), T)
        assert np.array_equal(P[r], ref), r
        kv_h, ix_h = oracle_request(orc, dc, r, T - 1, P[r, :n], nl[r:r + 1], nk[r:r + 1], [T - 1])
        I, M = orc.index_score_at(qih[r], wh[r], ix_h, 0, P[r, :n], max_pages=mp)
        assert (np.abs(G[r, :n] - I) <= 1e-3 * M).all(), r
        sel = orc.pool_topk(G[r, :n], P[r], n, 512)
        assert np.array_equal(idx[r], sel), r
        Oref, lref = orc.attention(qh[r], sel, kv_h, 0, rw[128 * r:128 * r + 128], 128, None, None, mp)
        assert attn_excess(O[r], Oref) <= TOL, r
        assert np.abs(L[r] - lref).max() <= 1e-2, r
