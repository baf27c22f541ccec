"""Parity at the full sizes of the decode and prefill workloads, on sampled requests.

The device builds every cache from seeded draws (the torch generators in synth) and runs
the step through the C ABI in the same launch configuration as the benchmark.  For a
few sampled requests (queries) the oracle packs, from the same seeded draws, the
entries it needs: page-aligned windows of the visible prefix, the GPU-selected entries
and the new entries.  Checked there: packed bytes bit-exact (whole pages of the windows,
main-KV records of the selected entries), index scores within 1e-3 * M on the windows
("DeepSeek's Attention and KV Cache", "DeepSeek-V3.2" indexer; "From MLA to DSA to
HCA/CSA", "CSA" scorer), the top-512 bit-exact on the GPU's own score row, attention
within 2e-2 max-abs beyond the bf16 output rounding (half an ulp of the exact value) and
lse within 1e-2 on the GPU-selected indices ("DeepSeek-V4":
selected entries plus the 128-row window).  One full 131072-entry row also reports the
overlap of the GPU's selection with the oracle's own top-512."""
import numpy as np
import pytest
import torch

import synth
from helpers import dev, host_bits

pytestmark = pytest.mark.gpu
TOL = 2e-2
PAGE, KVB = 128, 288


class DeviceCache:
    """n_req requests of max_pages pages each, filled by the library from seeded draws."""

    def __init__(self, csa2, n_req, max_pages, seed, frac=0.0):
        self.csa2, self.n_req, self.max_pages, self.seed, self.frac = csa2, n_req, max_pages, seed, frac
        n_pages = n_req * max_pages
        self.kv = torch.zeros(n_pages * csa2.KV_PAGE_BYTES, dtype=torch.uint8, device="cuda")
        self.idx = torch.zeros(n_pages * csa2.IDX_PAGE_BYTES, dtype=torch.uint8, device="cuda")
        self.c = csa2.make_cache(self.kv, self.idx, max_pages)
        self.ws = csa2.alloc_workspace(1, 64, 0, False)

    def draws(self, r, n):
        """Latents [n][512] and indexer keys [n][128] (device bf16) of request r's first n entries."""
        lat = synth.torch_normal_bf16_rows_with_outliers(self.seed + 1000 * r, n, 512, self.frac, 8.0, "cuda")
        key = synth.torch_normal_bf16_rows_with_outliers(self.seed + 1000 * r + 1, n, 128, self.frac, 8.0, "cuda")
        return lat, key

    def fill(self, n):
        for r in range(self.n_req):
            lat, key = self.draws(r, n)
            self.csa2.pack_kv(lat, key, torch.full((n,), r, dtype=torch.int32, device="cuda"),
                              torch.arange(n, dtype=torch.int64, device="cuda"), self.c, self.ws)
            del lat, key
        torch.cuda.synchronize()

    def pages(self, r):
        """Host copies of request r's main-KV and indexer pages."""
        kvp, ixp = self.csa2.KV_PAGE_BYTES, self.csa2.IDX_PAGE_BYTES
        m = self.max_pages
        return (self.kv[r * m * kvp:(r + 1) * m * kvp].cpu().numpy(),
                self.idx[r * m * ixp:(r + 1) * m * ixp].cpu().numpy())


def oracle_request(orc, dc, r, n_cached, positions, new_lat=None, new_key=None, new_pos=None):
    """Oracle-packed single-request pages holding only the entries at `positions`
    (cached ones regenerated from the seeded draws) plus the given new entries."""
    pos = np.unique(np.asarray(positions, np.int64))
    pos_c = pos[pos < n_cached]
    lat, key = dc.draws(r, n_cached)
    ix = torch.from_numpy(pos_c).cuda()
    lat_h, key_h = host_bits(lat[ix]), host_bits(key[ix])
    del lat, key
    kv_h, ix_h = orc.alloc_pages(dc.max_pages)
    orc.pack_kv(lat_h, key_h, np.zeros(len(pos_c), np.int32), pos_c, kv_h, ix_h, None, dc.max_pages)
    if new_lat is not None:
        orc.pack_kv(new_lat, new_key, np.zeros(len(new_pos), np.int32), np.asarray(new_pos, np.int64), kv_h, ix_h,
                    None, dc.max_pages)
    return kv_h, ix_h


def bf16_half_ulp(x):
    """Half a unit in the last place of bf16 (8 significant bits) at |x|: the rounding of an
    exact output to the bf16 output format alone can be off by this much."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


def attn_excess(O, Oref):
    """max over elements of |O - Oref| - half_ulp_bf16(Oref): must stay within 2e-2.  The
    bound is the stated 2e-2 max-abs plus the rounding the bf16 output format itself
    imposes (half an ulp of the exact value, 0.0625 at |O| in [16, 32), where the x8
    outlier layers put some outputs); nothing in it depends on how the kernel computes."""
    return float((np.abs(O - Oref) - bf16_half_ulp(Oref)).max())


def check_request(orc, csa2, dc, r, *, n_cached, nv, S_row, sel, q, q_idx, w, win_rows, O, L, windows,
                  new_lat=None, new_key=None, new_pos=None):
    """The sampled checks for one query of request r (see the module docstring)."""
    sel = np.asarray(sel)
    win_pos = np.concatenate([np.arange(s0, s1) for s0, s1 in windows])
    kv_h, ix_h = oracle_request(orc, dc, r, n_cached, np.concatenate([win_pos, sel[sel >= 0]]), new_lat, new_key,
                                new_pos)
    kv_g, ix_g = dc.pages(r)
    kvp, ixp = csa2.KV_PAGE_BYTES, csa2.IDX_PAGE_BYTES
    for s0, s1 in windows:  # page-aligned windows: whole pages bit-exact
        assert s0 % PAGE == 0 and (s1 % PAGE == 0 or s1 == nv)
        p0, p1 = s0 // PAGE, (s1 + PAGE - 1) // PAGE
        assert np.array_equal(kv_g[p0 * kvp:p1 * kvp], kv_h[p0 * kvp:p1 * kvp]), (r, s0)
        assert np.array_equal(ix_g[p0 * ixp:p1 * ixp], ix_h[p0 * ixp:p1 * ixp]), (r, s0)
        I, M = orc.index_score(q_idx, w, ix_h, 0, s0, s1, None, dc.max_pages)
        assert (np.abs(S_row[s0:s1] - I) <= 1e-3 * M).all(), (r, s0, np.abs(S_row[s0:s1] - I).max())
    for e in sel[sel >= 0]:  # main-KV records of the selected entries
        off = (e // PAGE) * kvp + (e % PAGE) * KVB
        assert np.array_equal(kv_g[off:off + KVB], kv_h[off:off + KVB]), (r, e)
    assert np.array_equal(sel, orc.topk(S_row[:nv], 512)), r
    Oref, lref = orc.attention(q, sel, kv_h, 0, win_rows, len(win_rows), None, None, dc.max_pages)
    err, exc = float(np.abs(O - Oref).max()), attn_excess(O, Oref)
    print(f"request {r}: attention max-abs error {err:.4f}, beyond the bf16 output rounding {exc:.4f} "
          f"(max |O| {float(np.abs(Oref).max()):.2f})")
    assert exc <= TOL, (r, err, exc)
    assert np.abs(L - lref).max() <= 1e-2, r


def _full_step(csa2, dc, B, T, seed, group=1, n_q=None, req=None, nvis=None, win=None, new=None, scores_ld=None):
    """One Full-mode step (pack the new entries, index, top-512, attention) with device draws."""
    n_q = B if n_q is None else n_q
    q = synth.torch_normal_bf16(seed + 1, (n_q, 64, 512), "cuda")
    q_idx = synth.torch_normal_bf16(seed + 2, (n_q, 64, 128), "cuda")
    w = synth.torch_normal_f32(seed + 3, (n_q, 64), "cuda")
    ld = scores_ld or T
    scores = torch.empty((n_q, ld), dtype=torch.float32, device="cuda")
    out = dict(topk_idx=torch.empty((n_q, 512), dtype=torch.int32, device="cuda"),
               out=torch.empty((n_q, 64, 512), dtype=torch.bfloat16, device="cuda"),
               lse=torch.empty((n_q, 64), dtype=torch.float32, device="cuda"), scores=scores, ld=ld)
    step = csa2.make_step(n_q=n_q, t_max=T, q=q, req=req, n_visible=nvis, window=win["rows"],
                          win_start=win["start"], win_len=win["len"], cache=dc.c, q_idx=q_idx, w=w, heads_I=64,
                          group=group, n_new=new["n"], new_latent=new["lat"], new_idx_key=new["key"],
                          new_req=new["req"], new_pos=new["pos"], **out)
    ws = csa2.alloc_workspace(n_q, 64, T, False)
    csa2.sparse_attn_full(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    return dict(q=q, q_idx=q_idx, w=w, **out)


def _decode_case(orc, csa2, B, T, seed, sampled, frac=0.0, full_row_overlap=False):
    mp = T // PAGE
    dc = DeviceCache(csa2, B, mp, seed, frac)
    dc.fill(T - 1)  # the step packs entry T-1 of every request
    new_lat = synth.torch_normal_bf16_rows_with_outliers(seed + 500, B, 512, 0.0, 1.0, "cuda")
    new_key = synth.torch_normal_bf16_rows_with_outliers(seed + 501, B, 128, 0.0, 1.0, "cuda")
    rows = synth.torch_normal_bf16(seed + 502, (B * 128, 512), "cuda")
    win = dict(rows=rows, start=torch.arange(B, dtype=torch.int64, device="cuda") * 128,
               len=torch.full((B,), 128, dtype=torch.int32, device="cuda"))
    new = dict(n=B, lat=new_lat, key=new_key, req=torch.arange(B, dtype=torch.int32, device="cuda"),
               pos=torch.full((B,), T - 1, dtype=torch.int64, device="cuda"))
    res = _full_step(csa2, dc, B, T, seed + 600, req=torch.arange(B, dtype=torch.int32, device="cuda"),
                     nvis=torch.full((B,), T, dtype=torch.int32, device="cuda"), win=win, new=new)
    S = res["scores"]
    idx = res["topk_idx"].cpu().numpy()
    O = res["out"].float().cpu().numpy()
    L = res["lse"].cpu().numpy()
    q, q_idx, w = host_bits(res["q"]), host_bits(res["q_idx"]), res["w"].cpu().numpy()
    nl, nk, rw = host_bits(new_lat), host_bits(new_key), host_bits(rows)
    windows = [(0, 4096), (T // 2, T // 2 + 4096), (T - 4096, T)]
    for r in sampled:
        check_request(orc, csa2, dc, r, n_cached=T - 1, nv=T, S_row=S[r].cpu().numpy(), sel=idx[r], q=q[r],
                      q_idx=q_idx[r], w=w[r], win_rows=rw[128 * r:128 * r + 128], O=O[r], L=L[r], windows=windows,
                      new_lat=nl[r:r + 1], new_key=nk[r:r + 1], new_pos=[T - 1])
    if full_row_overlap:
        r = sampled[0]
        _, ix_h = oracle_request(orc, dc, r, T - 1, np.arange(T - 1), nl[r:r + 1], nk[r:r + 1], [T - 1])
        I, _ = orc.index_score(q_idx[r], w[r], ix_h, 0, 0, T, None, mp)
        ov = len(np.intersect1d(orc.topk(I.astype(np.float32), 512), idx[r]))
        print(f"top-512 overlap with the oracle's own selection on a {T}-entry row: {ov}/512")
        assert ov >= 460
    return dc


def test_full_decode_64x131072(orc, csa2):
    # the benchmark's workload: 64 requests x 131072 entries, Full mode
    _decode_case(orc, csa2, 64, 131072, seed=510000, sampled=[0, 37, 63], full_row_overlap=True)


def test_million_token_decode_with_outliers_and_ratio2_layer(orc, csa2):
    # 8 requests x 1,048,576 entries, 1 % of entries x 8; then the ratio-2 layer's
    # 524,288 pooled entries
    dc = _decode_case(orc, csa2, 8, 1 << 20, seed=530000, sampled=[5], frac=0.01)
    del dc
    torch.cuda.empty_cache()
    _decode_case(orc, csa2, 8, 1 << 19, seed=540000, sampled=[2], frac=0.01)


def test_reuse_and_reindex_128x262144(orc, csa2):
    B, T = 128, 262144
    mp = T // PAGE
    dc = DeviceCache(csa2, B, mp, 520000)
    dc.fill(T)
    rows = synth.torch_normal_bf16(520502, (B * 128, 512), "cuda")
    req = torch.arange(B, dtype=torch.int32, device="cuda")
    nvis = torch.full((B,), T, dtype=torch.int32, device="cuda")
    common = dict(n_q=B, t_max=T, req=req, n_visible=nvis, window=rows,
                  win_start=torch.arange(B, dtype=torch.int64, device="cuda") * 128,
                  win_len=torch.full((B,), 128, dtype=torch.int32, device="cuda"), cache=dc.c)
    rw = host_bits(rows)
    # Reuse: given uniform random distinct indices, attention only
    q = synth.torch_normal_bf16(520601, (B, 64, 512), "cuda")
    sel = synth.torch_distinct_indices(520602, B, T, 512, "cuda")
    out = torch.empty((B, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    ws = csa2.alloc_workspace(B, 64, T, False)
    csa2.sparse_attn_reuse(csa2.make_step(q=q, topk_idx=sel, out=out, lse=lse, **common), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    qh, selh, O, L = host_bits(q), sel.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    for r in (0, 101):
        kv_h, _ = oracle_request(orc, dc, r, T, selh[r])
        Oref, lref = orc.attention(qh[r], selh[r], kv_h, 0, rw[128 * r:128 * r + 128], 128, None, None, mp)
        assert attn_excess(O[r], Oref) <= TOL, r
        assert np.abs(L[r] - lref).max() <= 1e-2, r
    # Reindex: the shared packed keys rescored by a fresh indexer query
    q_idx = synth.torch_normal_bf16(520603, (B, 64, 128), "cuda")
    w = synth.torch_normal_f32(520604, (B, 64), "cuda")
    scores = torch.empty((B, T), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, 512), dtype=torch.int32, device="cuda")
    csa2.sparse_attn_reindex(csa2.make_step(q=q, q_idx=q_idx, w=w, heads_I=64, topk_idx=idx, out=out, lse=lse,
                                            scores=scores, ld=T, **common), ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    idxh, O, L = idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    qih, wh = host_bits(q_idx), w.cpu().numpy()
    for r in (3, 127):
        check_request(orc, csa2, dc, r, n_cached=T, nv=T, S_row=scores[r].cpu().numpy(), sel=idxh[r], q=qh[r],
                      q_idx=qih[r], w=wh[r], win_rows=rw[128 * r:128 * r + 128], O=O[r], L=L[r],
                      windows=[(0, 4096), (123 * PAGE, 123 * PAGE + 4096), (T - 4096, T)])


@pytest.mark.parametrize("group", [1, 2])
def test_chunked_prefill_4096_on_262144(orc, csa2, group):
    # one request: 262144 cached entries, 4096 new tokens packed by the step and queried
    # causally (query i sees entries 0 .. n0 + i); indexer groups of one query (the
    # benchmark's prefill line) and of two
    n0, n_new = 262144, 4096
    T = n0 + n_new
    mp = T // PAGE
    dc = DeviceCache(csa2, 1, mp, 550000)
    dc.fill(n0)
    new_lat = synth.torch_normal_bf16_rows_with_outliers(550500, n_new, 512, 0.0, 1.0, "cuda")
    new_key = synth.torch_normal_bf16_rows_with_outliers(550501, n_new, 128, 0.0, 1.0, "cuda")
    # window of query i: the 128 latents ending at its own position (bf16, unquantised)
    lat_c, _ = dc.draws(0, n0)
    rows = torch.cat([lat_c[n0 - 127:], new_lat]).contiguous()
    del lat_c
    win = dict(rows=rows, start=torch.arange(n_new, dtype=torch.int64, device="cuda"),
               len=torch.full((n_new,), 128, dtype=torch.int32, device="cuda"))
    new = dict(n=n_new, lat=new_lat, key=new_key, req=torch.zeros(n_new, dtype=torch.int32, device="cuda"),
               pos=torch.arange(n0, T, dtype=torch.int64, device="cuda"))
    nvis = torch.arange(n0 + 1, T + 1, dtype=torch.int32, device="cuda")
    res = _full_step(csa2, dc, 1, T, 550600, group=group, n_q=n_new, req=torch.zeros(n_new, dtype=torch.int32,
                     device="cuda"), nvis=nvis, win=win, new=new)
    idx = res["topk_idx"].cpu().numpy()
    q, q_idx, w = host_bits(res["q"]), host_bits(res["q_idx"]), res["w"].cpu().numpy()
    nl, nk, rw = host_bits(new_lat), host_bits(new_key), host_bits(rows)
    for i in (0, 1, 2047, 4095):
        nv = n0 + i + 1
        S_row = res["scores"][i].cpu().numpy()
        windows = [(0, 4096), (n0 - 2048, nv)]  # pages hold every new entry packed by the step
        O = res["out"][i].float().cpu().numpy()
        L = res["lse"][i].cpu().numpy()
        check_request(orc, csa2, dc, 0, n_cached=n0, nv=nv, S_row=S_row, sel=idx[i], q=q[i], q_idx=q_idx[i], w=w[i],
                      win_rows=rw[i:i + 128], O=O, L=L, windows=windows, new_lat=nl, new_key=nk,
                      new_pos=np.arange(n0, T))
