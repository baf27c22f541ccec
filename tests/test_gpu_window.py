"""FP8 window ring through the C ABI ("DeepSeek's Attention and KV Cache - From MLA to
CSA2": "Four bits for the main KV, eight for the window" - 512 E4M3 bytes plus 16 E8M0
scales per entry; "Definition and the bounded cache" - position i in slot i mod 128):
csa2_pack_window is bit-exact against the oracle, and attention whose window keys come
from the ring matches the fp64 oracle within 2e-2 max-abs."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache, host_bits

pytestmark = pytest.mark.gpu
TOL = 2e-2
D = 512


def _rows(seed, n):
    rows = synth.normal_bf16(seed, (n, D), scale=2.0)
    rows[0, :32] = 0                                              # an all-zero block
    big = synth.normal_bf16(seed + 1, (n, D), scale=64.0)         # mixed magnitudes per block
    rows[1::3, 64:96] = big[1::3, 64:96]
    tiny = synth.normal_bf16(seed + 2, (n, D), scale=1e-30)
    rows[2::5, 128:160] = tiny[2::5, 128:160]
    return rows


def test_pack_window_bit_exact(orc, csa2):
    n_ring = 3
    ring = torch.zeros(n_ring * 128 * 528, dtype=torch.uint8, device="cuda")
    ring_h = orc.alloc_ring(n_ring)
    ws = csa2.alloc_workspace(1, 64, 128, False)
    for call, (n, p0) in enumerate([(130, 0), (97, 130), (40, 1000)]):  # positions wrap the ring
        rows = _rows(800 + call, n)
        req = (np.arange(n) % n_ring).astype(np.int32)
        pos = (p0 + np.arange(n) // n_ring).astype(np.int64)
        # one call must not write a slot twice
        assert len({(int(r), int(p) % 128) for r, p in zip(req, pos)}) == n
        csa2.pack_window(dev_bf16(rows), dev(req), dev(pos), ring, n_ring, ws)
        orc.pack_window(rows, req, pos, ring_h)
        assert csa2.check(ws) == (csa2.OK, 0)
        got = ring.cpu().numpy()
        assert np.array_equal(got, ring_h), np.flatnonzero(got != ring_h)[:10]


def test_pack_window_rejects_bad_request(csa2):
    ring = torch.zeros(2 * 128 * 528, dtype=torch.uint8, device="cuda")
    ws = csa2.alloc_workspace(1, 64, 128, False)
    rows = dev_bf16(synth.normal_bf16(810, (1, D)))
    csa2.pack_window(rows, dev(np.array([2], np.int32)), dev(np.array([0], np.int64)), ring, 2, ws)
    st, info = csa2.check(ws)
    assert st == csa2.ERR_DEVICE
    assert int(ring.sum().item()) == 0


def _attn_ring(orc, csa2, n_entries, idx, newest, win_len, seed, sinks=None, qscale=1.0):
    """One query per request; request r's ring holds its window entries of positions
    0 .. newest[r] (the query's own position is the newest)."""
    n_req = len(n_entries)
    assert len(newest) == n_req
    max_pages = (max(n_entries) + 127) // 128
    cache = Cache(n_req, max_pages)
    lat, key, req_e, pos_e = fill_cache(cache, n_entries, seed)
    kv_h, ix_h = orc.alloc_pages(cache.n_pages)
    orc.pack_kv(lat, key, req_e, pos_e, kv_h, ix_h, None, max_pages)
    # window entries of positions 0 .. newest[r] of request r, packed in order
    req_w = np.concatenate([np.full(int(t) + 1, r) for r, t in enumerate(newest)]).astype(np.int32)
    pos_w = np.concatenate([np.arange(int(t) + 1) for t in newest]).astype(np.int64)
    rows = synth.normal_bf16(seed + 7, (req_w.size, D))
    top = int(max(newest)) + 1
    ring = torch.zeros(n_req * 128 * 528, dtype=torch.uint8, device="cuda")
    ring_h = orc.alloc_ring(n_req)
    ws = csa2.alloc_workspace(len(newest), 64, int(max(n_entries)), False)
    for p in range(0, top, 128):  # a call never writes one slot twice
        sel = (pos_w >= p) & (pos_w < p + 128)
        csa2.pack_window(dev_bf16(np.ascontiguousarray(rows[sel])), dev(req_w[sel]), dev(pos_w[sel]), ring, n_req, ws)
        orc.pack_window(np.ascontiguousarray(rows[sel]), req_w[sel], pos_w[sel], ring_h)
    assert np.array_equal(ring.cpu().numpy(), ring_h)
    n_q = len(newest)
    req_q = np.arange(n_q, dtype=np.int32)
    q = synth.normal_bf16(seed + 3, (n_q, 64, D), scale=qscale)
    out = torch.zeros((n_q, 64, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((n_q, 64), dtype=torch.float32, device="cuda")
    extra = {} if sinks is None else {"sinks": dev(np.asarray(sinks, np.float32))}
    step = csa2.make_step(n_q=n_q, t_max=int(max(n_entries)), q=dev_bf16(q), req=dev(req_q),
                          n_visible=dev(np.array([n_entries[r] for r in req_q], np.int32)), window=None,
                          win_start=dev(np.array(newest, np.int64)), win_len=dev(np.array(win_len, np.int32)),
                          cache=cache.c, topk_idx=dev(np.ascontiguousarray(idx, np.int32)), out=out, lse=lse,
                          win_ring=ring, win_ring_reqs=n_req, **extra)
    csa2.sparse_attn_reuse(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    O = out.float().cpu().numpy()
    L = lse.cpu().numpy()
    for i in range(n_q):
        Oref, lref = orc.attention_ring(q[i], idx[i], kv_h, int(req_q[i]), ring_h, int(newest[i]), int(win_len[i]),
                                        None, None if sinks is None else np.asarray(sinks, np.float32), None, None,
                                        None, max_pages)
        err = np.abs(O[i] - Oref).max()
        assert err <= TOL, (i, err)
        fin = np.isfinite(lref)
        assert np.array_equal(fin, np.isfinite(L[i]))
        assert np.abs(L[i][fin] - lref[fin]).max() <= 1e-2


def test_attention_with_ring_window(orc, csa2):
    n = [1500, 700, 1200, 600]
    idx = np.stack([synth.distinct_indices(40 + i, n[i], 512) for i in range(4)])
    idx[3, 100:] = -1
    # newest positions past the ring's wrap; a short (bounded-replay) window; an empty one
    _attn_ring(orc, csa2, n, idx, newest=[300, 299, 127, 40], win_len=[128, 128, 31, 0], seed=58)


def test_attention_with_ring_window_peaky_and_sinks(orc, csa2):
    n = [900, 800]
    idx = np.stack([synth.distinct_indices(44 + i, n[i], 512) for i in range(2)])
    _attn_ring(orc, csa2, n, idx, newest=[513, 140], win_len=[128, 100], seed=59, qscale=6.0,
               sinks=synth.normal_f32(45, (64,)))


def test_attention_with_ring_window_key_split_pairs(orc, csa2):
    """64 queries: on 152 SMs each query takes a pair of CTAs, the first with the ring
    window, the second adding the first one's partial to its own."""
    n_q = 64
    n = [600 + 7 * i for i in range(n_q)]
    idx = np.stack([synth.distinct_indices(200 + i, n[i], 512) for i in range(n_q)])
    idx[5, 200:] = -1
    newest = [130 + 3 * i for i in range(n_q)]
    win_len = [128 if i % 9 else 77 for i in range(n_q)]
    _attn_ring(orc, csa2, n, idx, newest=newest, win_len=win_len, seed=60, sinks=synth.normal_f32(46, (64,)))
