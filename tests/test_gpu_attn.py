"""Sparse + window MQA parity (Reuse mode, given indices): bf16 output within 2e-2
max-abs of the fp64 oracle beyond the bf16 rounding of the exact output (half an ulp of
it; "DeepSeek's Attention and KV Cache", "DeepSeek-V4": 512
selected entries concatenated with the 128 window entries, one shared vector as key and
value; "From MLA to DSA to HCA/CSA", "What replaced MLA": K and V are the same tensor)."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache
from test_gpu_fullsize import attn_excess

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _reuse(orc, csa2, n_entries, idx, req_q, win_len, seed, qscale=1.0, win_rows=None, sinks=None, rope=None,
           win_start=None, outliers=0.0):
    n_req = len(n_entries)
    max_pages = (max(n_entries) + 127) // 128
    cache = Cache(n_req, max_pages)
    lat, key, req_e, pos_e = fill_cache(cache, n_entries, seed, outlier_frac=outliers)
    kv_h, ix_h = orc.alloc_pages(cache.n_pages)
    orc.pack_kv(lat, key, req_e, pos_e, kv_h, ix_h, None, max_pages)
    n_q = len(req_q)
    q = synth.normal_bf16(seed + 3, (n_q, 64, 512), scale=qscale)
    nwin = win_rows or 128 * n_q
    window = synth.normal_bf16(seed + 4, (nwin, 512))
    if win_start is None:
        win_start = [128 * i if win_rows is None else i for i in range(n_q)]
    win_start = np.array(win_start, np.int64)
    win_len = np.array(win_len, np.int32)
    nvis = np.array([n_entries[r] for r in req_q], np.int32)
    out = torch.zeros((n_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((n_q, 64), dtype=torch.float32, device="cuda")
    topk_idx = dev(np.ascontiguousarray(idx, np.int32))
    extra = {}
    if sinks is not None:
        extra["sinks"] = dev(np.ascontiguousarray(sinks, np.float32))
    if rope is not None:
        extra["rope_cos"] = dev(np.ascontiguousarray(np.cos(rope), np.float32))
        extra["rope_sin"] = dev(np.ascontiguousarray(np.sin(rope), np.float32))
    step = csa2.make_step(n_q=n_q, t_max=int(max(n_entries)), q=dev_bf16(q), req=dev(np.array(req_q, np.int32)),
                          n_visible=dev(nvis), window=dev_bf16(window), win_start=dev(win_start),
                          win_len=dev(win_len), cache=cache.c, topk_idx=topk_idx, out=out, lse=lse, **extra)
    ws = csa2.alloc_workspace(n_q, 64, int(max(n_entries)), False)
    csa2.sparse_attn_reuse(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    O = out.float().cpu().numpy()
    L = lse.cpu().numpy()
    for i in range(n_q):
        ws_ = int(win_start[i])
        if sinks is None and rope is None:
            Oref, lref = orc.attention(q[i], idx[i], kv_h, int(req_q[i]), window[ws_:ws_ + max(1, win_len[i])],
                                       int(win_len[i]), None, None, max_pages)
        else:
            # the oracle takes the angles the kernel saw (fp32), in fp64
            rc = None if rope is None else np.cos(rope[i]).astype(np.float32)
            rs = None if rope is None else np.sin(rope[i]).astype(np.float32)
            Oref, lref = orc.attention_ext(q[i], idx[i], kv_h, int(req_q[i]),
                                           window[ws_:ws_ + max(1, win_len[i])], int(win_len[i]), None,
                                           None if sinks is None else np.asarray(sinks, np.float32),
                                           rc, rs, None, max_pages)
        err = attn_excess(O[i], Oref)
        assert err <= TOL, (i, err)
        fin = np.isfinite(lref)
        assert np.array_equal(fin, np.isfinite(L[i]))
        if fin.any():  # a query with no key at all has lse = -inf in every head
            assert np.abs(L[i][fin] - lref[fin]).max() <= 1e-2
    return O


def test_attn_reuse_random_indices(orc, csa2):
    n = [2000, 900]
    idx = np.stack([synth.distinct_indices(1, 2000, 512), synth.distinct_indices(2, 900, 512)])
    _reuse(orc, csa2, n, idx, [0, 1], [128, 128], seed=50)


def test_attn_padding_window_lengths_and_duplicates(orc, csa2):
    n = [700, 300]
    a = synth.distinct_indices(3, 300, 512)          # 300 valid + 212 x -1
    b = np.full(512, -1, np.int32)                   # window only
    c = synth.distinct_indices(4, 700, 512)
    c[:64] = c[64:128]                               # duplicates are attended twice
    d = np.full(512, -1, np.int32)
    d[:3] = [5, 6, 699]
    idx = np.stack([a, b, c, d])
    _reuse(orc, csa2, n, idx, [1, 0, 0, 0], [128, 57, 1, 0], seed=51)


def test_attn_peaky_queries(orc, csa2):
    """Q x 8 makes the softmax peaky, so the 2e-2 bound is a real constraint."""
    n = [1500]
    idx = np.stack([synth.distinct_indices(5, 1500, 512), synth.distinct_indices(6, 1500, 512)])
    _reuse(orc, csa2, n, idx, [0, 0], [128, 100], seed=52, qscale=8.0)


def test_attn_shared_window_rows_prefill_style(orc, csa2):
    """Consecutive queries share a window buffer with shifted starts (chunked prefill)."""
    n = [1200]
    n_q = 3
    idx = np.stack([synth.distinct_indices(10 + i, 1200, 512) for i in range(n_q)])
    _reuse(orc, csa2, n, idx, [0] * n_q, [128, 128, 128], seed=53, win_rows=130)


@pytest.mark.parametrize("n_q", [3, 45, 64, 80])
def test_attn_sinks_and_partial_rope(orc, csa2, n_q):
    """Per-head sinks join the softmax; the query's trailing 64 channels are rotated at
    its position and the output rotated back ("From MLA to DSA to HCA/CSA", "The sliding
    window" and "What replaced MLA").  On 152 SMs: 3 queries take 5 CTAs each and 45 take
    3 (every CTA combines a slice of the heads), 64 take a pair (the second CTA adds the
    first one's partial, sinks and rotation in its epilogue), 80 one CTA each."""
    n = [1800]
    idx = np.stack([synth.distinct_indices(20 + i, 1800, 512) for i in range(n_q)])
    idx[-1, 100:] = -1                   # a short selection
    sinks = 2.0 * synth.normal_f32(21, (64,))
    sinks[:4] = [-30.0, 0.0, 8.0, 30.0]  # negligible, even, dominant, overwhelming
    rope = synth.rng(22).uniform(-np.pi, np.pi, (n_q, 32))
    wl = [[128, 77, 0][i % 3] for i in range(n_q)]
    _reuse(orc, csa2, n, idx, [0] * n_q, wl, seed=54, qscale=2.0, sinks=sinks, rope=rope)


@pytest.mark.parametrize("n_q", [2, 90])
def test_attn_outlier_entries_peaky(orc, csa2, n_q):
    """5 % of the entries x 8 (large E4M3 block scales) and peaky queries (Q x 8): outputs
    reach |O| of several units, where the bf16 output rounding itself is a visible part
    of the error; the bound stays 2e-2 beyond half an ulp of the exact output."""
    n = [3000]
    idx = np.stack([synth.distinct_indices(90 + i, 3000, 512) for i in range(n_q)])
    _reuse(orc, csa2, n, idx, [0] * n_q, [128] * n_q, seed=59, qscale=8.0, outliers=0.05)


def test_attn_rope_only_and_sinks_only(orc, csa2):
    n = [900]
    idx = np.stack([synth.distinct_indices(23, 900, 512), synth.distinct_indices(24, 900, 512)])
    rope = synth.rng(25).uniform(-np.pi, np.pi, (2, 32))
    _reuse(orc, csa2, n, idx, [0, 0], [128, 128], seed=55, qscale=4.0, rope=rope)
    _reuse(orc, csa2, n, idx, [0, 0], [128, 3], seed=56, sinks=synth.normal_f32(26, (64,)))


def test_attn_bounded_replay_window(orc, csa2):
    """SWA bounded replay ("DeepSeek-V4.1", bounded replay): a replay from position s
    lets the query at i see the local keys [max(s, i - 127), i]; the window rows of a
    chunk are one buffer and each query's start and length follow that rule."""
    n = [1000]
    s0, base = 40, 0                          # replay starts at position 40 of the window buffer
    pos = [40, 41, 100, 167, 168, 300]        # query positions (buffer rows)
    starts = [max(s0, i - 127) for i in pos]
    lens = [i - st + 1 for i, st in zip(pos, starts)]
    assert lens == [1, 2, 61, 128, 128, 128]
    idx = np.stack([synth.distinct_indices(30 + i, 1000, 512) for i in range(len(pos))])
    _reuse(orc, csa2, n, idx, [0] * len(pos), lens, seed=57, win_rows=301 + base, win_start=starts)


@pytest.mark.parametrize("n_q", [3, 34, 45, 60, 80])
def test_attn_key_tile_splits(orc, csa2, n_q):
    """Batches smaller than the SM count split each query's key tiles over a cluster of CTAs
    that merge their partial outputs by their maxima and sums of exponentials (partials in
    the workspace, one cluster barrier); on 152 SMs these batch sizes take 5, 4, 3, 2 and 1
    CTAs per query.  Rows
    mix full selections, short selections (empty tiles in some splits), window-only rows
    and rows with no key at all."""
    n = [700, 300]
    pats = []
    for i in range(n_q):
        k = i % 5
        if k == 0:
            pats.append(synth.distinct_indices(60 + i, 700, 512))
        elif k == 1:
            pats.append(synth.distinct_indices(60 + i, 300, 512))      # 300 valid, then -1
        elif k == 2:
            pats.append(np.full(512, -1, np.int32))                    # window only
        elif k == 3:
            a = np.full(512, -1, np.int32)
            a[:3] = [0, 299, 150]
            pats.append(a)
        else:
            a = synth.distinct_indices(60 + i, 700, 512)
            a[300:] = -1                                               # the last two tiles empty
            pats.append(a)
    req = [0 if i % 5 in (0, 4) else 1 for i in range(n_q)]
    win = [[128, 57, 0, 128, 1][i % 5] if i % 7 else 0 for i in range(n_q)]
    win[2] = 0                                                         # a row with no key at all
    _reuse(orc, csa2, n, np.stack(pats), req, win, seed=58 + n_q)
