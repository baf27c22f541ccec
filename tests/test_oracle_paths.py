"""Pins of the oracle's cache packing, index score, top-k and attention against
library routines (numpy dot / softmax), brute force on tiny inputs, special cases and
invariants stated on the pages:

* "DeepSeek's Attention and KV Cache - From MLA to CSA2": "DeepSeek-V3.2" (index score,
  top-k), "DeepSeek-V4" (512 selected + 128 window entries, shared-KV MQA),
  "DeepSeek-V4.1" (FP4 entries dequantised before attention).
* "From MLA to DSA to HCA/CSA": "The indexer" (ReLU makes each head's vote
  non-negative; selection is head-uniform), "CSA" (-1 sentinel), "What replaced MLA"
  (K and V are the same tensor)."""
import numpy as np
import pytest

import synth


def _softmax(x):
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def _cache(orc, n_req, n_entries, seed, max_pages=None, block_table=None, outliers=0.0):
    mp = max_pages or (n_entries + 127) // 128
    n_pages = n_req * mp if block_table is None else int(np.max(block_table)) + 1
    kv, ix = orc.alloc_pages(n_pages)
    lat = synth.normal_bf16_rows_with_outliers(seed, n_req * n_entries, 512, outliers, 8.0)
    key = synth.normal_bf16_rows_with_outliers(seed + 1, n_req * n_entries, 128, outliers, 8.0)
    req = np.repeat(np.arange(n_req), n_entries).astype(np.int32)
    pos = np.tile(np.arange(n_entries), n_req).astype(np.int64)
    orc.pack_kv(lat, key, req, pos, kv, ix, block_table, mp)
    return kv, ix, lat, key, mp


def test_pack_readback_equals_block_quantisation(orc):
    kv, ix, lat, key, mp = _cache(orc, 2, 300, 11)
    for (r, s) in [(0, 0), (0, 127), (0, 128), (1, 299), (1, 5)]:
        row = r * 300 + s
        c, sc = orc.quant_vector(synth.bf16_to_f32(lat[row]))
        assert np.array_equal(orc.read_main(kv, r, s, None, mp), orc.dequant_vector(c, sc))
        c, sc = orc.quant_vector(synth.bf16_to_f32(key[row]))
        assert np.array_equal(orc.read_idx(ix, r, s, None, mp), orc.dequant_vector(c, sc))


def test_page_layout_has_no_aliasing(orc):
    """Every entry of a full page reads back its own values (the layout is a bijection)."""
    kv, ix, lat, key, mp = _cache(orc, 1, 128, 12)
    assert ix.size == 128 * 72 and kv.size == 128 * 288
    for s in range(128):
        c, sc = orc.quant_vector(synth.bf16_to_f32(key[s]))
        assert np.array_equal(orc.read_idx(ix, 0, s, None, mp), orc.dequant_vector(c, sc))
        c, sc = orc.quant_vector(synth.bf16_to_f32(lat[s]))
        assert np.array_equal(orc.read_main(kv, 0, s, None, mp), orc.dequant_vector(c, sc))


def test_block_table_indirection(orc):
    bt = np.array([[3, 0], [1, 2]], np.int32)        # request 0 -> pages 3, 0 ; request 1 -> 1, 2
    kv, ix, lat, key, mp = _cache(orc, 2, 256, 13, max_pages=2, block_table=bt)
    kv2, ix2, _, _, _ = _cache(orc, 2, 256, 13, max_pages=2)
    for r in range(2):
        for s in (0, 100, 128, 255):
            assert np.array_equal(orc.read_main(kv, r, s, bt, 2), orc.read_main(kv2, r, s, None, 2))
            assert np.array_equal(orc.read_idx(ix, r, s, bt, 2), orc.read_idx(ix2, r, s, None, 2))


def _qhat(orc, q_bits):
    out = []
    for j in range(q_bits.shape[0]):
        c, sc = orc.quant_vector(synth.bf16_to_f32(q_bits[j]))
        out.append(orc.dequant_vector(c, sc))
    return np.array(out)


def test_index_score_one_head_is_relu_dot(orc):
    kv, ix, lat, key, mp = _cache(orc, 1, 200, 21)
    q = synth.normal_bf16(22, (1, 128))
    I, M = orc.index_score(q, np.ones(1, np.float32), ix, 0, 0, 200, None, mp)
    khat = np.array([orc.read_idx(ix, 0, s, None, mp) for s in range(200)])
    ref = np.maximum(khat @ _qhat(orc, q)[0] / np.sqrt(128.0), 0.0)
    assert np.allclose(I, ref, rtol=1e-13, atol=1e-13) and np.array_equal(I, M)


def test_index_score_linear_in_w_and_nonnegative_votes(orc):
    kv, ix, lat, key, mp = _cache(orc, 1, 150, 31)
    H = 8
    q = synth.normal_bf16(32, (H, 128))
    w = synth.normal_f32(33, H)
    I, M = orc.index_score(q, w, ix, 0, 0, 150, None, mp)
    per_head = []
    for j in range(H):
        e = np.zeros(H, np.float32); e[j] = 1.0
        Ij, Mj = orc.index_score(q, e, ix, 0, 0, 150, None, mp)
        assert (Ij >= 0).all()                 # each ReLU vote is non-negative
        per_head.append(Ij)
    per_head = np.array(per_head)
    assert np.allclose(I, w.astype(np.float64) @ per_head, rtol=1e-12, atol=1e-12)
    assert np.allclose(M, np.abs(w).astype(np.float64) @ per_head, rtol=1e-12, atol=1e-12)
    assert (np.abs(I) <= M + 1e-12).all()
    Ipos, Mpos = orc.index_score(q, np.abs(w), ix, 0, 0, 150, None, mp)
    assert (Ipos >= 0).all() and np.allclose(Ipos, Mpos)
    # head permutation leaves the score unchanged
    perm = np.random.default_rng(0).permutation(H)
    Ip, _ = orc.index_score(np.ascontiguousarray(q[perm]), np.ascontiguousarray(w[perm]), ix, 0, 0, 150, None, mp)
    assert np.allclose(Ip, I, rtol=1e-12, atol=1e-12)


def _brute_topk(s, k):
    s = np.where(s == 0, np.float32(0), s)
    order = sorted(range(len(s)), key=lambda i: (-float(s[i]), i))
    pick = sorted(order[:k])
    return np.array(pick + [-1] * (k - len(pick)), np.int32)


@pytest.mark.parametrize("n,k", [(0, 4), (3, 8), (8, 8), (50, 8), (1000, 16), (700, 512)])
def test_topk_brute_force(orc, n, k):
    g = np.random.default_rng(n * 7 + k)
    s = g.standard_normal(n).astype(np.float32)
    if n > 10:
        s[g.integers(0, n, n // 3)] = s[0]          # planted ties
        s[g.integers(0, n, 5)] = -0.0
        s[g.integers(0, n, 5)] = 0.0
    got = orc.topk(s, k)
    assert np.array_equal(got, _brute_topk(s, k))


def test_topk_ties_take_lowest_index(orc):
    s = np.zeros(100, np.float32)
    s[::2] = -0.0
    assert np.array_equal(orc.topk(s, 10), np.arange(10))
    s = np.ones(20, np.float32); s[15] = 2.0
    assert np.array_equal(orc.topk(s, 3), [0, 1, 15])


def test_attention_dense_when_k_covers_everything(orc):
    T, H, W = 40, 4, 6
    kv, ix, lat, key, mp = _cache(orc, 1, T, 41)
    q = synth.normal_bf16(42, (H, 512))
    win = synth.normal_bf16(43, (W, 512))
    idx = np.concatenate([np.random.default_rng(1).permutation(T), -np.ones(8, int)]).astype(np.int32)
    O, lse = orc.attention(q, idx, kv, 0, win, W, None, None, mp)
    keys = np.concatenate([np.array([orc.read_main(kv, 0, s, None, mp) for s in range(T)]),
                           synth.bf16_to_f32(win).astype(np.float64)])
    S = synth.bf16_to_f32(q).astype(np.float64) @ keys.T / np.sqrt(512.0)
    P = _softmax(S)
    assert np.allclose(O, P @ keys, rtol=1e-10, atol=1e-12)
    ref_lse = S.max(1) + np.log(np.exp(S - S.max(1, keepdims=True)).sum(1))
    assert np.allclose(lse, ref_lse, rtol=1e-12)


def test_attention_special_cases(orc):
    kv, ix, lat, key, mp = _cache(orc, 1, 64, 51)
    q = synth.normal_bf16(52, (3, 512))
    win = synth.normal_bf16(53, (4, 512))
    one = np.array([17, -1, -1], np.int32)
    O, lse = orc.attention(q, one, kv, 0, win, 0, None, None, mp)
    k17 = orc.read_main(kv, 0, 17, None, mp)
    assert np.array_equal(O, np.tile(k17, (3, 1)))       # a single key is returned exactly
    assert np.allclose(lse, synth.bf16_to_f32(q).astype(np.float64) @ k17 / np.sqrt(512))
    O, lse = orc.attention(q, np.full(4, -1, np.int32), kv, 0, win, 0, None, None, mp)
    assert not O.any() and np.isneginf(lse).all()        # no keys at all
    idx = np.array([5, 9, 30, 2], np.int32)
    O1, l1 = orc.attention(q, idx, kv, 0, win, 4, None, None, mp)
    O2, l2 = orc.attention(q, idx[::-1].copy(), kv, 0, win, 4, None, None, mp)
    assert np.allclose(O1, O2, rtol=1e-12, atol=1e-14) and np.allclose(l1, l2)
    # duplicate (window overlaps selection): counted twice, no de-duplication
    O3, _ = orc.attention(q, np.array([5, 5], np.int32), kv, 0, win, 0, None, None, mp)
    assert np.allclose(O3, np.tile(orc.read_main(kv, 0, 5, None, mp), (3, 1)))


def test_index_score_bf16_one_head_and_linearity(orc):
    """The bf16 reference score ("DeepSeek-V3.2", the lightning indexer; "From MLA to DSA to
    HCA/CSA", "CSA" scorer: ReLU of the scaled query-key product, weighted per head and
    summed) with one head of weight 1 is ReLU(q . k) / sqrt(128) of the unquantised bf16
    values, computed here with numpy; the full score is then linear in w (which, with the
    one-head case, fixes every head's term).  A dropped ReLU, a missing 128^-1/2, a
    transposed operand or a quantised input fails one of these."""
    T, H = 300, 6
    keys = synth.normal_bf16(901, (T, 128))
    q = synth.normal_bf16(902, (H, 128))
    kf = synth.bf16_to_f32(keys).astype(np.float64)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    terms = np.maximum(kf @ qf.T / np.sqrt(128.0), 0.0)          # [T][H] per-head votes
    assert (terms == 0).any() and (terms > 0).any()              # ReLU active on both sides
    for j in range(H):
        Ij = orc.index_score_bf16(np.ascontiguousarray(q[j:j + 1]), np.ones(1, np.float32), keys)
        assert np.allclose(Ij, terms[:, j], rtol=1e-13, atol=1e-13)
    w = synth.normal_f32(903, (H,))
    I = orc.index_score_bf16(q, w, keys)
    assert np.allclose(I, terms @ w.astype(np.float64), rtol=1e-12, atol=1e-12)
    # the unquantised score differs from the FP4 one (the inputs are not quantised here)
    kv, ix = orc.alloc_pages(3)
    orc.pack_kv(synth.normal_bf16(904, (T, 512)), keys, np.zeros(T, np.int32), np.arange(T, dtype=np.int64), kv, ix,
                None, 3)
    I4, _ = orc.index_score(q, w, ix, 0, 0, T, None, 3)
    assert not np.allclose(I4, I, rtol=1e-6, atol=1e-6)


def test_fp4_selection_recall_against_bf16_scores(orc):
    """Recall of the top-512 chosen on FP4 query and key against the top-512 of the bf16
    score ("DeepSeek-V4": 99.7 % for V4's trained indexer).  On synthetic N(0,1) data the
    figure is model-free and only reported; it must be far above chance (512 / T)."""
    import synth
    T = 6144
    keys = synth.normal_bf16(880, (T, 128))
    kv, ix = orc.alloc_pages((T + 127) // 128)
    orc.pack_kv(synth.normal_bf16(881, (T, 512)), keys, np.zeros(T, np.int32), np.arange(T, dtype=np.int64), kv, ix,
                None, (T + 127) // 128)
    rec = []
    for t in range(3):
        q = synth.normal_bf16(882 + t, (64, 128))
        w = np.abs(synth.normal_f32(890 + t, (64,)))   # non-negative head weights, as in a trained indexer's
        I4, _ = orc.index_score(q, w, ix, 0, 0, T, None, (T + 127) // 128)
        Ib = orc.index_score_bf16(q, w, keys)
        a = set(orc.topk(I4.astype(np.float32), 512).tolist())
        b = set(orc.topk(Ib.astype(np.float32), 512).tolist())
        rec.append(len(a & b) / 512)
    print(f"FP4 top-512 recall of the bf16 top-512 (synthetic N(0,1)): {np.round(rec, 3).tolist()}")
    assert min(rec) > 5 * 512 / T
