"""Index-score parity: |gpu - oracle| <= 1e-3 * M where M = sum_j |w_j| ReLU(...), the
sum of the absolute head terms ("DeepSeek's Attention and KV Cache", "DeepSeek-V3.2"
index score; "From MLA to DSA to HCA/CSA", "The indexer" / "CSA" scorer code).  FP4 x FP4
products are exact in fp32, so the difference is the fp32 accumulation order only;
1e-3 relative to M bounds it with a wide margin."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


def _run(orc, csa2, n_entries, heads_I, group, seed, qscale=1.0, outliers=0.0, shuffled=False):
    n_req = len(n_entries)
    max_pages = (max(n_entries) + 127) // 128
    bt = None
    if shuffled:  # every request's pages scattered over the whole cache
        bt = np.random.default_rng(seed).permutation(n_req * max_pages).astype(np.int32).reshape(n_req, max_pages)
    cache = Cache(n_req, max_pages, block_table=bt)
    lat, key, req_e, pos_e = fill_cache(cache, n_entries, seed, outliers)
    kv_h, ix_h = orc.alloc_pages(cache.n_pages)
    orc.pack_kv(lat, key, req_e, pos_e, kv_h, ix_h, bt, max_pages)
    # queries: `group` consecutive queries per request, visibility shrinking by one
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
        I, M = orc.index_score(q_idx[q], w[q], ix_h, int(req_q[q]), 0, nv, bt, max_pages)
        err = np.abs(g[q, :nv].astype(np.float64) - I)
        bad = np.nonzero(err > 1e-3 * M)[0]
        assert bad.size == 0, (q, bad[:5], g[q, bad[:5]], I[bad[:5]], M[bad[:5]])
        assert np.isnan(g[q, nv:]).all(), "entries beyond the visible prefix must not be written"
    return g


@pytest.mark.parametrize("heads_I,group", [(64, 1), (32, 1), (64, 2), (32, 2)])
def test_index_scores_ragged(orc, csa2, heads_I, group):
    _run(orc, csa2, [1000, 333, 129], heads_I, group, seed=10 + heads_I + group)


def test_index_scores_outliers_and_single_tile(orc, csa2):
    _run(orc, csa2, [5, 128, 257], 64, 1, seed=31, outliers=0.02)


def test_index_scores_peaky_query(orc, csa2):
    _run(orc, csa2, [700], 64, 1, seed=41, qscale=8.0)


@pytest.mark.parametrize("heads_I,group,shuffled", [(64, 1, False), (32, 1, True), (64, 2, True), (32, 2, False)])
def test_index_scores_many_tiles_per_cta(orc, csa2, heads_I, group, shuffled):
    """40 requests of 2,000-12,000 entries: every persistent CTA runs about 14 tiles across
    group boundaries, so the accumulator rotation, the per-issuer scale slots and the
    query-slot switches at short segments all turn over several times (tile counts per
    group mostly not multiples of the three issuers / six accumulators)."""
    rng = np.random.default_rng(70 + heads_I + group)
    n_entries = [int(x) for x in rng.integers(2000, 12001, size=40)]
    _run(orc, csa2, n_entries, heads_I, group, seed=71 + heads_I + group, shuffled=shuffled)
