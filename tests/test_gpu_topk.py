"""Top-k parity, bit-exact against the oracle on the same fp32 score rows: the 512
largest, equal scores by lower index, -0 == +0, ascending output, -1 padding
("DeepSeek's Attention and KV Cache", "DeepSeek-V3.2" top-k; "From MLA to DSA to
HCA/CSA", "CSA": -1 sentinel when fewer than k entries are visible)."""
import numpy as np
import pytest
import torch

from helpers import dev

pytestmark = pytest.mark.gpu


def _rows(seed, lens, t_max):
    g = np.random.default_rng(seed)
    S = g.standard_normal((len(lens), t_max)).astype(np.float32) * 5
    for r, n in enumerate(lens):
        if n > 20:
            S[r, g.integers(0, n, n // 10)] = S[r, 3]         # ties
            S[r, g.integers(0, n, 7)] = -0.0
            S[r, g.integers(0, n, 7)] = 0.0
    return S


def _check(orc, csa2, S, lens):
    n_q, t_max = S.shape
    ld = ((t_max + 3) // 4) * 4
    Sp = np.zeros((n_q, ld), np.float32)
    Sp[:, :t_max] = S
    out = torch.full((n_q, 512), -7, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(n_q, 64, t_max, False)
    csa2.topk(dev(Sp), ld, dev(np.array(lens, np.int32)), n_q, t_max, 512, out, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    got = out.cpu().numpy()
    for r, n in enumerate(lens):
        ref = orc.topk(S[r, :n], 512)
        assert np.array_equal(got[r], ref), (r, n, np.nonzero(got[r] != ref)[0][:8])


def test_topk_ragged_lengths(orc, csa2):
    lens = [0, 1, 5, 511, 512, 513, 4103, 40000, 70001]
    _check(orc, csa2, _rows(1, lens, max(lens)), lens)


def test_topk_many_rows_decode_shape(orc, csa2):
    lens = [16384] * 24
    _check(orc, csa2, _rows(2, lens, 16384), lens)


def test_topk_massive_ties_use_exact_refinement(orc, csa2):
    t = 20000
    S = np.zeros((4, t), np.float32)
    S[1] = 1.5                                   # every entry equal
    S[2, ::2] = -0.0                             # +0 / -0 mixture
    g = np.random.default_rng(3)
    S[3] = 2.0
    S[3, g.integers(0, t, 100)] = 3.0 + g.random(100).astype(np.float32)   # 100 above, 19900 tied below
    _check(orc, csa2, S, [t, t, t, t])


def test_topk_threshold_bin_crowded(orc, csa2):
    # many distinct values inside one 11-bit bin around the threshold
    g = np.random.default_rng(4)
    t = 50000
    S = (1.0 + g.random((2, t)) * 0.2).astype(np.float32)
    _check(orc, csa2, S, [t, 30000])


def test_topk_long_rows_block_bound(orc, csa2):
    # long rows select through the 32-entry block-maximum lower bound; one 1M-entry row
    lens = [131072, 131072, 262144, 1048576]
    _check(orc, csa2, _rows(5, lens, max(lens)), lens)


def test_topk_increasing_rows_overflow_to_whole_row(orc, csa2):
    # increasing scores make the block bound as loose as it gets (every entry of the last
    # 512 blocks is a candidate): the staged lists overflow and the leader selects over
    # the whole row; exact ties across blocks ride along
    t = 70000
    S = np.stack([np.arange(t, dtype=np.float32), np.repeat(np.arange(t // 40, dtype=np.float32), 40)[:t]])
    _check(orc, csa2, S, [t, t])
