"""csa2_topk_noalloc: the top-k for callers that cannot allocate device memory.

A serving engine that gives all of its device memory to a KV-cache pool at start-up, or
a host thread that must not stall on cudaMalloc/cudaFree (which can synchronise the
device), cannot hand the library a workspace.  This entry point keeps its scratch in a
fixed array inside the library instead.  Its result must equal the workspace version's
bit for bit (top-k is integer work), on two calls in a row since the calls share the
array, and equal the oracle's top-k ("DeepSeek-V3.2" top-k, "DeepSeek-V4.1" k = 512;
"CSA: two changes to HCA" -1 sentinel) on rows that reach each branch of its own
three-kernel path: fewer than k visible entries (identity and -1 padding, empty rows,
negative counts clamped to 0), a threshold bin small enough for the rank selection, one
that needs the bitonic sort, one that overflows the candidate buffer (exact radix
refinement over the row: all-equal rows, thousands of distinct values in one bin, a
mixture of +0 and -0).  The array's error word is read back after every call.  This
file is collected last on purpose."""
import numpy as np
import pytest
import torch

from helpers import dev

pytestmark = pytest.mark.gpu


def _scores(seed, n_q, t):
    g = np.random.default_rng(seed)
    S = (g.standard_normal((n_q, t)) * 5).astype(np.float32)
    S[:, ::97] = S[:, :1]          # ties across the row
    S[0, :] = 1.0                  # one row of identical scores
    return S


def test_noalloc_topk_matches_workspace_topk_twice(csa2):
    t = 20000
    ld = t
    for call, (seed, n_q) in enumerate([(1, 96), (2, 128)]):
        S = dev(_scores(seed, n_q, t))
        nvis = dev(np.array([t - (i * 37) % 900 for i in range(n_q)], np.int32))
        ref = torch.full((n_q, 512), -7, dtype=torch.int32, device="cuda")
        got = torch.full((n_q, 512), -9, dtype=torch.int32, device="cuda")
        ws = csa2.alloc_workspace(n_q, 64, t, False)
        csa2.topk(S, ld, nvis, n_q, t, 512, ref, ws)
        csa2.topk_noalloc(S, ld, nvis, n_q, t, 512, got)
        torch.cuda.synchronize()
        assert csa2.check(ws) == (csa2.OK, 0)
        assert csa2.topk_noalloc_check() == (csa2.OK, 0)
        assert torch.equal(got, ref), f"call {call}: rows differ {torch.nonzero((got != ref).any(1)).flatten()[:8]}"


def _special_rows(t):
    """Rows aimed at the branches of the three-kernel path, with their visible counts."""
    g = np.random.default_rng(11)
    rows, nvis = [], []

    def add(row, nv):
        rows.append(np.asarray(row, np.float32))
        nvis.append(nv)

    base = g.standard_normal(t).astype(np.float32)
    add(base, 0)                                    # empty row: all -1
    add(base, -5)                                   # negative count: clamped to 0
    add(base, 300)                                  # fewer than k: identity then -1
    add(base, 512)                                  # exactly k
    add(base, 513)                                  # one more than k
    add(np.ones(t), t)                              # all equal: threshold bin overflows
    r = -np.abs(g.standard_normal(t)).astype(np.float32) - 1.0
    r[g.choice(t, 300, replace=False)] = 3.0 + g.random(300).astype(np.float32)
    z = g.choice(np.setdiff1d(np.arange(t), np.nonzero(r > 0)[0]), 900, replace=False)
    r[z] = np.where(g.random(900) < 0.5, np.float32(0.0), np.float32(-0.0))
    add(r, t)                                       # +0 / -0 ties in a small threshold bin (rank path)
    r = -np.abs(g.standard_normal(t)).astype(np.float32) - 1.0
    r[g.choice(t, 200, replace=False)] = 4.0
    r[g.choice(np.nonzero(r < 0)[0], 2500, replace=False)] = 1.0 + 0.25 * g.random(2500).astype(np.float32)
    add(r, t)                                       # 2,500 candidates in one bin (bitonic path)
    r = 1.0 + 0.25 * g.random(t).astype(np.float32)
    add(r, t)                                       # every entry in one bin, distinct values (refinement)
    r = np.where(g.random(t) < 0.5, np.float32(0.0), np.float32(-0.0))
    r[g.choice(t, 100, replace=False)] = -1.0
    add(r, t)                                       # +0 / -0 everywhere (refinement over signed zeros)
    add(g.standard_normal(t).astype(np.float32), t - 3)
    return np.stack(rows), np.array(nvis, np.int32)


def test_noalloc_topk_special_rows_against_oracle(orc, csa2):
    t = 20000
    S_h, nv_h = _special_rows(t)
    n_q = S_h.shape[0]
    S = dev(S_h)
    nvis = dev(nv_h)
    ws = csa2.alloc_workspace(n_q, 64, t, False)
    for call in range(2):
        ref = torch.full((n_q, 512), -7, dtype=torch.int32, device="cuda")
        got = torch.full((n_q, 512), -9, dtype=torch.int32, device="cuda")
        csa2.topk(S, t, nvis, n_q, t, 512, ref, ws)
        csa2.topk_noalloc(S, t, nvis, n_q, t, 512, got)
        torch.cuda.synchronize()
        assert csa2.topk_noalloc_check() == (csa2.OK, 0)
        assert csa2.check(ws) == (csa2.OK, 0)
        g_h, r_h = got.cpu().numpy(), ref.cpu().numpy()
        for i in range(n_q):
            want = orc.topk(S_h[i, :max(0, int(nv_h[i]))], 512)
            assert np.array_equal(g_h[i], want), f"call {call} row {i}: noalloc differs from the oracle"
            assert np.array_equal(r_h[i], want), f"call {call} row {i}: workspace top-k differs from the oracle"


def test_noalloc_topk_rejects_too_many_rows(csa2):
    st = csa2.lib.csa2_topk_noalloc(None, 0, None, 129, 10, 512, None, None)
    assert st == csa2.ERR_WORKSPACE
    assert b"128" in csa2.lib.csa2_last_error()
