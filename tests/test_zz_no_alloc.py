"""csa2_topk_noalloc: the top-k for callers that cannot allocate device memory.

A serving engine that gives all of its device memory to a KV-cache pool at start-up, or
a host thread that must not stall on cudaMalloc/cudaFree (which can synchronise the
device), cannot hand the library a workspace.  This entry point keeps its scratch in a
fixed array inside the library instead.  Its result must equal the workspace version's
bit for bit (top-k is integer work), on two calls in a row since the calls share the
array.  This file is collected last on purpose."""
import ctypes

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
        assert torch.equal(got, ref), f"call {call}: rows differ {torch.nonzero((got != ref).any(1)).flatten()[:8]}"


def test_noalloc_topk_rejects_too_many_rows(csa2):
    st = csa2.lib.csa2_topk_noalloc(None, 0, None, 129, 10, 512, None, None)
    assert st == csa2.ERR_WORKSPACE
    assert b"128" in csa2.lib.csa2_last_error()
