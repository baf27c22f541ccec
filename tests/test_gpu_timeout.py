"""The device-side failure path: every pipeline wait of the indexer and attention kernels is
bounded, and a wait that runs out records CSA2_ERR_TIMEOUT (info 5) in the workspace error
word, after which the kernel waits (with its fixed bound) for the copies and MMAs it has in
flight, frees its tensor memory and returns, so that the context stays usable.  The test
shortens the bound with csa2_debug_set_wait_limit so that waits of a real Full step run out
(no fault, trap or endless loop is involved: nothing is wrong with the inputs), checks the
reported status, then restores the default and checks that the next identical step is
green and reproduces the outputs of a step run before, bit for bit."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


def _step(csa2, cache, B, T, seed):
    q = synth.normal_bf16(seed, (B, 64, 512))
    q_idx = synth.normal_bf16(seed + 1, (B, 64, 128))
    w = synth.normal_f32(seed + 2, (B, 64))
    win = synth.normal_bf16(seed + 3, (128 * B, 512))
    new_lat = synth.normal_bf16(seed + 4, (B, 512))
    new_key = synth.normal_bf16(seed + 5, (B, 128))
    out = torch.zeros((B, 64, 512), dtype=torch.bfloat16, device="cuda")
    topk_idx = torch.zeros((B, 512), dtype=torch.int32, device="cuda")
    step = csa2.make_step(n_q=B, t_max=T, q=dev_bf16(q), req=dev(np.arange(B, dtype=np.int32)),
                          n_visible=dev(np.full(B, T, np.int32)), window=dev_bf16(win),
                          win_start=dev(np.arange(B, dtype=np.int64) * 128), win_len=dev(np.full(B, 128, np.int32)),
                          cache=cache.c, topk_idx=topk_idx, out=out, q_idx=dev_bf16(q_idx), w=dev(w), n_new=B,
                          new_latent=dev_bf16(new_lat), new_idx_key=dev_bf16(new_key),
                          new_req=dev(np.arange(B, dtype=np.int32)), new_pos=dev(np.full(B, T - 1, np.int64)))
    return step, out, topk_idx


@pytest.mark.parametrize("B", [2, 100])   # attention with cluster-merged key splits, and one CTA per query
def test_wait_timeout_is_reported_and_the_next_call_is_green(csa2, B):
    T = 4096
    cache = Cache(n_req=B, max_pages=T // 128)
    fill_cache(cache, [T - 1] * B, seed=700)
    step, out, topk_idx = _step(csa2, cache, B, T, seed=710)
    ws = csa2.alloc_workspace(B, 64, T, True)
    csa2.sparse_attn_full(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    o_ref, idx_ref = out.clone(), topk_idx.clone()
    try:
        csa2.debug_set_wait_limit(100)          # 100 ns: real copies and MMAs take longer
        csa2.sparse_attn_full(step, ws)
        st, info = csa2.check(ws)               # the call returned and the stream drained
        assert (st, info) == (csa2.ERR_TIMEOUT, 5), (st, info)
    finally:
        csa2.debug_set_wait_limit(0)
    out.zero_()
    topk_idx.zero_()
    csa2.sparse_attn_full(step, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    assert torch.equal(topk_idx, idx_ref)
    assert torch.equal(out, o_ref)
