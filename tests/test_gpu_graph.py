"""A whole layer step captured in a CUDA graph: the C ABI launches only on the caller's
stream and neither allocates nor synchronises inside a step, so the Full-mode step
(pack, indexer, top-k, attention — chained by programmatic dependent launch; at this
batch size the attention runs as clusters of key splits merged through the workspace)
can be captured after one eager call and replayed; the replays reproduce the eager
outputs bit for bit."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


def test_full_step_captured_and_replayed(csa2):
    B, T = 3, 2500
    mp = (T + 127) // 128
    cache = Cache(B, mp)
    fill_cache(cache, [T - 1] * B, seed=995)
    q = dev_bf16(synth.normal_bf16(996, (B, 64, 512)))
    qi = dev_bf16(synth.normal_bf16(997, (B, 64, 128)))
    w = dev(synth.normal_f32(998, (B, 64)))
    win = dev_bf16(synth.normal_bf16(999, (B * 128, 512)))
    new_lat = dev_bf16(synth.normal_bf16(1001, (B, 512)))
    new_key = dev_bf16(synth.normal_bf16(1002, (B, 128)))
    o = dict(topk_idx=torch.empty((B, 512), dtype=torch.int32, device="cuda"),
             out=torch.empty((B, 64, 512), dtype=torch.bfloat16, device="cuda"),
             lse=torch.empty((B, 64), dtype=torch.float32, device="cuda"),
             scores=torch.empty((B, T), dtype=torch.float32, device="cuda"), ld=T)
    step = csa2.make_step(n_q=B, t_max=T, q=q, req=dev(np.arange(B, dtype=np.int32)),
                          n_visible=dev(np.full(B, T, np.int32)), window=win,
                          win_start=dev(np.arange(B, dtype=np.int64) * 128), win_len=dev(np.full(B, 128, np.int32)),
                          cache=cache.c, q_idx=qi, w=w, n_new=B, new_latent=new_lat, new_idx_key=new_key,
                          new_req=dev(np.arange(B, dtype=np.int32)), new_pos=dev(np.full(B, T - 1, np.int64)), **o)
    ws = csa2.alloc_workspace(B, 64, T, False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        csa2.sparse_attn_full(step, ws, stream=s)          # eager: also sets the per-device kernel attributes
    s.synchronize()
    assert csa2.check(ws, s) == (csa2.OK, 0)
    eager = {k: v.clone() for k, v in o.items() if torch.is_tensor(v)}
    for v in o.values():
        if torch.is_tensor(v):
            v.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        csa2.sparse_attn_full(step, ws, stream=s)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for k, v in eager.items():
            assert torch.equal(o[k], v), k
    assert csa2.check(ws) == (csa2.OK, 0)
