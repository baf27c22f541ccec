"""The packed cache is a plain byte format: pages written by the library, saved to disk and
loaded back into fresh device memory give bit-identical scores, selection and attention
("DeepSeek's Attention and KV Cache", "DeepSeek-V4.1": the global cache persists; the
pages fix only the entry sizes, the layout is this library's and is stated in csa2.h)."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16, fill_cache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mx", [False, True])
def test_saved_and_reloaded_cache_is_equivalent(csa2, tmp_path, mx):
    B, T = 2, 3000
    mp = (T + 127) // 128
    cache = Cache(B, mp, mx=mx)
    fill_cache(cache, [T] * B, seed=990)
    np.save(tmp_path / "kv.npy", cache.kv.cpu().numpy())
    np.save(tmp_path / "idx.npy", cache.idx.cpu().numpy())
    kv2 = torch.from_numpy(np.load(tmp_path / "kv.npy")).cuda()
    idx2 = torch.from_numpy(np.load(tmp_path / "idx.npy")).cuda()
    c2 = csa2.make_cache(kv2, idx2, mp, idx_format=csa2.IDX_MXFP4 if mx else csa2.IDX_E4M3_16)
    q = dev_bf16(synth.normal_bf16(991, (B, 64, 512)))
    qi = dev_bf16(synth.normal_bf16(992, (B, 64, 128)))
    w = dev(synth.normal_f32(993, (B, 64)))
    win = dev_bf16(synth.normal_bf16(994, (B * 128, 512)))
    common = dict(n_q=B, t_max=T, q=q, req=dev(np.arange(B, dtype=np.int32)), n_visible=dev(np.full(B, T, np.int32)),
                  window=win, win_start=dev(np.arange(B, dtype=np.int64) * 128),
                  win_len=dev(np.full(B, 128, np.int32)), q_idx=qi, w=w)
    res = []
    for c in (cache.c, c2):
        o = dict(topk_idx=torch.empty((B, 512), dtype=torch.int32, device="cuda"),
                 out=torch.empty((B, 64, 512), dtype=torch.bfloat16, device="cuda"),
                 lse=torch.empty((B, 64), dtype=torch.float32, device="cuda"),
                 scores=torch.empty((B, T), dtype=torch.float32, device="cuda"), ld=T)
        ws = csa2.alloc_workspace(B, 64, T, False)
        csa2.sparse_attn_reindex(csa2.make_step(cache=c, **common, **o), ws)
        assert csa2.check(ws) == (csa2.OK, 0)
        res.append(o)
    for k in ("scores", "topk_idx", "out", "lse"):
        assert torch.equal(res[0][k], res[1][k]), k
