"""Shared helpers for the GPU parity tests: move seeded synthetic inputs to the device,
build caches through the library, and copy results back for the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Cache:
    """A paged cache on the GPU plus its host twin written by the oracle from the same inputs."""

    def __init__(self, n_req: int, max_pages: int, block_table: np.ndarray | None = None, n_pages: int | None = None,
                 mx: bool = False):
        from fp4_compressed_sparse_csa2_gb300 import csa2
        self.n_req, self.max_pages, self.mx = n_req, max_pages, mx
        self.n_pages = n_pages or (n_req * max_pages if block_table is None else int(block_table.max()) + 1)
        self.kv = torch.zeros(self.n_pages * csa2.KV_PAGE_BYTES, dtype=torch.uint8, device="cuda")
        idx_page = csa2.IDX_MX_PAGE_BYTES if mx else csa2.IDX_PAGE_BYTES
        self.idx = torch.zeros(self.n_pages * idx_page, dtype=torch.uint8, device="cuda")
        self.bt_np = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
        self.bt = None if block_table is None else dev(self.bt_np)
        self.c = csa2.make_cache(self.kv, self.idx, max_pages, self.bt,
                                 idx_format=csa2.IDX_MXFP4 if mx else csa2.IDX_E4M3_16)
        self.ws = csa2.alloc_workspace(1, 64, 0, False)

    def pack(self, lat_bits, key_bits, req, pos):
        from fp4_compressed_sparse_csa2_gb300 import csa2
        csa2.pack_kv(dev_bf16(lat_bits), dev_bf16(key_bits), dev(req.astype(np.int32)), dev(pos.astype(np.int64)),
                     self.c, self.ws)

    def host(self):
        return self.kv.cpu().numpy(), self.idx.cpu().numpy()


def fill_cache(cache: Cache, n_entries: list[int], seed: int, outlier_frac: float = 0.0):
    """Pack n_entries[r] seeded N(0,1) entries at positions 0.. of each request; returns host inputs."""
    lats, keys, reqs, poss = [], [], [], []
    for r, n in enumerate(n_entries):
        if n == 0:
            continue
        lats.append(synth.normal_bf16_rows_with_outliers(seed + 101 * r, n, 512, outlier_frac, 8.0))
        keys.append(synth.normal_bf16_rows_with_outliers(seed + 101 * r + 1, n, 128, outlier_frac, 8.0))
        reqs.append(np.full(n, r, np.int32))
        poss.append(np.arange(n, dtype=np.int64))
    lat, key, req, pos = (np.concatenate(x) for x in (lats, keys, reqs, poss))
    cache.pack(lat, key, req, pos)
    return lat, key, req, pos
