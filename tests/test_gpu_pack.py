"""Pack parity: the cache bytes written by csa2_pack_kv equal the oracle's, bit for bit
("DeepSeek's Attention and KV Cache", "DeepSeek-V4.1": E2M1 with one E4M3 scale per 16
channels, block maximum mapped onto 6; "DeepSeek-V4.1-Flash and the 890-byte KV cache",
section 3: 72-byte indexer key in the same format)."""
import numpy as np
import pytest

import synth
from helpers import Cache, fill_cache

pytestmark = pytest.mark.gpu


def _oracle_pages(orc, cache, lat, key, req, pos):
    kv, ix = orc.alloc_pages(cache.n_pages)
    orc.pack_kv(lat, key, req, pos, kv, ix, cache.bt_np, cache.max_pages)
    return kv, ix


def _assert_same(orc, cache, lat, key, req, pos):
    kv_h, ix_h = _oracle_pages(orc, cache, lat, key, req, pos)
    kv_g, ix_g = cache.host()
    bad = np.nonzero(kv_g != kv_h)[0]
    assert bad.size == 0, f"main-KV bytes differ at {bad[:8]}: gpu {kv_g[bad[:8]]} oracle {kv_h[bad[:8]]}"
    bad = np.nonzero(ix_g != ix_h)[0]
    assert bad.size == 0, f"indexer bytes differ at {bad[:8]}: gpu {ix_g[bad[:8]]} oracle {ix_h[bad[:8]]}"


def test_pack_random_ragged(orc, csa2):
    cache = Cache(n_req=3, max_pages=3)
    lat, key, req, pos = fill_cache(cache, [300, 130, 1], seed=5)
    _assert_same(orc, cache, lat, key, req, pos)


def test_pack_block_table_and_outliers(orc, csa2):
    bt = np.array([[4, 1], [0, 3]], np.int32)
    cache = Cache(n_req=2, max_pages=2, block_table=bt, n_pages=5)
    lat, key, req, pos = fill_cache(cache, [256, 200], seed=6, outlier_frac=0.05)
    _assert_same(orc, cache, lat, key, req, pos)


def _adversarial_rows():
    """Blocks of 16 values hitting the codec's edge cases, as bf16 bit patterns."""
    f = np.float32
    blocks = [
        np.zeros(16, f),                                   # zero block -> scale 0, +0 codes
        -np.zeros(16, f),                                  # negative zeros
        np.full(16, 2.0 ** -20, f) * np.array([1, -1] * 8, f),   # scale underflows to 0
        np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75, -2.5, -3.5, -5, 0], f),  # ties
        np.array([6.375] + [1.0] * 15, f),                 # amax/6 on an E4M3 midpoint
        np.array([1e30, -1e30] + [3.0] * 14, f),           # scale saturates at 448
        np.array([6 * 2.0 ** -8] + [2.0 ** -9] * 15, f),   # subnormal E4M3 scale
        np.array([448 * 6, -448 * 6] + [1.0] * 14, f),     # largest representable block
        np.array([0.1, -0.01, 0.001, -0.0001] * 4, f),     # tiny negatives -> signed zero codes
    ]
    # every bf16 value in [-6, 6] with the block max pinned at 6 (scale exactly 1)
    allbf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    inr = allbf[np.isfinite(allbf) & (np.abs(allbf) <= 6.0)]
    for i in range(0, inr.size, 15):
        chunk = inr[i:i + 15]
        blocks.append(np.concatenate([[6.0], chunk, np.zeros(15 - chunk.size)]).astype(f))
    # every positive finite bf16 value as a block maximum (all scale codes and their rounding)
    pos = allbf[np.isfinite(allbf) & (allbf > 0)]
    for v in pos[::3]:
        blocks.append((np.array([1, -1 / 3, 1 / 7, -0.5] * 4, f) * v).astype(f))
    x = np.concatenate(blocks)
    pad = (-x.size) % 512
    x = np.concatenate([x, np.zeros(pad, f)]).reshape(-1, 512)
    return synth.bf16_bits(x)


def test_pack_adversarial_and_exhaustive_codec(orc, csa2):
    lat = _adversarial_rows()
    n = lat.shape[0]
    key = np.ascontiguousarray(lat[:, :128])
    pages = (n + 127) // 128
    cache = Cache(n_req=1, max_pages=pages)
    req = np.zeros(n, np.int32)
    pos = np.arange(n, dtype=np.int64)
    cache.pack(lat, key, req, pos)
    _assert_same(orc, cache, lat, key, req, pos)


def test_pack_rejects_out_of_range_positions(orc, csa2):
    cache = Cache(n_req=1, max_pages=1)
    lat = synth.normal_bf16(1, (2, 512))
    key = synth.normal_bf16(2, (2, 128))
    cache.pack(lat, key, np.zeros(2, np.int32), np.array([5, 128], np.int64))  # 128 is beyond one page
    st, info = csa2.check(cache.ws)
    assert st == csa2.ERR_DEVICE and info == 2
    assert csa2.check(cache.ws) == (csa2.OK, 0)   # the error word was cleared
