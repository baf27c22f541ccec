"""Pins of the oracle's E4M3 / E2M1 codecs against the format definitions on
"DeepSeek's Attention and KV Cache - From MLA to CSA2", "A Precision Primer",
against torch's independent float8_e4m3fn cast, and by brute-force nearest search."""
import json
import os

import numpy as np
import pytest
import torch

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formats.json")))


def test_e2m1_decode_matches_printed_magnitudes(orc):
    mags = [orc.e2m1_decode(c) for c in range(8)]
    assert mags == GOLD["e2m1_magnitudes"]
    assert [orc.e2m1_decode(8 | c) for c in range(8)] == [-m for m in GOLD["e2m1_magnitudes"]]
    vals = [orc.e2m1_decode(c) for c in range(16)]
    assert all(np.isfinite(vals))  # no Inf / NaN in E2M1


def test_e4m3_decode_range(orc):
    vals = np.array([orc.e4m3_decode(c) for c in range(256)])
    fin = vals[np.isfinite(vals)]
    assert fin.max() == GOLD["e4m3_max"] and fin.min() == -GOLD["e4m3_max"]
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF]) and np.isnan(vals).sum() == 2
    assert GOLD["e4m3_max"] * max(GOLD["e2m1_magnitudes"]) == GOLD["block_range"]
    pos = np.sort(np.unique(fin[fin > 0]))
    assert pos.size == 126 and pos[0] == 2.0 ** -9            # smallest subnormal
    # decode agrees with torch's float8_e4m3fn for every finite code
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = np.isfinite(vals)
    assert np.array_equal(vals[ok], t[ok])


def _e4m3_inputs():
    g = np.random.default_rng(1)
    # all bf16 patterns (finite), random fp32 across binades, and grid midpoints +- 1 ulp
    bf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[np.isfinite(bf)]
    rnd = (g.standard_normal(200000) * np.exp2(g.uniform(-14, 10, 200000))).astype(np.float32)
    return np.concatenate([bf, rnd])


def test_e4m3_encode_matches_torch_rn_even(orc):
    x = _e4m3_inputs()
    x = x[np.abs(x) <= 464.0]            # torch saturates up to 464, then NaN
    # grid midpoints and their fp32 neighbours
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    pos = np.sort(np.unique(t[np.isfinite(t) & (t >= 0)]))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    mids = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    x = np.concatenate([x, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(v) for v in x], dtype=np.uint8)
    # torch maps -0 -> 0x80 and tiny negatives to 0x80 as well; compare as codes
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:10]], got[bad[:10]], ref[bad[:10]])


def test_e4m3_encode_saturates(orc):
    for v in [448.0, 464.0, 480.0, 1e6, 3.0e38]:
        assert orc.e4m3_encode(v) == 0x7E and orc.e4m3_encode(-v) == 0xFE


def _brute_e2m1(y):
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    a = min(abs(float(y)), 6.0)
    d = np.abs(mags - a)
    best = np.nonzero(d == d.min())[0]
    c = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
    return int(c) | (8 if np.signbit(y) else 0)


def test_e2m1_encode_exhaustive_bf16(orc):
    bf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[np.isfinite(bf)]
    got = np.array([orc.e2m1_encode(v) for v in bf])
    ref = np.array([_brute_e2m1(v) for v in bf])
    assert np.array_equal(got, ref)


def test_e2m1_ties_round_to_even(orc):
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for y, c in ties.items():
        assert orc.e2m1_encode(y) == c and orc.e2m1_encode(-y) == (c | 8)
    assert orc.e2m1_encode(-0.1) == 8      # sign kept on a zero magnitude
    assert orc.e2m1_encode(7.0) == 7 and orc.e2m1_encode(-100.0) == 15


def test_quant_block_maps_max_onto_six(orc):
    g = np.random.default_rng(3)
    for _ in range(200):
        x = (g.standard_normal(16) * np.exp2(g.uniform(-8, 6))).astype(np.float32)
        codes, sc = orc.quant_block16(x)
        s = orc.e4m3_decode(sc)
        amax = np.abs(x).max()
        assert s == orc.e4m3_decode(orc.e4m3_encode(np.float32(amax) / np.float32(6.0)))
        deq = np.array([orc.e2m1_decode(c) for c in codes]) * s
        # each element is the nearest grid point of x/s (ties even), saturated at +-6 s
        for xi, ci in zip(x, codes):
            assert ci == _brute_e2m1(np.float32(xi) / np.float32(s))
        assert np.abs(deq).max() <= 6 * s


def test_quant_block_zero_scale_is_plus_zero(orc):
    x = np.full(16, 2.0 ** -14, np.float32)     # amax / 6 < 2^-10 -> scale rounds to 0
    x[3] = -x[3]
    codes, sc = orc.quant_block16(x)
    assert sc == 0 and not codes.any()
    codes, sc = orc.quant_block16(np.zeros(16, np.float32))
    assert sc == 0 and not codes.any()


def test_dequant_is_exact_and_roundtrips(orc):
    """Values on the grid (e2m1 x e4m3) survive pack -> dequant -> pack unchanged."""
    g = np.random.default_rng(5)
    for _ in range(100):
        sc = int(g.integers(1, 0x7E))
        codes = g.integers(0, 16, 16).astype(np.uint8)
        codes[0] = 7  # keep the block max at 6 x scale so the scale is recovered
        x = np.array([orc.e2m1_decode(c) for c in codes]) * orc.e4m3_decode(sc)
        assert np.array_equal(x.astype(np.float32).astype(np.float64), x)   # exact in fp32
        c2, s2 = orc.quant_block16(x.astype(np.float32))
        mag = lambda c: c & 7
        assert s2 == sc
        assert np.array_equal([orc.e2m1_decode(c) for c in c2], [orc.e2m1_decode(c) for c in codes])
