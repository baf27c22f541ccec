"""Pins of the oracle's FP8 window ring ("DeepSeek's Attention and KV Cache - From MLA to
CSA2": "Four bits for the main KV, eight for the window" gives the 528-byte entry, 512
E4M3 bytes plus 16 E8M0 scales; "Definition and the bounded cache" gives slot i mod W).

The scale rule (the pages are silent) is pinned by brute force: the exponent is the
smallest e with amax <= 448 * 2^e.  The element codec is the E4M3 codec already pinned
exhaustively; here: round trips on the grid, the half-ulp error bound, the ring's slot
arithmetic, and attention over ring entries equal to attention over the same rows."""
import math

import numpy as np
import pytest

import synth

D = 512


def _smallest_e(amax: float) -> int:
    if amax == 0.0:
        return -127
    e = -140
    while not amax <= math.ldexp(448.0, e):
        e += 1
    return max(-127, min(127, e))


def test_entry_size():
    assert 512 * 1 + 16 == 528  # 512 E4M3 bytes + 16 E8M0 scales


def test_scale_exponent_brute_force(orc):
    vals = [0.0, 448.0, 448.0 * 2.0 ** -3, np.nextafter(448.0, 1e9), np.nextafter(448.0, 0.0), 1.0, 0.5, 3.75,
            2.0 ** -126, 2.0 ** -133, 1e30, 6.0, 7.0, 224.0, 225.0]
    vals += list(np.abs(synth.normal_f32(700, (2000,))) * np.exp(synth.normal_f32(701, (2000,)) * 5))
    for a in vals:
        a = float(np.float32(a))
        assert orc.e8m0_exponent(a) == _smallest_e(a), a


def _row_scales(orc, ring, r, p):
    rec = ring[(r * 128 + p % 128) * 528:(r * 128 + p % 128 + 1) * 528]
    return rec[:512], rec[512:].astype(np.int32) - 127


def test_pack_no_clip_minimal_scale_and_error_bound(orc):
    rows = synth.normal_bf16(702, (40, D), scale=3.0)
    rows[5, :32] = 0                                   # an all-zero block
    ring = orc.alloc_ring(2)
    req = np.array([i % 2 for i in range(40)], np.int32)
    pos = np.arange(40, dtype=np.int64)
    orc.pack_window(rows, req, pos, ring)
    x = synth.bf16_to_f32(rows).astype(np.float64)
    for i in range(40):
        codes, e = _row_scales(orc, ring, req[i], pos[i])
        v = orc.read_window(ring, req[i], pos[i])
        for b in range(16):
            blk = x[i, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            assert e[b] == _smallest_e(amax)
            sc = 2.0 ** e[b]
            assert np.all(np.abs(v[32 * b:32 * b + 32]) <= 448.0 * sc)
            # half an E4M3 ulp: 2^-4 relative in the normal range, 2^-10 * scale below it
            err = np.abs(v[32 * b:32 * b + 32] - blk)
            assert np.all(err <= np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * sc) * (1 + 1e-12))
            if amax > 0:
                assert np.abs(v[32 * b:32 * b + 32]).max() > 224.0 * sc * (1 - 2 ** -4)  # top octave used


def test_grid_values_round_trip(orc):
    """Rows already on the grid (E4M3 values times 2^e with one element at 448 * 2^e)
    pack to exactly those codes and scales."""
    rng = synth.rng(703)
    codes = rng.integers(0, 0x7E, size=(8, D)).astype(np.uint8)          # no NaN pattern
    codes |= (rng.integers(0, 2, size=(8, D)) << 7).astype(np.uint8)
    e = rng.integers(-20, 10, size=(8, 16))
    codes[:, ::32] = 0x7E                                                 # 448 in every block
    vals = np.array([[orc.e4m3_decode(int(c)) for c in row] for row in codes]) * np.repeat(2.0 ** e, 32, axis=1)
    rows = synth.bf16_bits(vals.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(rows).astype(np.float64), vals)  # exact in bf16
    ring = orc.alloc_ring(1)
    orc.pack_window(rows, np.zeros(8, np.int32), np.arange(8, dtype=np.int64), ring)
    for i in range(8):
        c, ee = _row_scales(orc, ring, 0, i)
        assert np.array_equal(ee, e[i])
        # +0 and -0 both decode to 0; compare values, and the codes away from zero
        nz = vals[i] != 0
        assert np.array_equal(c[nz], codes[i][nz])
        assert np.array_equal(orc.read_window(ring, 0, i), vals[i])


def test_ring_slots_wrap(orc):
    rows = synth.normal_bf16(704, (3, D))
    ring = orc.alloc_ring(3)
    orc.pack_window(rows[:1], [2], [5], ring)
    first = orc.read_window(ring, 2, 5)
    orc.pack_window(rows[1:2], [2], [5 + 128], ring)                      # same slot, later position
    assert np.array_equal(orc.read_window(ring, 2, 5), orc.read_window(ring, 2, 133))
    assert not np.array_equal(orc.read_window(ring, 2, 5), first)
    assert np.all(ring[:2 * 128 * 528] == 0)                               # other requests untouched


def test_attention_over_ring_equals_attention_over_rows(orc):
    rows = synth.normal_bf16(705, (300, D))
    ring = orc.alloc_ring(1)
    orc.pack_window(rows, np.zeros(300, np.int32), np.arange(300, dtype=np.int64), ring)
    kv, _ = orc.alloc_pages(1)
    q = synth.normal_bf16(706, (4, D), scale=2.0)
    idx = np.full(4, -1, np.int32)
    for win_pos, win_len in ((299, 128), (140, 100), (10, 11), (5, 0)):
        ring_rows = np.stack([orc.read_window(ring, 0, win_pos - i) for i in range(max(win_len, 1))])
        bits = synth.bf16_bits(ring_rows.astype(np.float32))
        assert np.array_equal(synth.bf16_to_f32(bits).astype(np.float64), ring_rows)  # exact in bf16
        O1, l1 = orc.attention_ring(q, idx, kv, 0, ring, win_pos, win_len)
        O2, l2 = orc.attention_ext(q, idx, kv, 0, bits, win_len)
        np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
