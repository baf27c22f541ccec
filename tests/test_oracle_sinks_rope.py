"""Pins of the oracle's attention sinks and partial RoPE ("From MLA to DSA to HCA/CSA").

* "The sliding window": one sink logit per head is appended to each score row before
  the softmax and dropped after it; it has no value vector, so the surviving weights
  sum to 1 - p_sink.  Pinned by the two-call identity that this implies (the output
  shrinks by exactly e^lse0 / (e^lse0 + e^sink), lse becomes logaddexp(lse0, sink)),
  by the limit sink -> -inf and by the no-key case.
* "What replaced MLA": the trailing 64 channels of q are rotated at the query position
  and the output is rotated back with the negated angle, so each entry contributes
  through R_{-t} R_s = R_{s-t}, relative distance only.  Pinned by the identity
  rotation, by that relative-distance property with exact 90-degree rotations of bf16
  rows (a sign flip and a swap), and by the single-key case where the query's angle
  equals the key's (the output is the unrotated value)."""
import numpy as np
import pytest

import synth

D = 512


def _rot90_rows(bits: np.ndarray) -> np.ndarray:
    """Rotate the trailing 64 channels of bf16 rows by 90 degrees, exactly: with
    rotate_half pairing (448 + i, 480 + i), (a, b) -> (a cos - b sin, b cos + a sin)
    at cos 0, sin 1 is (-b, a)."""
    out = bits.copy()
    a = bits[..., 448:480].copy()
    b = bits[..., 480:512].copy()
    out[..., 448:480] = b ^ np.uint16(0x8000)
    out[..., 480:512] = a
    return out


def _angles(seed, n=32):
    th = synth.rng(seed).uniform(-np.pi, np.pi, n)
    return np.cos(th), np.sin(th), th


def _empty_kv(orc):
    kv, _ = orc.alloc_pages(1)
    return kv


def test_no_sinks_no_rope_is_plain_attention(orc):
    kv = _empty_kv(orc)
    q = synth.normal_bf16(901, (4, D))
    win = synth.normal_bf16(902, (50, D))
    idx = np.full(8, -1, np.int32)
    O0, l0 = orc.attention(q, idx, kv, 0, win, 50)
    O1, l1 = orc.attention_ext(q, idx, kv, 0, win, 50)
    assert np.array_equal(O0, O1) and np.array_equal(l0, l1)
    c = np.ones(32)
    s = np.zeros(32)
    O2, l2 = orc.attention_ext(q, idx, kv, 0, win, 50, rope_cos=c, rope_sin=s)
    assert np.array_equal(O0, O2) and np.array_equal(l0, l2)


def test_sink_shrinks_the_output_by_its_share(orc):
    kv = _empty_kv(orc)
    heads = 6
    q = synth.normal_bf16(903, (heads, D), scale=2.0)
    win = synth.normal_bf16(904, (40, D))
    idx = np.full(4, -1, np.int32)
    sinks = np.array([-3.0, 0.0, 0.5, 2.0, 6.0, -40.0])
    O0, l0 = orc.attention(q, idx, kv, 0, win, 40)
    O1, l1 = orc.attention_ext(q, idx, kv, 0, win, 40, sinks=sinks)
    share = np.exp(l0) / (np.exp(l0) + np.exp(sinks))  # weight left to the real keys
    np.testing.assert_allclose(O1, O0 * share[:, None], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, np.logaddexp(l0, sinks), rtol=1e-13, atol=1e-13)
    # a sink far below every score changes nothing (to fp64)
    O2, l2 = orc.attention_ext(q, idx, kv, 0, win, 40, sinks=np.full(heads, -1e4))
    np.testing.assert_allclose(O2, O0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l2, l0, rtol=0, atol=1e-15)


def test_sink_with_no_keys(orc):
    kv = _empty_kv(orc)
    q = synth.normal_bf16(905, (3, D))
    win = synth.normal_bf16(906, (1, D))
    idx = np.full(4, -1, np.int32)
    O, l = orc.attention_ext(q, idx, kv, 0, win, 0, sinks=np.array([0.25, -1.0, 3.0]))
    assert np.all(O == 0.0)
    np.testing.assert_array_equal(l, [0.25, -1.0, 3.0])
    O, l = orc.attention_ext(q, idx, kv, 0, win, 0)
    assert np.all(O == 0.0) and np.all(np.isneginf(l))


def test_rope_depends_on_relative_angle_only(orc):
    """Rotating every key by 90 degrees and the query's angle by 90 degrees leaves the
    output unchanged (R_{-(t+phi)} R_{s+phi} = R_{-t} R_s)."""
    kv = _empty_kv(orc)
    q = synth.normal_bf16(907, (5, D), scale=1.5)
    win = synth.normal_bf16(908, (64, D))
    idx = np.full(4, -1, np.int32)
    c, s, _ = _angles(909)
    O0, l0 = orc.attention_ext(q, idx, kv, 0, win, 64, rope_cos=c, rope_sin=s)
    # angle + 90 degrees: cos -> -sin, sin -> cos (exact)
    O1, l1 = orc.attention_ext(q, idx, kv, 0, _rot90_rows(win), 64, rope_cos=-s, rope_sin=c)
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)
    # and the rotation is not the identity: without the query's extra 90 degrees it differs
    O2, _ = orc.attention_ext(q, idx, kv, 0, _rot90_rows(win), 64, rope_cos=c, rope_sin=s)
    assert np.max(np.abs(O2 - O0)) > 1e-3


def test_rope_undoes_the_value_rotation_at_the_query_position(orc):
    """One key v rotated by 90 degrees (as cached), query at the same angle: the output
    is v itself; at angle 0 it is the rotated row."""
    kv = _empty_kv(orc)
    v = synth.normal_bf16(910, (1, D))
    vr = _rot90_rows(v)
    q = synth.normal_bf16(911, (2, D))
    idx = np.full(4, -1, np.int32)
    zeros, ones = np.zeros(32), np.ones(32)
    O, _ = orc.attention_ext(q, idx, kv, 0, vr, 1, rope_cos=zeros, rope_sin=ones)
    np.testing.assert_allclose(O, np.repeat(synth.bf16_to_f32(v).astype(np.float64), 2, axis=0), rtol=0,
                               atol=0)
    O, _ = orc.attention_ext(q, idx, kv, 0, vr, 1, rope_cos=ones, rope_sin=zeros)
    np.testing.assert_allclose(O, np.repeat(synth.bf16_to_f32(vr).astype(np.float64), 2, axis=0), rtol=0,
                               atol=0)


def test_rope_pairs_half_split_channels(orc):
    """A query with a single non-zero channel 448 + i, rotated by angle i, puts its mass
    on channels 448 + i and 480 + i only: score against window rows that are unit
    vectors e_{448+i} and e_{480+i} gives cos and sin."""
    kv = _empty_kv(orc)
    one = synth.bf16_bits(np.array([1.0], np.float32))[0]
    i = 5
    q = np.zeros((1, D), np.uint16)
    q[0, 448 + i] = one
    win = np.zeros((2, D), np.uint16)
    win[0, 448 + i] = one
    win[1, 480 + i] = one
    idx = np.full(4, -1, np.int32)
    th = np.zeros(32)
    th[i] = 0.7
    # one window row at a time: lse = scale * (q_rot . row)
    for row, expect in ((0, np.cos(0.7)), (1, np.sin(0.7))):
        _, l = orc.attention_ext(q, idx, kv, 0, win[row:row + 1], 1, scale=1.0, rope_cos=np.cos(th),
                                 rope_sin=np.sin(th))
        assert l[0] == pytest.approx(expect, abs=1e-15)
