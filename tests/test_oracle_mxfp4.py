"""Pins of the oracle's MXFP4 indexer key ("DeepSeek's Attention and KV Cache - From MLA to
CSA2": "A Precision Primer", block scaling with MX formats and E8M0, and "DeepSeek-V4", the
indexer in four bits; "From First Principles: DeepSeek-V4.1-Flash Inference", "What's in a
cell": 64 bytes of nibbles plus four E8M0 scales, 68 bytes).

Pinned here: the printed worked example (block maximum 3 + delta takes the E8M0 scale 1 and
leaves the rungs 4 and 6 unused, where the E4M3 scale lands the maximum on 6), the entry
size from the bits per element, the exponent rule by brute force over every positive bf16
amax, the element codes by a brute-force nearest search over the printed magnitudes, the
page layout (every byte of a full page written once, every entry read back), round trips
of on-grid records, and the index score's one-head reduction and linearity in w."""
import json
import math
import os

import numpy as np

import synth

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mx_scale_example.json")))
FMT = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formats.json")))
MAGS = FMT["e2m1_magnitudes"]


def _smallest_e(amax: float) -> int:
    """Brute force: the smallest e in [-127, 127] with amax <= 6 * 2^e (-127 for zero)."""
    if amax == 0.0:
        return -127
    for e in range(-127, 128):
        if amax <= math.ldexp(6.0, e):
            return e
    return 127


def _nearest_code(y: float) -> int:
    """Brute-force E2M1 code: nearest printed magnitude, ties to the even code, sign bit 3."""
    a = min(abs(y), 6.0)
    best = min(range(8), key=lambda c: (abs(MAGS[c] - a), c % 2))
    return (8 if math.copysign(1.0, y) < 0 else 0) | best


def _decode(code: int, sc: int) -> float:
    v = MAGS[code & 7] * math.ldexp(1.0, sc - 127)
    return -v if code & 8 else v


def test_entry_size_from_bits_per_element(orc):
    bpe = G["bits_per_element"]
    assert 4 + 8 / G["mx_block"] == bpe["mxfp4"] and 4 + 8 / 16 == bpe["nvfp4"]
    k = G["mxfp4_indexer_key_bytes"]
    assert 128 * bpe["mxfp4"] / 8 == k["total"] == k["nibbles"] + k["scales"] == orc.IDX_MX_BYTES == 68
    assert 128 // G["mx_block"] == k["scales"] and orc.IDX_MX_PAGE_BYTES == 128 * 68


def test_worked_example_block_max_three_plus_delta(orc):
    ex = G["worked_example"]
    rng = np.random.default_rng(11)
    for k in range(1, 32):
        delta = k / 64.0                           # 3 + delta < 3.5 on the bf16 grid (step 1/64)
        x = (rng.uniform(-1, 1, 32) * 3).astype(np.float32)
        x[rng.integers(32)] = ex["block_max_base"] + delta
        x = synth.bf16_to_f32(synth.bf16_bits(x))
        codes, sc = orc.mx_quant_block32(x)
        assert 2.0 ** (sc - 127) == ex["e8m0_scale"]
        i = int(np.argmax(np.abs(x)))
        assert MAGS[codes[i] & 7] == ex["max_quantizes_to"]
        assert not any(MAGS[c & 7] in ex["unused_rungs"] for c in codes)
        # the block-16 E4M3 codec of the same values lands the maximum on 6
        blk = i // 16 * 16
        c16, s16 = orc.quant_block16(x[blk:blk + 16])
        assert MAGS[c16[i - blk] & 7] == ex["e4m3_max_lands_on"]
    assert round(math.log2(3 / 0.5), 2) == ex["binades_used"] and round(math.log2(6 / 0.5), 2) == ex["binades_full"]


def test_exponent_rule_every_positive_bf16(orc):
    bits = np.arange(1, 0x7F80, dtype=np.uint32)       # every positive finite bf16
    vals = (bits << 16).view(np.float32)
    for v in vals[::7]:
        assert orc.mx_exponent(float(v)) == _smallest_e(float(v)), v
    for v in vals[-300:]:
        assert orc.mx_exponent(float(v)) == _smallest_e(float(v)), v
    assert orc.mx_exponent(0.0) == G["e8m0_min_log2"]
    assert orc.mx_exponent(float(vals[-1])) <= G["e8m0_max_log2"]


def test_element_codes_brute_force(orc):
    rng = np.random.default_rng(12)
    for t in range(300):
        x = rng.standard_normal(32) * math.exp(rng.uniform(-20, 20))
        x[rng.integers(32, size=3)] = 0.0
        x = synth.bf16_to_f32(synth.bf16_bits(x.astype(np.float32)))
        codes, sc = orc.mx_quant_block32(x)
        e = sc - 127
        assert e == _smallest_e(float(np.abs(x).max()))
        for xi, c in zip(x, codes):
            assert c == _nearest_code(math.ldexp(float(xi), -e)), (xi, e)


def test_page_layout_every_byte_once_and_read_back(orc):
    keys = synth.normal_bf16(13, (128, 128), scale=2.0)
    pages = orc.alloc_idx_mx_pages(2)
    pages[:] = 0xEE
    req = np.zeros(128, np.int32)
    pos = np.arange(128, dtype=np.int64) + 128        # page 1 of request 0
    orc.pack_idx_mx(keys, req, pos, pages, max_pages=2)
    assert (pages[:8704] == 0xEE).all()               # page 0 untouched
    # every byte of page 1 rewritten: pack twice with different fill, compare
    pages2 = orc.alloc_idx_mx_pages(2)
    pages2[:] = 0x11
    orc.pack_idx_mx(keys, req, pos, pages2, max_pages=2)
    assert (pages[8704:] == pages2[8704:]).all()
    x = synth.bf16_to_f32(keys)
    for e in range(128):
        v = orc.read_idx_mx(pages, 0, 128 + e, max_pages=2)
        for b in range(4):
            codes, sc = orc.mx_quant_block32(x[e, 32 * b:32 * b + 32])
            assert v[32 * b:32 * b + 32].tolist() == [_decode(c, sc) for c in codes]


def test_round_trip_on_grid(orc):
    rng = np.random.default_rng(14)
    vals = np.zeros((64, 128), np.float32)
    for i in range(64):
        for b in range(4):
            e = int(rng.integers(-20, 20))
            codes = rng.integers(16, size=32)
            codes[rng.integers(32)] = int(rng.choice([6, 7, 14, 15]))   # block max on 4 or 6
            vals[i, 32 * b:32 * b + 32] = [_decode(int(c), e + 127) for c in codes]
    bits = synth.bf16_bits(vals)
    assert (synth.bf16_to_f32(bits) == vals).all()
    pages = orc.alloc_idx_mx_pages(1)
    orc.pack_idx_mx(bits, np.zeros(64, np.int32), np.arange(64, dtype=np.int64), pages, max_pages=1)
    for i in range(64):
        assert orc.read_idx_mx(pages, 0, i, max_pages=1).tolist() == vals[i].astype(np.float64).tolist()


def test_index_score_one_head_and_linearity(orc):
    keys = synth.normal_bf16(15, (300, 128))
    pages = orc.alloc_idx_mx_pages(3)
    orc.pack_idx_mx(keys, np.zeros(300, np.int32), np.arange(300, dtype=np.int64), pages, max_pages=3)
    q = synth.normal_bf16(16, (8, 128))
    qf = synth.bf16_to_f32(q)
    # one head, w = 1: ReLU(qhat . khat) / sqrt(128), qhat decoded from the block codes
    for j in range(8):
        qh = []
        for b in range(4):
            codes, sc = orc.mx_quant_block32(qf[j, 32 * b:32 * b + 32])
            qh += [_decode(int(c), sc) for c in codes]
        I, M = orc.index_score_mx(q[j:j + 1], np.ones(1, np.float32), pages, 0, 0, 300, max_pages=3)
        kh = np.stack([orc.read_idx_mx(pages, 0, s, max_pages=3) for s in range(300)])
        ref = np.maximum(kh @ np.array(qh), 0.0) / math.sqrt(128.0)
        assert np.allclose(I, ref, rtol=1e-13, atol=1e-13) and np.allclose(M, ref, rtol=1e-13, atol=1e-13)
    # linearity in w: the 8-head score is the w-weighted sum of one-head scores
    w = synth.normal_f32(17, (8,))
    I8, M8 = orc.index_score_mx(q, w, pages, 0, 0, 300, max_pages=3)
    parts = [orc.index_score_mx(q[j:j + 1], np.ones(1, np.float32), pages, 0, 0, 300, max_pages=3)[0]
             for j in range(8)]
    assert np.allclose(I8, sum(float(w[j]) * parts[j] for j in range(8)), rtol=1e-12, atol=1e-12)
    assert np.allclose(M8, sum(abs(float(w[j])) * parts[j] for j in range(8)), rtol=1e-12, atol=1e-12)
    assert (M8 >= np.abs(I8) - 1e-12).all()


def test_mxfp4_less_accurate_than_e4m3_blocks(orc):
    # the page's seeded latent: the E4M3 / 16 codec gives 0.0912; the MX format wastes part
    # of the ladder (power-of-two scale, block of 32), so its error is larger
    rng = np.random.default_rng(0)
    latent = rng.standard_normal(512)
    latent *= np.sqrt(512) / np.linalg.norm(latent)
    x = latent.astype(np.float32)
    deq = []
    for b in range(16):
        codes, sc = orc.mx_quant_block32(x[32 * b:32 * b + 32])
        deq += [_decode(int(c), sc) for c in codes]
    rel_mx = np.linalg.norm(np.array(deq) - latent) / np.linalg.norm(latent)
    codes, scales = orc.quant_vector(x)
    rel_nv = np.linalg.norm(orc.dequant_vector(codes, scales) - latent) / np.linalg.norm(latent)
    assert round(float(rel_nv), 4) == 0.0912 and rel_mx > rel_nv
