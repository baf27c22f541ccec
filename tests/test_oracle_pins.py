"""Pins of the oracle against numbers printed on the pages: the FP4 quantizer check
and the KV bytes-per-token arithmetic of four model generations.

Sources: "DeepSeek's Attention and KV Cache - From MLA to CSA2, From First Principles"
(sections "The Cost Being Cut", "What V3 stored", "DeepSeek-V4", "DeepSeek-V4.1" with
its "Check it in numpy" output, "The Arithmetic, Rebuilt"); "DeepSeek-V4.1-Flash and the
890-byte KV cache" (sections 1, 3, 8); "From First Principles: DeepSeek-V4.1-Flash
Inference" ("FP4 main KV: smaller cells")."""
import json
import os
from fractions import Fraction

import numpy as np

from oracle import accounting as acc

G = os.path.join(os.path.dirname(__file__), "golden")
TOY = json.load(open(os.path.join(G, "fp4_quantizer_toy.json")))
KV = json.load(open(os.path.join(G, "kv_bytes_per_token.json")))
FMT = json.load(open(os.path.join(G, "formats.json")))


def test_fp4_quantizer_toy_reproduces_printed_error(orc):
    rng = np.random.default_rng(0)
    latent = rng.standard_normal(512)
    latent *= np.sqrt(512) / np.linalg.norm(latent)
    assert round(float(np.abs(latent).max()), 3) == TOY["max_abs_latent"]
    codes, scales = orc.quant_vector(latent.astype(np.float32))
    deq = orc.dequant_vector(codes, scales)
    rel = np.linalg.norm(deq - latent) / np.linalg.norm(latent)
    assert round(float(rel), 4) == TOY["rel_l2_error"]
    # bytes per 512-channel entry: fp16, fp8, fp4 + E4M3/16
    b = TOY["bytes_per_512ch_entry"]
    assert (512 * 2, 512 * 1, int(acc.e2m1_e4m3_16(512))) == (b["fp16"], b["fp8"], b["fp4_e4m3_16"])


def test_entry_sizes():
    assert acc.e2m1_e4m3_16(512) == FMT["main_kv_entry_bytes"] == 288
    assert Fraction(512 * 4, 8) == FMT["main_kv_nibble_bytes"]
    assert Fraction(512, 16) == FMT["main_kv_scale_bytes"]
    assert acc.e2m1_e4m3_16(128) == FMT["indexer_entry_bytes_main_format"] == 72
    assert acc.mxfp4(128) == FMT["indexer_entry_bytes_mxfp4"] == 68
    # FP8 window entry: 512 E4M3 bytes + 16 E8M0 scales (one per 32)
    assert acc.block_format_bytes(512, 8, 32, 1) == FMT["fp8_window_entry_bytes"]
    # the oracle's page layout uses exactly these entry sizes
    import oracle
    assert oracle.KV_BYTES == 288 and oracle.IDX_BYTES == 72
    assert oracle.KV_PAGE_BYTES == 128 * 288 and oracle.IDX_PAGE_BYTES == 128 * 72


def test_bytes_per_token_four_generations():
    # DeepSeek LLM 67B: 95 layers, 8 KV heads, head dim 128, bf16
    v1 = acc.dense_bytes_per_token(95, 8, 128, 2)
    assert v1 == KV["v1_67b"]
    # V3.2: 61 layers x (656 B MLA row + 132 B FP8 indexer key)
    v32 = acc.bytes_per_token([(61, 1, 656 + 132)])
    assert v32 == KV["v32"]
    # V4-Flash: 21 CSA layers at m = 4 (584 B row + 68 B MXFP4 key), 20 HCA at m = 128 (584 B)
    v4 = acc.bytes_per_token([(21, 4, 584 + acc.mxfp4(128)), (20, 128, 584)])
    assert v4 == Fraction(351425, 100) and round(v4) == KV["v4_flash"]
    # V4.1-Flash: 2.5 entries x (288 + 68) = 890; with a 72 B indexer key: 900, within ~1 %
    v41 = acc.v41_flash(acc.mxfp4(128))
    assert v41 == KV["v41_flash"]
    v41_72 = acc.v41_flash(72)
    assert v41_72 == 900 and abs(v41_72 - v41) / v41 < 0.012
    # ratios
    assert round(v1 / v41) == KV["reduction_v1_to_v41"]
    assert round(float(v32 / v4), 1) == KV["factor_v32_to_v4"]
    assert round(float(v4 / v41), 1) == KV["factor_v4_to_v41"]
    v3 = 61 * 576 * 2
    assert round(v1 / v3, 1) == KV["factor_v1_to_v3"]
    assert round(v3 / v32, 1) == KV["factor_v3_to_v32"]


def test_v3_cache_and_window_state():
    # 576 x 2 B x 62 layers x 128K tokens = 8.72 GiB (with the MTP layer)
    assert round(576 * 2 * 62 * 128 * 1024 / 2 ** 30, 2) == KV["v3_flashmla_gib_128k"]
    assert round(61 * 576 * 2 * 131072 / 1e9, 1) == KV["v3_gb_128k"]
    assert round(acc.window_state_bytes(40, 128, 528) / 1e6, 1) == KV["window_state_mb_v41"]
    assert round(float(acc.v41_flash(acc.mxfp4(128))) * 1_000_000 / 1e9, 2) == KV["v41_one_million_tokens_gb"]
