"""KV-cache byte accounting -- TEST INFRASTRUCTURE ONLY (part of the CPU oracle).

Bytes per token of global KV = sum over layer groups of
(layers keeping their own entries) x (entries per token = 1/m) x (bytes per entry),
as stated on [P4] "From First Principles: DeepSeek-V4.1-Flash Inference", "The bill",
and as the four-lever product on [P1] "DeepSeek's Attention and KV Cache - From MLA to
CSA2", "The Cost Being Cut" and its "Test Yourself" answer 1 (L x 2 H_kv d_h x b).

Entry sizes come from the formats: [P1] "A Precision Primer" (E2M1, E4M3, E8M0, block
sizes) and "DeepSeek-V4.1 ... Four bits for the main KV" (288 B), [P3] section 3 (72 B
indexer key in the main-KV format), [P1] "DeepSeek-V4" (584 B row, 68 B MXFP4 key).
"""
from __future__ import annotations

from fractions import Fraction


def dense_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """L x 2 H_kv d_h x b: K and V per head per layer [P1 Test Yourself, answer 1]."""
    return layers * 2 * kv_heads * head_dim * bytes_per_elem


def block_format_bytes(channels: int, elem_bits: int, block: int, scale_bytes: int) -> Fraction:
    """Bytes of one entry in a block-scaled format: elements plus one scale per block."""
    return Fraction(channels * elem_bits, 8) + Fraction(channels, block) * scale_bytes


def e2m1_e4m3_16(channels: int) -> Fraction:
    """E2M1 elements with one E4M3 scale per 16 channels, no global scale [P1 "DeepSeek-V4.1"]."""
    return block_format_bytes(channels, 4, 16, 1)


def mxfp4(channels: int) -> Fraction:
    """MXFP4: E2M1 elements with one E8M0 scale per 32 [P1 "A Precision Primer"]."""
    return block_format_bytes(channels, 4, 32, 1)


def bytes_per_token(groups) -> Fraction:
    """Sum over (layers, compression ratio m, bytes per entry) of layers x (1/m) x bytes [P4 "The bill"]."""
    return sum((Fraction(layers) / m * Fraction(b) for layers, m, b in groups), Fraction(0))


def v41_flash(indexer_bytes) -> Fraction:
    """Four caches: three encoder Full layers at m = 2 and one decoder Full layer at m = 1
    [P3 section 2; P4 "CSA2: four layers keep their own copy"]."""
    entry = e2m1_e4m3_16(512) + Fraction(indexer_bytes)
    return bytes_per_token([(3, 2, entry), (1, 1, entry)])


def window_state_bytes(layers: int, window: int, entry_bytes: int) -> int:
    """Bounded sliding-window state per sequence: layers x window x bytes [P1 "The Arithmetic, Rebuilt"]."""
    return layers * window * entry_bytes
