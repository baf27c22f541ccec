"""The in-call quantisation of the indexer query, byte for byte.

"DeepSeek's Attention and KV Cache", "DeepSeek-V4": the indexer's query-key product
multiplies entirely in FP4, so the quantised query is a byte-exact quantity like the
cache.  After a csa2_index_score call the workspace holds each query group's packed
query (header 256 bytes, then one group of N = G * heads_I rows per G consecutive
queries, N * 64 nibble bytes followed by the scale atoms: 1024 bytes of E4M3 codes, or
512 of E8M0 codes for MXFP4).  Row n of a group is head n % heads_I of query
g * G + n // heads_I.  The layout is the indexer page's operand layout restated here
from its definition in csa2.h: the nibble of row n, channel c at
(n / 8) * 512 + (c / 32) * 128 + (n % 8) * 16 + (c % 32) / 2 (even c in the low nibble);
the E4M3 scale of block b (16 channels) at nib + (b / 4) * 512 + (n % 32) * 16 +
(n / 32) * 4 + b % 4; the E8M0 code of block b (32 channels) at
nib + (n % 32) * 16 + (n / 32) * 4 + b.

The GPU's codes and scale codes are compared with the oracle's quantisation of the same
bf16 rows (oracle.quant_vector, oracle.mx_quant_block32) for both key formats, 64 and 32
indexer heads and groups of 1 and 2, on N(0,1) rows and on the adversarial blocks of
the pack test (zero and negative-zero blocks, E2M1 ties, E4M3 midpoints, saturation,
subnormal scales, every bf16 value in [-6, 6] at scale 1, every third positive bf16
value as a block maximum)."""
import numpy as np
import pytest
import torch

import synth
from helpers import Cache, dev, dev_bf16
from test_gpu_pack import _adversarial_rows

pytestmark = pytest.mark.gpu
HEADER = 256


def _unpack_group(buf, N, mx):
    """Codes [N][128] and scale codes [N][8] (E4M3) or [N][4] (E8M0) of one packed group."""
    nib = N * 64
    codes = np.zeros((N, 128), np.uint8)
    for n in range(N):
        for c in range(0, 128, 2):
            byte = buf[(n // 8) * 512 + (c // 32) * 128 + (n % 8) * 16 + (c % 32) // 2]
            codes[n, c] = byte & 0xF
            codes[n, c + 1] = byte >> 4
    if mx:
        sc = np.array([[buf[nib + (n % 32) * 16 + (n // 32) * 4 + b] for b in range(4)] for n in range(N)], np.uint8)
    else:
        sc = np.array([[buf[nib + (b // 4) * 512 + (n % 32) * 16 + (n // 32) * 4 + b % 4] for b in range(8)]
                       for n in range(N)], np.uint8)
    return codes, sc


def _oracle_row(orc, bits, mx):
    x = synth.bf16_to_f32(bits)
    if not mx:
        return orc.quant_vector(x)
    codes, sc = [], []
    for b in range(4):
        c, s = orc.mx_quant_block32(x[32 * b:32 * b + 32])
        codes.append(c)
        sc.append(s)
    return np.concatenate(codes), np.array(sc, np.uint8)


def _check(orc, csa2, q_bits, heads_I, G, mx):
    n_q = q_bits.shape[0]
    T = 256
    cache = Cache(n_req=1, max_pages=2, mx=mx)
    lat = synth.normal_bf16(70, (T, 512))
    key = synth.normal_bf16(71, (T, 128))
    cache.pack(lat, key, np.zeros(T, np.int32), np.arange(T, dtype=np.int64))
    w = synth.normal_f32(72, (n_q, heads_I))
    scores = torch.zeros((n_q, T), dtype=torch.float32, device="cuda")
    ws = csa2.alloc_workspace(n_q, heads_I, T, False)
    csa2.index_score(dev_bf16(q_bits), dev(w), heads_I, dev(np.zeros(n_q, np.int32)),
                     dev(np.full(n_q, T, np.int32)), n_q, G, T, cache.c, scores, T, ws)
    assert csa2.check(ws) == (csa2.OK, 0)
    N = G * heads_I
    gbytes = N * 64 + (512 if mx else 1024)
    host = ws.cpu().numpy()
    n_groups = (n_q + G - 1) // G
    for g in range(n_groups):
        codes, sc = _unpack_group(host[HEADER + g * gbytes:HEADER + (g + 1) * gbytes], N, mx)
        for n in range(N):
            q = g * G + n // heads_I
            if q >= n_q:
                continue
            oc, os_ = _oracle_row(orc, q_bits[q, n % heads_I], mx)
            bad = np.nonzero(codes[n] != oc)[0]
            assert bad.size == 0, f"group {g} row {n}: codes differ at channels {bad[:8]}"
            assert np.array_equal(sc[n], os_), f"group {g} row {n}: scale codes {sc[n]} vs {os_}"


@pytest.mark.parametrize("mx", [False, True])
@pytest.mark.parametrize("heads_I,G", [(64, 1), (64, 2), (32, 1), (32, 2)])
def test_packed_query_random(orc, csa2, heads_I, G, mx):
    n_q = 5 if G == 2 else 3   # a short last group when G = 2
    q = synth.normal_bf16(80 + heads_I + G, (n_q, heads_I, 128))
    q[0, 0] = synth.normal_bf16(81, (128,), 8.0)          # a peaky head
    _check(orc, csa2, q, heads_I, G, mx)


@pytest.mark.parametrize("mx", [False, True])
def test_packed_query_adversarial_blocks(orc, csa2, mx):
    rows = _adversarial_rows().reshape(-1, 128)          # the pack test's edge-case blocks, 128 channels a row
    heads_I, G = 64, 2
    n_q = (rows.shape[0] + heads_I - 1) // heads_I
    pad = n_q * heads_I - rows.shape[0]
    rows = np.concatenate([rows, np.zeros((pad, 128), np.uint16)])
    _check(orc, csa2, rows.reshape(n_q, heads_I, 128), heads_I, G, mx)
