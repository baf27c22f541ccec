"""CSA2 CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU implementation of one CSA2 attention layer
(FP4 cache packing, lightning-indexer scores, top-k selection and shared-KV MQA
over the selected entries plus a sliding window).  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it; the product library
never routes through it.  It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (fp64, plain loops); this module loads it
with ctypes and marshals numpy arrays.  Each wrapper names the passage it
follows; the page titles are:

* [P1] "DeepSeek's Attention and KV Cache - From MLA to CSA2, From First Principles"
* [P2] "From MLA to DSA to HCA/CSA: DeepSeek V3.2 and V4 Attention"
* [P3] "DeepSeek-V4.1-Flash and the 890-byte KV cache"
* [P4] "From First Principles: DeepSeek-V4.1-Flash Inference"

Parity pins for every function are in ``tests/test_oracle_*.py``.  Parity
unpinned: nothing in this module (model-quality effects of the FP4 cache need
trained weights and are out of scope).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D = 512          # main-KV latent width [P1 "DeepSeek-V4.1", FP4 main KV]
DI = 128         # indexer key width [P1 "DeepSeek-V3.2", lightning indexer]
PAGE = 128       # entries per cache page (this build's layout reading)
KV_BYTES = 288   # 256 B nibbles + 32 E4M3 scales [P1 "DeepSeek-V4.1"]
IDX_BYTES = 72   # 64 B nibbles + 8 E4M3 scales [P3 section 3]
KV_PAGE_BYTES = PAGE * KV_BYTES
IDX_PAGE_BYTES = PAGE * IDX_BYTES
IDX_MX_BYTES = 68  # MXFP4 indexer key: 64 B nibbles + 4 E8M0 scales [P1 "DeepSeek-V4"; P4 "What's in a cell"]
IDX_MX_PAGE_BYTES = PAGE * IDX_MX_BYTES


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def _declare(L):
    L.or_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.or_e4m3_decode.restype = ctypes.c_double
    L.or_e4m3_encode.argtypes = [ctypes.c_float]
    L.or_e4m3_encode.restype = ctypes.c_uint8
    L.or_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.or_e2m1_decode.restype = ctypes.c_double
    L.or_e2m1_encode.argtypes = [ctypes.c_float]
    L.or_e2m1_encode.restype = ctypes.c_uint8
    L.or_quant_block16.argtypes = [_f32p, _u8p, _u8p]
    L.or_quant_vector.argtypes = [_f32p, ctypes.c_int64, _u8p, _u8p]
    L.or_pack_kv.argtypes = [_u16p, _u16p, _i32p, _i64p, ctypes.c_int64, _u8p, _u8p, _i32p,
                             ctypes.c_int32]
    L.or_read_main.argtypes = [_u8p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _f64p]
    L.or_read_idx.argtypes = [_u8p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _f64p]
    L.or_index_score.argtypes = [_u16p, _f32p, ctypes.c_int32, _u8p, _i32p, ctypes.c_int32,
                                 ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, _f64p, _f64p]
    L.or_topk.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _i32p]
    L.or_attention.argtypes = [_u16p, ctypes.c_int32, _i32p, ctypes.c_int32, _u8p, _i32p,
                               ctypes.c_int32, ctypes.c_int32, _u16p, ctypes.c_int32,
                               ctypes.c_double, _f64p, _f64p]
    L.or_attention_ext.argtypes = [_u16p, ctypes.c_int32, _i32p, ctypes.c_int32, _u8p, _i32p,
                                   ctypes.c_int32, ctypes.c_int32, _u16p, ctypes.c_int32,
                                   ctypes.c_double, _f64p, _f64p, _f64p, _f64p, _f64p]
    L.or_e8m0_exponent.argtypes = [ctypes.c_double]
    L.or_e8m0_exponent.restype = ctypes.c_int32
    L.or_pack_window.argtypes = [_u16p, _i32p, _i64p, ctypes.c_int64, _u8p]
    L.or_read_window.argtypes = [_u8p, ctypes.c_int32, ctypes.c_int64, _f64p]
    L.or_attention_ring.argtypes = [_u16p, ctypes.c_int32, _i32p, ctypes.c_int32, _u8p, _i32p,
                                    ctypes.c_int32, ctypes.c_int32, _u8p, ctypes.c_int64, ctypes.c_int32,
                                    ctypes.c_double, _f64p, _f64p, _f64p, _f64p, _f64p]
    L.or_mx_exponent.argtypes = [ctypes.c_double]
    L.or_mx_exponent.restype = ctypes.c_int32
    L.or_mx_quant_block32.argtypes = [_f32p, _u8p, _u8p]
    L.or_pack_idx_mx.argtypes = [_u16p, _i32p, _i64p, ctypes.c_int64, _u8p, _i32p, ctypes.c_int32]
    L.or_read_idx_mx.argtypes = [_u8p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _f64p]
    L.or_index_score_mx.argtypes = [_u16p, _f32p, ctypes.c_int32, _u8p, _i32p, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, _f64p, _f64p]
    L.or_block_pool.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i32p]
    L.or_block_pool.restype = ctypes.c_int64
    L.or_index_score_at.argtypes = [_u16p, _f32p, ctypes.c_int32, _u8p, _i32p, ctypes.c_int32, ctypes.c_int32,
                                    _i32p, ctypes.c_int64, ctypes.c_int32, _f64p, _f64p]
    L.or_index_score_bf16.argtypes = [_u16p, _f32p, ctypes.c_int32, _u16p, ctypes.c_int64, _f64p]
    for f in ("or_quant_block16", "or_quant_vector", "or_pack_kv", "or_read_main", "or_read_idx",
              "or_index_score", "or_topk", "or_attention", "or_attention_ext", "or_pack_window",
              "or_read_window", "or_attention_ring", "or_mx_quant_block32", "or_pack_idx_mx",
              "or_read_idx_mx", "or_index_score_mx", "or_index_score_at", "or_index_score_bf16"):
        getattr(L, f).restype = None


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(t)


def _bt(block_table):
    if block_table is None:
        return None, None
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    return bt, _p(bt, _i32p)


# ----------------------------------------------------------------- codecs [P1]

def e4m3_decode(code: int) -> float:
    """E4M3 value of an 8-bit code (bias 7, subnormals, single NaN, max 448) [P1 precision primer]."""
    return lib().or_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(x: float) -> int:
    """Round-to-nearest-even onto the E4M3 grid with saturation to +-448 [P1 precision primer]."""
    return lib().or_e4m3_encode(float(x))


def e2m1_decode(code: int) -> float:
    """E2M1 value: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; bit 3 = sign [P1 precision primer]."""
    return lib().or_e2m1_decode(int(code) & 0xF)


def e2m1_encode(y: float) -> int:
    """Nearest E2M1 magnitude, ties to even, |y| > 6 -> 6, sign kept [P1 precision primer]."""
    return lib().or_e2m1_encode(float(y))


def quant_block16(x) -> tuple[np.ndarray, int]:
    """Codes and scale code of one 16-channel block: E4M3 scale = block max / 6 [P1 "DeepSeek-V4.1"]."""
    xf = np.ascontiguousarray(x, dtype=np.float32)
    assert xf.shape == (16,)
    codes = np.zeros(16, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().or_quant_block16(_p(xf, _f32p), _p(codes, _u8p), _p(sc, _u8p))
    return codes, int(sc[0])


def quant_vector(x) -> tuple[np.ndarray, np.ndarray]:
    """Block-16 codes [n] and scale codes [n/16] of an fp32 vector [P1 "DeepSeek-V4.1"]."""
    xf = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert xf.size % 16 == 0
    codes = np.zeros(xf.size, np.uint8)
    scales = np.zeros(xf.size // 16, np.uint8)
    lib().or_quant_vector(_p(xf, _f32p), xf.size // 16, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def dequant_vector(codes, scales) -> np.ndarray:
    """v = e2m1(code) * e4m3(scale of its 16-block), fp64."""
    L = lib()
    out = np.array([L.or_e2m1_decode(int(c)) for c in codes], dtype=np.float64)
    sc = np.array([L.or_e4m3_decode(int(s)) for s in scales], dtype=np.float64)
    return out * np.repeat(sc, 16)


# --------------------------------------------------------------- cache [P1][P3]

def alloc_pages(n_pages: int) -> tuple[np.ndarray, np.ndarray]:
    """Zeroed main-KV and indexer-K page arrays."""
    return (np.zeros(n_pages * KV_PAGE_BYTES, np.uint8), np.zeros(n_pages * IDX_PAGE_BYTES, np.uint8))


def pack_kv(latent_bf16, idx_key_bf16, req, pos, kv_pages, idx_pages, block_table=None, max_pages=0):
    """Quantise and write n new entries: 288 B main KV + 72 B indexer K each [P1 "DeepSeek-V4.1"; P3 §3].

    latent_bf16: uint16 [n][512] (bf16 bit patterns); idx_key_bf16: uint16 [n][128].
    """
    lat = np.ascontiguousarray(latent_bf16, dtype=np.uint16)
    key = np.ascontiguousarray(idx_key_bf16, dtype=np.uint16)
    req = np.ascontiguousarray(req, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    n = lat.shape[0]
    assert lat.shape == (n, D) and key.shape == (n, DI) and req.shape == (n,) and pos.shape == (n,)
    bt, btp = _bt(block_table)
    lib().or_pack_kv(_p(lat, _u16p), _p(key, _u16p), _p(req, _i32p), _p(pos, _i64p), n,
                     _p(kv_pages, _u8p), _p(idx_pages, _u8p), btp, int(max_pages))


def read_main(kv_pages, r, s, block_table=None, max_pages=0) -> np.ndarray:
    out = np.zeros(D, np.float64)
    bt, btp = _bt(block_table)
    lib().or_read_main(_p(kv_pages, _u8p), btp, int(max_pages), int(r), int(s), _p(out, _f64p))
    return out


def read_idx(idx_pages, r, s, block_table=None, max_pages=0) -> np.ndarray:
    out = np.zeros(DI, np.float64)
    bt, btp = _bt(block_table)
    lib().or_read_idx(_p(idx_pages, _u8p), btp, int(max_pages), int(r), int(s), _p(out, _f64p))
    return out


# ------------------------------------------------------------ index score [P1][P2]

def index_score(q_idx_bf16, w, idx_pages, r, s0, s1, block_table=None, max_pages=0):
    """I[s] = sum_j w_j ReLU(qhat_j . khat_s / sqrt(128)) for s in [s0, s1), and M[s] (|w| version).

    [P1 "DeepSeek-V3.2", the lightning indexer; P2 "The indexer" and "CSA" scorer code;
    P1 "DeepSeek-V4" "the indexer in four bits": query and key both in FP4.]
    """
    q = np.ascontiguousarray(q_idx_bf16, dtype=np.uint16)
    heads = q.shape[0]
    assert q.shape == (heads, DI)
    wf = np.ascontiguousarray(w, dtype=np.float32)
    assert wf.shape == (heads,)
    n = max(0, int(s1) - int(s0))
    I = np.zeros(n, np.float64)
    M = np.zeros(n, np.float64)
    bt, btp = _bt(block_table)
    if n:
        lib().or_index_score(_p(q, _u16p), _p(wf, _f32p), heads, _p(idx_pages, _u8p), btp,
                             int(max_pages), int(r), int(s0), int(s1), _p(I, _f64p), _p(M, _f64p))
    return I, M


# -------------------------------------------------------------------- top-k [P2]

def topk(scores, k: int = 512) -> np.ndarray:
    """k largest scores (ties -> lower index), returned ascending, -1 padded [P2 "CSA" sentinel]."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    out = np.zeros(k, np.int32)
    lib().or_topk(_p(s, _f32p), s.size, int(k), _p(out, _i32p))
    return out


# ------------------------------------------------------------- attention [P1][P2]

def attention(q_bf16, idx, kv_pages, r, win_bf16, win_len, scale=None, block_table=None, max_pages=0):
    """Shared-KV MQA over the selected entries plus the window rows (K == V), fp64.

    [P1 "DeepSeek-V4": 512 selected entries concatenated with 128 window entries;
    P2 "What replaced MLA": K and V are the same tensor.]  Returns (O [H][512], lse [H]).
    """
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    heads = q.shape[0]
    assert q.shape == (heads, D)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    win = np.ascontiguousarray(win_bf16, dtype=np.uint16).reshape(-1, D)
    assert win.shape[0] >= win_len
    if scale is None:
        scale = D ** -0.5
    O = np.zeros((heads, D), np.float64)
    lse = np.zeros(heads, np.float64)
    bt, btp = _bt(block_table)
    lib().or_attention(_p(q, _u16p), heads, _p(ix, _i32p), ix.size, _p(kv_pages, _u8p), btp,
                       int(max_pages), int(r), _p(win, _u16p), int(win_len), float(scale),
                       _p(O, _f64p), _p(lse, _f64p))
    return O, lse


# ------------------------------------------- sinks and partial RoPE [P2]

def attention_ext(q_bf16, idx, kv_pages, r, win_bf16, win_len, scale=None, sinks=None, rope_cos=None,
                  rope_sin=None, block_table=None, max_pages=0):
    """attention() with per-head sinks and the partial RoPE of the query and output, fp64.

    [P2 "From MLA to DSA to HCA/CSA", "What replaced MLA": the trailing 64 channels of q
    are rotated at the query position (rotate_half pairs channel 448 + i with 480 + i)
    and the output is rotated back with -sin; "The sliding window": one sink logit per
    head joins the softmax and has no value vector.]  sinks: [H] natural-log logits;
    rope_cos / rope_sin: [32] angles of the query position.  Returns (O [H][512], lse [H]).
    """
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    heads = q.shape[0]
    assert q.shape == (heads, D)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    win = np.ascontiguousarray(win_bf16, dtype=np.uint16).reshape(-1, D)
    assert win.shape[0] >= win_len
    if scale is None:
        scale = D ** -0.5
    O = np.zeros((heads, D), np.float64)
    lse = np.zeros(heads, np.float64)
    bt, btp = _bt(block_table)
    sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    assert (rope_cos is None) == (rope_sin is None)
    c = None if rope_cos is None else np.ascontiguousarray(rope_cos, dtype=np.float64)
    s = None if rope_sin is None else np.ascontiguousarray(rope_sin, dtype=np.float64)
    if sk is not None:
        assert sk.shape == (heads,)
    if c is not None:
        assert c.shape == (32,) and s.shape == (32,)
    lib().or_attention_ext(_p(q, _u16p), heads, _p(ix, _i32p), ix.size, _p(kv_pages, _u8p), btp,
                           int(max_pages), int(r), _p(win, _u16p), int(win_len), float(scale),
                           None if sk is None else _p(sk, _f64p), None if c is None else _p(c, _f64p),
                           None if s is None else _p(s, _f64p), _p(O, _f64p), _p(lse, _f64p))
    return O, lse


# ------------------------------------------------------------- FP8 window ring [P1]
WIN, WIN_BYTES = 128, 528


def e8m0_exponent(amax: float) -> int:
    """The window block's scale exponent: the smallest e with amax <= 448 * 2^e, clamped
    to [-127, 127] (an all-zero block: -127)."""
    return int(lib().or_e8m0_exponent(float(amax)))


def alloc_ring(n_req: int) -> np.ndarray:
    """A window ring of W = 128 slots of 528 bytes per request."""
    return np.zeros(n_req * WIN * WIN_BYTES, np.uint8)


def pack_window(rows_bf16, req, pos, ring):
    """Pack bf16 window rows into slot pos mod 128 of each request's ring.

    [P1 "Four bits for the main KV, eight for the window": 512 E4M3 bytes plus 16 E8M0
    scales, 528 bytes; "Definition and the bounded cache": position i in slot i mod W.]
    """
    rows = np.ascontiguousarray(rows_bf16, dtype=np.uint16).reshape(-1, D)
    req = np.ascontiguousarray(req, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    assert rows.shape[0] == req.size == pos.size
    lib().or_pack_window(_p(rows, _u16p), _p(req, _i32p), _p(pos, _i64p), rows.shape[0], _p(ring, _u8p))


def read_window(ring, r: int, p: int) -> np.ndarray:
    """Dequantised window entry of position p of request r (fp64, exact)."""
    out = np.zeros(D, np.float64)
    lib().or_read_window(_p(ring, _u8p), int(r), int(p), _p(out, _f64p))
    return out


def attention_ring(q_bf16, idx, kv_pages, r, ring, win_pos, win_len, scale=None, sinks=None, rope_cos=None,
                   rope_sin=None, block_table=None, max_pages=0):
    """attention_ext() with the window keys taken from the FP8 ring: the entries of
    positions win_pos - win_len + 1 .. win_pos of request r.  Returns (O [H][512], lse [H])."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    heads = q.shape[0]
    assert q.shape == (heads, D)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    if scale is None:
        scale = D ** -0.5
    O = np.zeros((heads, D), np.float64)
    lse = np.zeros(heads, np.float64)
    bt, btp = _bt(block_table)
    sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    c = None if rope_cos is None else np.ascontiguousarray(rope_cos, dtype=np.float64)
    s = None if rope_sin is None else np.ascontiguousarray(rope_sin, dtype=np.float64)
    lib().or_attention_ring(_p(q, _u16p), heads, _p(ix, _i32p), ix.size, _p(kv_pages, _u8p), btp,
                            int(max_pages), int(r), _p(ring, _u8p), int(win_pos), int(win_len), float(scale),
                            None if sk is None else _p(sk, _f64p), None if c is None else _p(c, _f64p),
                            None if s is None else _p(s, _f64p), _p(O, _f64p), _p(lse, _f64p))
    return O, lse


# ------------------------------------------------ MXFP4 indexer key [P1][P3][P4]

def mx_exponent(amax: float) -> int:
    """E8M0 exponent of an MXFP4 block: the smallest e with amax <= 6 * 2^e, clamped to
    [-127, 127] (-127 for an all-zero block) [P1 precision primer, MX formats and E8M0]."""
    return int(lib().or_mx_exponent(float(amax)))


def mx_quant_block32(x) -> tuple[np.ndarray, int]:
    """E2M1 codes [32] and E8M0 code (e + 127) of one 32-element MXFP4 block."""
    xf = np.ascontiguousarray(x, dtype=np.float32)
    assert xf.shape == (32,)
    codes = np.zeros(32, np.uint8)
    sc = np.zeros(1, np.uint8)
    lib().or_mx_quant_block32(_p(xf, _f32p), _p(codes, _u8p), _p(sc, _u8p))
    return codes, int(sc[0])


def alloc_idx_mx_pages(n_pages: int) -> np.ndarray:
    """Zeroed MXFP4 indexer-K pages (8704 B = 128 x 68 each)."""
    return np.zeros(n_pages * IDX_MX_PAGE_BYTES, np.uint8)


def pack_idx_mx(idx_key_bf16, req, pos, idx_pages, block_table=None, max_pages=0):
    """Write n indexer keys (uint16 bf16 bits [n][128]) as 68-byte MXFP4 entries
    [P1 "DeepSeek-V4"; P4 "What's in a cell": 64 B of nibbles + four E8M0 scales]."""
    key = np.ascontiguousarray(idx_key_bf16, dtype=np.uint16)
    req = np.ascontiguousarray(req, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    n = key.shape[0]
    assert key.shape == (n, DI) and req.shape == (n,) and pos.shape == (n,)
    bt, btp = _bt(block_table)
    lib().or_pack_idx_mx(_p(key, _u16p), _p(req, _i32p), _p(pos, _i64p), n, _p(idx_pages, _u8p), btp,
                         int(max_pages))


def read_idx_mx(idx_pages, r, s, block_table=None, max_pages=0) -> np.ndarray:
    """Dequantised MXFP4 key of entry s of request r: e2m1(code) * 2^(scale code - 127)."""
    out = np.zeros(DI, np.float64)
    bt, btp = _bt(block_table)
    lib().or_read_idx_mx(_p(idx_pages, _u8p), btp, int(max_pages), int(r), int(s), _p(out, _f64p))
    return out


def index_score_mx(q_idx_bf16, w, idx_pages, r, s0, s1, block_table=None, max_pages=0):
    """index_score over MXFP4 keys with the query quantised to MXFP4 (fp64 sums)."""
    q = np.ascontiguousarray(q_idx_bf16, dtype=np.uint16)
    heads = q.shape[0]
    assert q.shape == (heads, DI)
    wf = np.ascontiguousarray(w, dtype=np.float32)
    assert wf.shape == (heads,)
    n = max(0, int(s1) - int(s0))
    I = np.zeros(n, np.float64)
    M = np.zeros(n, np.float64)
    bt, btp = _bt(block_table)
    if n:
        lib().or_index_score_mx(_p(q, _u16p), _p(wf, _f32p), heads, _p(idx_pages, _u8p), btp,
                                int(max_pages), int(r), int(s0), int(s1), _p(I, _f64p), _p(M, _f64p))
    return I, M


# ------------------------------------------ hierarchical sparse indexer [P1][P4]
POOL_BLOCK = 8       # positions per block [P1 "The hierarchical indexer"]
POOL_BLOCKS = 2048   # blocks kept
POOL = POOL_BLOCK * POOL_BLOCKS


def block_pool(scores, n_visible: int, block: int = POOL_BLOCK, keep: int = POOL_BLOCKS) -> tuple[np.ndarray, int]:
    """Candidate pool of a Full layer's score row: the visible positions of the `keep`
    blocks of `block` positions with the largest block maxima (ties -> lower block),
    ascending, -1 padded to keep * block; and their count [P1 "The hierarchical indexer";
    P4 "The Hierarchical Sparse Indexer"]."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    assert s.size >= n_visible
    pool = np.zeros(keep * block, np.int32)
    n = lib().or_block_pool(_p(s, _f32p), int(n_visible), int(block), int(keep), _p(pool, _i32p))
    return pool, int(n)


def index_score_at(q_idx_bf16, w, idx_pages, r, positions, mx=False, block_table=None, max_pages=0):
    """index_score (or index_score_mx) at the listed positions of request r."""
    q = np.ascontiguousarray(q_idx_bf16, dtype=np.uint16)
    heads = q.shape[0]
    wf = np.ascontiguousarray(w, dtype=np.float32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    I = np.zeros(pos.size, np.float64)
    M = np.zeros(pos.size, np.float64)
    bt, btp = _bt(block_table)
    if pos.size:
        lib().or_index_score_at(_p(q, _u16p), _p(wf, _f32p), heads, _p(idx_pages, _u8p), btp, int(max_pages),
                                int(r), _p(pos, _i32p), pos.size, int(bool(mx)), _p(I, _f64p), _p(M, _f64p))
    return I, M


def pool_topk(pool_scores, pool, n: int, k: int = 512) -> np.ndarray:
    """A Reindex layer's own top-k inside the pool: the k largest of the pool's scores
    (slot i scores position pool[i]; ties -> lower position, as the pool is ascending),
    returned as positions ascending, -1 padded [P4 "The Hierarchical Sparse Indexer"]."""
    slots = topk(np.ascontiguousarray(pool_scores, dtype=np.float32)[:n], k)
    return np.where(slots >= 0, np.asarray(pool)[np.maximum(slots, 0)], -1).astype(np.int32)


def index_score_bf16(q_idx_bf16, w, keys_bf16) -> np.ndarray:
    """The index score from the unquantised bf16 query and keys (fp64): the reference for
    the recall of the FP4 selection [P1 "DeepSeek-V4", 99.7 % recall quoted for V4]."""
    q = np.ascontiguousarray(q_idx_bf16, dtype=np.uint16)
    k = np.ascontiguousarray(keys_bf16, dtype=np.uint16)
    heads = q.shape[0]
    wf = np.ascontiguousarray(w, dtype=np.float32)
    I = np.zeros(k.shape[0], np.float64)
    lib().or_index_score_bf16(_p(q, _u16p), _p(wf, _f32p), heads, _p(k, _u16p), k.shape[0], _p(I, _f64p))
    return I
