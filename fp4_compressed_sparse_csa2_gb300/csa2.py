"""Thin ctypes binding of libcsa2 (include/csa2.h): argument marshalling only.

Every function takes torch tensors on the current CUDA device (PyTorch provides the
device memory and the stream) and forwards raw pointers to the C ABI; all work runs in
the library's CUDA kernels.  There is no CPU fallback: importing this module without
the built library raises immediately.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

# sizes fixed by the pages (mirrors the enum in include/csa2.h)
D, DI, BLOCK = 512, 128, 16
KV_BYTES, IDX_BYTES, WIN_BYTES, IDX_MX_BYTES = 288, 72, 528, 68
TOPK, WIN, HEADS, PAGE = 512, 128, 64, 128
KV_PAGE_BYTES, IDX_PAGE_BYTES, IDX_MX_PAGE_BYTES = PAGE * KV_BYTES, PAGE * IDX_BYTES, PAGE * IDX_MX_BYTES
IDX_E4M3_16, IDX_MXFP4 = 0, 1  # indexer-K formats (csa2_cache.idx_format)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_DEVICE = range(7)
TRACE_KINDS = {"pack": 0, "index": 1, "topk_hist": 2, "topk_select": 3, "topk_final": 4, "attn": 5, "topk": 6,
               "pool": 7, "pool_gather": 8, "pool_map": 9, "pool_bmax": 10,
               "pack_window": 12}
POOL_BLOCK, POOL_BLOCKS, POOL = 8, 2048, 16384  # hierarchical indexer: block, blocks kept, pool positions


class Csa2Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"csa2 status {status}: {msg}")
        self.status = status


class csa2_cache(ctypes.Structure):
    _fields_ = [("kv", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("max_pages", ctypes.c_int32), ("n_pages", ctypes.c_int32), ("idx_format", ctypes.c_int32)]


class csa2_step(ctypes.Structure):
    _fields_ = [("n_q", ctypes.c_int64), ("heads", ctypes.c_int32), ("heads_I", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("group", ctypes.c_int32), ("t_max", ctypes.c_int64),
                ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("req", ctypes.c_void_p), ("n_visible", ctypes.c_void_p), ("window", ctypes.c_void_p),
                ("win_start", ctypes.c_void_p), ("win_len", ctypes.c_void_p), ("n_new", ctypes.c_int64),
                ("new_latent", ctypes.c_void_p), ("new_idx_key", ctypes.c_void_p), ("new_req", ctypes.c_void_p),
                ("new_pos", ctypes.c_void_p), ("cache", csa2_cache), ("topk_idx", ctypes.c_void_p),
                ("scores", ctypes.c_void_p), ("ld", ctypes.c_int64), ("softmax_scale", ctypes.c_float),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("sinks", ctypes.c_void_p),
                ("rope_cos", ctypes.c_void_p), ("rope_sin", ctypes.c_void_p), ("win_ring", ctypes.c_void_p),
                ("win_ring_reqs", ctypes.c_int32), ("pool", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libcsa2.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.csa2_last_error.restype = ctypes.c_char_p
    L.csa2_workspace_bytes.argtypes = [i64, i32, i64, i32]
    L.csa2_workspace_bytes.restype = sz
    L.csa2_workspace_bytes_pool.argtypes = [i64, i32, i64, i32]
    L.csa2_workspace_bytes_pool.restype = sz
    L.csa2_pack_kv.argtypes = [vp, vp, vp, vp, i64, ctypes.POINTER(csa2_cache), vp, sz, vp]
    L.csa2_index_score.argtypes = [vp, vp, i32, vp, vp, i64, i32, i64, ctypes.POINTER(csa2_cache), vp, i64, vp,
                                   sz, vp]
    L.csa2_topk.argtypes = [vp, i64, vp, i64, i64, i32, vp, vp, sz, vp]
    L.csa2_pack_window.argtypes = [vp, vp, vp, i64, vp, i32, vp, sz, vp]
    for f in ("csa2_sparse_attn_full", "csa2_sparse_attn_reindex", "csa2_sparse_attn_reuse"):
        getattr(L, f).argtypes = [ctypes.POINTER(csa2_step), vp, sz, vp]
    L.csa2_topk_noalloc.argtypes = [vp, i64, vp, i64, i64, i32, vp, vp]
    L.csa2_topk_noalloc.restype = ctypes.c_int
    L.csa2_debug_set_wait_limit.argtypes = [ctypes.c_uint64]
    L.csa2_debug_set_wait_limit.restype = ctypes.c_int
    L.csa2_probe_mma.argtypes = [i32, i32, i32, i32, i32, vp, vp]
    L.csa2_probe_mma.restype = ctypes.c_int
    L.csa2_topk_noalloc_check.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    L.csa2_topk_noalloc_check.restype = ctypes.c_int
    L.csa2_check.argtypes = [vp, vp, ctypes.POINTER(i32)]
    L.csa2_launch_count.restype = i64
    L.csa2_trace_enable.argtypes = [i32]
    L.csa2_trace_read.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
    for f in ("csa2_pack_kv", "csa2_pack_window", "csa2_index_score", "csa2_topk", "csa2_sparse_attn_full",
              "csa2_sparse_attn_reindex", "csa2_sparse_attn_reuse", "csa2_check", "csa2_trace_enable",
              "csa2_trace_read"):
        getattr(L, f).restype = ctypes.c_int
    return L


lib = _load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int):
    if status != OK:
        raise Csa2Error(status, lib.csa2_last_error().decode())


def make_cache(kv: torch.Tensor, idx: torch.Tensor, max_pages: int, block_table: torch.Tensor | None = None,
               idx_format: int = IDX_E4M3_16):
    """csa2_cache over uint8 page arrays kv [n_pages*36864] and idx [n_pages*9216]
    (or [n_pages*8704] with idx_format = IDX_MXFP4)."""
    n_pages = kv.numel() // KV_PAGE_BYTES
    assert idx.numel() // (IDX_MX_PAGE_BYTES if idx_format == IDX_MXFP4 else IDX_PAGE_BYTES) == n_pages
    c = csa2_cache(_ptr(kv), _ptr(idx), _ptr(block_table), int(max_pages), int(n_pages), int(idx_format))
    c._keep = (kv, idx, block_table)
    return c


def workspace_bytes(n_q: int, heads_I: int, t_max: int, scores_in_ws: bool, pool: bool = False) -> int:
    f = lib.csa2_workspace_bytes_pool if pool else lib.csa2_workspace_bytes
    return int(f(int(n_q), int(heads_I), int(t_max), int(bool(scores_in_ws))))


def alloc_workspace(n_q: int, heads_I: int, t_max: int, scores_in_ws: bool, device="cuda",
                    pool: bool = False) -> torch.Tensor:
    n = workspace_bytes(n_q, heads_I, t_max, scores_in_ws, pool)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def pack_kv(latent, idx_key, req, pos, cache: csa2_cache, ws, stream=None):
    n = 0 if latent is None else latent.shape[0]
    _check(lib.csa2_pack_kv(_ptr(latent), _ptr(idx_key), _ptr(req), _ptr(pos), n, ctypes.byref(cache), _ptr(ws),
                            ws.numel(), _stream(stream)))


def pack_window(rows, req, pos, ring, n_ring, ws, stream=None):
    """FP8 window entries of bf16 rows [n][512] into slot pos % 128 of each request's ring
    (uint8 [n_ring * 128 * 528])."""
    n = 0 if rows is None else rows.shape[0]
    _check(lib.csa2_pack_window(_ptr(rows), _ptr(req), _ptr(pos), n, _ptr(ring), int(n_ring), _ptr(ws), ws.numel(),
                                _stream(stream)))


def index_score(q_idx, w, heads_I, req, n_visible, n_q, group, t_max, cache, scores, ld, ws, stream=None):
    _check(lib.csa2_index_score(_ptr(q_idx), _ptr(w), int(heads_I), _ptr(req), _ptr(n_visible), int(n_q),
                                int(group), int(t_max), ctypes.byref(cache), _ptr(scores), int(ld), _ptr(ws),
                                ws.numel(), _stream(stream)))


def topk(scores, ld, n_visible, n_q, t_max, k, out_idx, ws, stream=None):
    _check(lib.csa2_topk(_ptr(scores), int(ld), _ptr(n_visible), int(n_q), int(t_max), int(k), _ptr(out_idx),
                         _ptr(ws), ws.numel(), _stream(stream)))


def topk_noalloc(scores, ld, n_visible, n_q, t_max, k, out_idx, stream=None):
    """csa2_topk without a workspace: scratch is a fixed array inside the library (n_q <= 128)."""
    _check(lib.csa2_topk_noalloc(_ptr(scores), int(ld), _ptr(n_visible), int(n_q), int(t_max), int(k),
                                 _ptr(out_idx), _stream(stream)))


def topk_noalloc_check(stream=None) -> tuple[int, int]:
    """(status, info) of the fixed array's error word after the last csa2_topk_noalloc; clears it."""
    info = ctypes.c_int32(0)
    st = lib.csa2_topk_noalloc_check(_stream(stream), ctypes.byref(info))
    return st, info.value


def make_step(*, n_q, t_max, q, req, n_visible, window, win_start, win_len, cache, topk_idx, out, q_idx=None,
              w=None, heads_I=64, group=1, n_new=0, new_latent=None, new_idx_key=None, new_req=None, new_pos=None,
              scores=None, ld=0, softmax_scale=0.0, lse=None, sinks=None, rope_cos=None,
              rope_sin=None, win_ring=None, win_ring_reqs=0, pool=None) -> csa2_step:
    s = csa2_step(int(n_q), HEADS, int(heads_I), TOPK, int(group), int(t_max), _ptr(q), _ptr(q_idx), _ptr(w),
                  _ptr(req), _ptr(n_visible), _ptr(window), _ptr(win_start), _ptr(win_len), int(n_new),
                  _ptr(new_latent), _ptr(new_idx_key), _ptr(new_req), _ptr(new_pos), cache, _ptr(topk_idx),
                  _ptr(scores), int(ld), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(sinks), _ptr(rope_cos),
                  _ptr(rope_sin), _ptr(win_ring), int(win_ring_reqs), _ptr(pool))
    s._keep = (q, req, n_visible, window, win_start, win_len, cache, topk_idx, out, q_idx, w, new_latent,
               new_idx_key, new_req, new_pos, scores, lse, sinks, rope_cos, rope_sin, win_ring, pool)
    return s


def sparse_attn_full(step: csa2_step, ws, stream=None):
    _check(lib.csa2_sparse_attn_full(ctypes.byref(step), _ptr(ws), ws.numel(), _stream(stream)))


def sparse_attn_reindex(step: csa2_step, ws, stream=None):
    _check(lib.csa2_sparse_attn_reindex(ctypes.byref(step), _ptr(ws), ws.numel(), _stream(stream)))


def sparse_attn_reuse(step: csa2_step, ws, stream=None):
    _check(lib.csa2_sparse_attn_reuse(ctypes.byref(step), _ptr(ws), ws.numel(), _stream(stream)))


def check(ws, stream=None) -> tuple[int, int]:
    """(status, info) of the device-side error word; clears it.  Synchronises the stream."""
    info = ctypes.c_int32(0)
    st = lib.csa2_check(_ptr(ws), _stream(stream), ctypes.byref(info))
    return st, info.value


def probe_mma(kind: int, n: int, iters: int, issuers: int, n_ctas: int, cycles, stream=None):
    """Tensor-core throughput probe: cycles (int64 [n_ctas], device) per CTA for `iters` MMAs
    of M = 128 and the given N per issuer (kind 0 f16, 1 NVFP4)."""
    _check(lib.csa2_probe_mma(int(kind), int(n), int(iters), int(issuers), int(n_ctas), _ptr(cycles), _stream(stream)))


def debug_set_wait_limit(ns: int):
    """Bound (ns) of the pipeline waits of kernels launched afterwards; 0 = the default 2 s."""
    _check(lib.csa2_debug_set_wait_limit(int(ns)))


def launch_count() -> int:
    return int(lib.csa2_launch_count())


def trace_enable(on: bool):
    _check(lib.csa2_trace_enable(int(bool(on))))


def trace_read(kind: str) -> tuple[float, int]:
    ms, n = ctypes.c_double(0), ctypes.c_int64(0)
    _check(lib.csa2_trace_read(TRACE_KINDS[kind], ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value
