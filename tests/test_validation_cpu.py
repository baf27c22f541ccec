"""The C ABI's synchronous argument validation, on the host (no GPU): every call that gets
a bad size, an unsupported shape, a NULL or misaligned pointer, a short or misaligned
workspace, a t_max beyond the cache, an unknown key format or a misuse of the candidate
pool returns its status and a message before anything is launched."""
import ctypes

import pytest

A = 0x7F0000000000          # a 256-byte aligned stand-in address (never dereferenced)
MIS = A + 8                 # misaligned by 8 bytes


@pytest.fixture(scope="module")
def lib():
    from fp4_compressed_sparse_csa2_gb300 import build
    build.build()
    from fp4_compressed_sparse_csa2_gb300 import csa2
    return csa2


def _p(x):
    return ctypes.c_void_p(x)


def _cache(csa2, **kw):
    c = csa2.csa2_cache(_p(A), _p(A), None, 4, 8, 0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _status(csa2, st, want, text=None):
    assert st == want, (st, csa2.lib.csa2_last_error())
    if text:
        assert text.encode() in csa2.lib.csa2_last_error(), csa2.lib.csa2_last_error()


def test_topk_arguments(lib):
    c = lib
    L = c.lib
    _status(c, L.csa2_topk(_p(A), 1024, _p(A), 2, 1000, 256, _p(A), _p(A), 1 << 20, None), c.ERR_UNSUPPORTED, "512")
    _status(c, L.csa2_topk(_p(A), 1000 - 4, _p(A), 2, 1000, 512, _p(A), _p(A), 1 << 20, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_topk(_p(A), 1002, _p(A), 2, 1000, 512, _p(A), _p(A), 1 << 20, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_topk(_p(MIS), 1024, _p(A), 2, 1000, 512, _p(A), _p(A), 1 << 20, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_topk(None, 1024, _p(A), 2, 1000, 512, _p(A), _p(A), 1 << 20, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_topk(_p(A), 1024, _p(A), -1, 1000, 512, _p(A), _p(A), 1 << 20, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_topk(_p(A), 1024, _p(A), 2, 1000, 512, _p(A), None, 1 << 20, None), c.ERR_WORKSPACE)
    _status(c, L.csa2_topk(_p(A), 1024, _p(A), 2, 1000, 512, _p(A), _p(MIS), 1 << 20, None), c.ERR_WORKSPACE)
    _status(c, L.csa2_topk(_p(A), 1024, _p(A), 2, 1000, 512, _p(A), _p(A), 16, None), c.ERR_WORKSPACE, "smaller")
    _status(c, L.csa2_topk_noalloc(_p(A), 1024, _p(A), 129, 1000, 512, _p(A), None), c.ERR_WORKSPACE, "128")


def test_index_score_arguments(lib):
    c = lib
    L = c.lib
    ws = c.workspace_bytes(2, 64, 512, False)
    good = _cache(c)

    def call(cache, heads=64, group=1, t_max=512, ld=512, q=A, scores=A, wsp=A, wsb=ws):
        return L.csa2_index_score(_p(q), _p(A), heads, _p(A), _p(A), 2, group, t_max, ctypes.byref(cache),
                                  _p(scores) if scores else None, ld, _p(wsp) if wsp else None, wsb, None)
    _status(c, call(good, heads=48), c.ERR_UNSUPPORTED)
    _status(c, call(good, group=3), c.ERR_UNSUPPORTED)
    _status(c, call(good, t_max=4 * 128 + 1, ld=1024), c.ERR_INVALID_ARG, "t_max")     # beyond the cache
    _status(c, call(good, q=MIS), c.ERR_INVALID_ARG)
    _status(c, call(good, scores=0), c.ERR_INVALID_ARG)
    _status(c, call(good, ld=500), c.ERR_INVALID_ARG)
    _status(c, call(_cache(c, idx=_p(A + 16))), c.ERR_INVALID_ARG, "cache.idx")
    _status(c, call(_cache(c, max_pages=0)), c.ERR_INVALID_ARG)
    _status(c, call(_cache(c, idx_format=7)), c.ERR_INVALID_ARG, "idx_format")
    _status(c, call(good, wsb=ws - 256), c.ERR_WORKSPACE)
    _status(c, call(good, wsp=MIS), c.ERR_WORKSPACE)
    assert L.csa2_index_score(_p(A), _p(A), 64, _p(A), _p(A), 2, 1, 512, None, _p(A), 512, _p(A), ws, None) \
        == c.ERR_INVALID_ARG


def test_pack_arguments(lib):
    c = lib
    L = c.lib
    good = _cache(c)
    _status(c, L.csa2_pack_kv(_p(A), _p(A), _p(A), _p(A), -1, ctypes.byref(good), _p(A), 256, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_pack_kv(_p(MIS), _p(A), _p(A), _p(A), 3, ctypes.byref(good), _p(A), 256, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_pack_kv(_p(A), _p(A), None, _p(A), 3, ctypes.byref(good), _p(A), 256, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_pack_kv(_p(A), _p(A), _p(A), _p(A), 3, ctypes.byref(_cache(c, kv=_p(A + 64))), _p(A), 256,
                              None), c.ERR_INVALID_ARG, "cache.kv")
    _status(c, L.csa2_pack_kv(_p(A), _p(A), _p(A), _p(A), 3, ctypes.byref(good), _p(A), 64, None), c.ERR_WORKSPACE)
    _status(c, L.csa2_pack_window(_p(A), _p(A), _p(A), 3, _p(A), 0, _p(A), 256, None), c.ERR_INVALID_ARG)
    _status(c, L.csa2_pack_window(_p(A), _p(A), _p(A), 3, _p(MIS), 2, _p(A), 256, None), c.ERR_INVALID_ARG)


def _step(csa2, **kw):
    s = csa2.csa2_step()
    s.n_q, s.heads, s.heads_I, s.topk, s.group, s.t_max = 2, 64, 64, 512, 1, 512
    for f in ("q", "q_idx", "w", "req", "n_visible", "window", "win_start", "win_len", "topk_idx", "out"):
        setattr(s, f, A)
    s.cache = _cache(csa2)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_step_arguments(lib):
    c = lib
    L = c.lib
    big = 1 << 26

    def run(fn, s, wsb=big, wsp=A):
        return getattr(L, fn)(ctypes.byref(s), _p(wsp) if wsp else None, wsb, None)
    _status(c, run("csa2_sparse_attn_full", _step(c, heads=32)), c.ERR_UNSUPPORTED, "heads")
    _status(c, run("csa2_sparse_attn_full", _step(c, topk=256)), c.ERR_UNSUPPORTED, "512")
    _status(c, run("csa2_sparse_attn_reindex", _step(c, heads_I=16)), c.ERR_UNSUPPORTED)
    _status(c, run("csa2_sparse_attn_reuse", _step(c, q=MIS)), c.ERR_INVALID_ARG)
    _status(c, run("csa2_sparse_attn_reuse", _step(c, window=None)), c.ERR_INVALID_ARG, "window")
    _status(c, run("csa2_sparse_attn_reuse", _step(c, rope_cos=A)), c.ERR_INVALID_ARG, "rope")
    _status(c, run("csa2_sparse_attn_reuse", _step(c, out=None)), c.ERR_INVALID_ARG)
    _status(c, run("csa2_sparse_attn_reuse", _step(c, t_max=4 * 128 + 128)), c.ERR_INVALID_ARG, "t_max")
    _status(c, run("csa2_sparse_attn_full", _step(c, n_new=1)), c.ERR_INVALID_ARG, "new_latent")
    _status(c, run("csa2_sparse_attn_reindex", _step(c, scores=A, ld=510)), c.ERR_INVALID_ARG, "ld")
    # candidate pool: aligned, group 1, pool-slot scores need ld >= 16384
    _status(c, run("csa2_sparse_attn_reindex", _step(c, pool=MIS)), c.ERR_INVALID_ARG, "pool")
    _status(c, run("csa2_sparse_attn_reindex", _step(c, pool=A, group=2)), c.ERR_UNSUPPORTED, "group 1")
    _status(c, run("csa2_sparse_attn_reindex", _step(c, pool=A, scores=A, ld=4096)), c.ERR_INVALID_ARG, "16384")
    # workspace
    _status(c, run("csa2_sparse_attn_full", _step(c), wsb=1024), c.ERR_WORKSPACE)
    _status(c, run("csa2_sparse_attn_full", _step(c), wsp=MIS), c.ERR_WORKSPACE)
    need = c.workspace_bytes(2, 64, 512, True)
    need_pool = c.workspace_bytes(2, 64, 512, True, pool=True)
    assert need_pool > need
    _status(c, run("csa2_sparse_attn_full", _step(c, pool=A), wsb=need), c.ERR_WORKSPACE)
    assert L.csa2_check(None, None, None) == c.ERR_WORKSPACE
