"""The C-ABI library builds, loads without a GPU and exports every entry point that
include/csa2.h declares; the binding's constants match the header's."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z_0-9]+)\s*\(", src)))


def _lib():
    from fp4_compressed_sparse_csa2_gb300 import build
    return ctypes.CDLL(build.build())


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert {"csa2_pack_kv", "csa2_index_score", "csa2_topk", "csa2_sparse_attn_full", "csa2_sparse_attn_reindex",
            "csa2_sparse_attn_reuse", "csa2_workspace_bytes", "csa2_last_error", "csa2_check"} <= set(names)
    L = _lib()
    for n in names:
        assert hasattr(L, n), n


def test_header_constants_match_binding():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    consts = dict((k, int(v)) for k, v in re.findall(r"(CSA2_[A-Z_]+)\s*=\s*(\d+)", src))
    _lib()
    from fp4_compressed_sparse_csa2_gb300 import csa2
    assert consts["CSA2_KV_BYTES"] == csa2.KV_BYTES == 288
    assert consts["CSA2_IDX_BYTES"] == csa2.IDX_BYTES == 72
    assert consts["CSA2_PAGE"] * 288 == consts["CSA2_KV_PAGE_BYTES"] == csa2.KV_PAGE_BYTES
    assert consts["CSA2_PAGE"] * 72 == consts["CSA2_IDX_PAGE_BYTES"] == csa2.IDX_PAGE_BYTES
    assert consts["CSA2_TOPK"] == 512 and consts["CSA2_WIN"] == 128 and consts["CSA2_HEADS"] == 64
    assert consts["CSA2_OK"] == 0


def test_workspace_and_validation_on_host():
    _lib()
    from fp4_compressed_sparse_csa2_gb300 import csa2
    n = csa2.workspace_bytes(64, 64, 131072, True)
    assert n >= 64 * 131072 * 4 and n % 256 == 0
    assert csa2.workspace_bytes(64, 64, 131072, False) < n
    # argument validation fails before any launch (no GPU needed)
    st = csa2.lib.csa2_topk(None, 0, None, 1, 10, 100, None, None, 0, None)
    assert st == csa2.ERR_UNSUPPORTED and b"512" in csa2.lib.csa2_last_error()
    st = csa2.lib.csa2_sparse_attn_reuse(None, None, 0, None)
    assert st == csa2.ERR_INVALID_ARG
