"""The C ABI without a GPU: the library loads, exports every declared symbol, and
its host-side argument checks reject bad calls before launching anything."""
import ctypes
import os
import re

import pytest

from sparse_attention_lightning_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_attention_lightning_gb300 import build
    build.build()
    return _abi.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(dsa_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert names == set(_abi.EXPORTS), names ^ set(_abi.EXPORTS)
    for n in names:
        assert hasattr(L, n), n
    assert L.dsa_abi_version() == _abi.ABI_VERSION == 4


def _problem(**kw):
    base = dict(num_seqs=1, total_q=4, total_k=64, max_q_len=4, max_k_len=64, h_idx=4, d_idx=32,
                h=8, d_c=64, d_rope=16, top_k=8, idx_dtype=0, kv_dtype=0, out_dtype=0,
                sm_scale=0.0, cu_q=4096, cu_k=8192)
    base.update(kw)
    return _abi.DsaProblem(**base)


def _ws_size(L, p, op):
    n = ctypes.c_size_t(0)
    rc = L.dsa_workspace_size(ctypes.byref(p), op, ctypes.byref(n))
    return rc, n.value


def test_workspace_sizes(L):
    p = _problem()
    for op in (1, 2, 3, 4, 5):
        rc, n = _ws_size(L, p, op)
        assert rc == 0 and n >= _abi.STATUS_BYTES and n % 256 == 0
    assert _ws_size(L, p, 99)[0] == _abi.DSA_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value,code", [
    ("top_k", 0, _abi.DSA_ERR_UNSUPPORTED), ("top_k", 4096, _abi.DSA_ERR_UNSUPPORTED),
    ("d_idx", 24, _abi.DSA_ERR_UNSUPPORTED), ("h_idx", 0, _abi.DSA_ERR_UNSUPPORTED),
    ("h", 129, _abi.DSA_ERR_UNSUPPORTED), ("d_c", 8, _abi.DSA_ERR_UNSUPPORTED),
    ("d_rope", 8, _abi.DSA_ERR_UNSUPPORTED), ("num_seqs", 0, _abi.DSA_ERR_INVALID_ARG),
    ("max_k_len", 65, _abi.DSA_ERR_INVALID_ARG), ("cu_q", 0, _abi.DSA_ERR_INVALID_ARG),
    ("idx_dtype", 7, _abi.DSA_ERR_INVALID_ARG), ("kv_dtype", 2, _abi.DSA_ERR_UNSUPPORTED),
])
def test_descriptor_checks(L, field, value, code):
    p = _problem(**{field: value})
    assert _ws_size(L, p, _abi.OP_FUSED_FORWARD)[0] == code
    assert L.dsa_last_error()


def test_mxfp8_descriptor(L):
    # MXFP8 scales cover 32 elements: d_idx must be a multiple of 32
    assert _ws_size(L, _problem(idx_dtype=_abi.DSA_MXFP8_E4M3, d_idx=64), 5)[0] == 0
    assert _ws_size(L, _problem(idx_dtype=_abi.DSA_MXFP8_E4M3, d_idx=48), 5)[0] == \
        _abi.DSA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,code", [
    (dict(page_size=48, max_pages=2, num_pages=4, block_table=1 << 16), _abi.DSA_ERR_UNSUPPORTED),
    (dict(page_size=384, max_pages=1, num_pages=4, block_table=1 << 16), _abi.DSA_ERR_UNSUPPORTED),
    (dict(page_size=64, max_pages=1, num_pages=4, block_table=None), _abi.DSA_ERR_INVALID_ARG),
    (dict(page_size=64, max_pages=1, num_pages=4, block_table=(1 << 16) + 4),
     _abi.DSA_ERR_INVALID_ARG),
    (dict(page_size=16, max_pages=3, num_pages=4, block_table=1 << 16), _abi.DSA_ERR_INVALID_ARG),
    (dict(page_size=128, max_pages=1, num_pages=0, block_table=1 << 16), _abi.DSA_ERR_INVALID_ARG),
    (dict(page_size=1 << 14, max_pages=1, num_pages=1 << 17, block_table=1 << 16),
     _abi.DSA_ERR_UNSUPPORTED),
])
def test_paged_descriptor_checks(L, kw, code):
    # page sizes: powers of two >= 16; the block table must exist, be aligned and
    # cover max_k_len (64 keys here); the cache must stay below 2^31 rows
    p = _problem(**kw)
    assert _ws_size(L, p, _abi.OP_FUSED_FORWARD)[0] == code
    assert L.dsa_last_error()
    ok = _problem(page_size=32, max_pages=2, num_pages=3, block_table=1 << 16)
    assert _ws_size(L, ok, _abi.OP_FUSED_FORWARD)[0] == _abi.DSA_OK


def test_pointer_and_workspace_checks_launch_nothing(L):
    p = _problem()
    P = ctypes.byref(p)
    A = 1 << 20  # 16-byte aligned fake addresses: the checks must fail before any use
    # null q_idx
    assert L.dsa_fused_indexer(P, None, A, A, None, None, A, None, A, 1 << 20, None) == 1
    # misaligned k_idx
    assert L.dsa_fused_indexer(P, A, A + 4, A, None, None, A, None, A, 1 << 20, None) == 1
    # FP8 without scales
    p8 = _problem(idx_dtype=2)
    assert L.dsa_indexer_scores(ctypes.byref(p8), A, A, A, None, None, A, 64, A, 256, None) == 1
    # workspace too small / missing
    rc, need = _ws_size(L, p, _abi.OP_FUSED_FORWARD)
    assert L.dsa_fused_forward(P, A, A, A, None, None, A, A, A, None, None, None, A, need - 256,
                               None) == _abi.DSA_ERR_WORKSPACE
    assert L.dsa_sparse_mla_attn(P, A, A, A, A, None, None, 0, None) == _abi.DSA_ERR_WORKSPACE
    # scores leading dimension below max_k_len
    assert L.dsa_topk(P, A, 63, A, None, A, 256, None) == _abi.DSA_ERR_INVALID_ARG


def test_status_strings(L):
    for c in range(6):
        assert L.dsa_status_str(c)
    assert L.dsa_status_str(42) == b"unknown status"
