"""The C-ABI library builds, loads and exports every symbol that
include/grbeam.h declares; host-side argument checks run without a GPU."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from beam_decode_gb300 import binding as B
from beam_decode_gb300.build import LIB, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "grbeam.h")


def header_symbols():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gr_[a-z_0-9]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    build()
    return B.lib()


def test_header_symbols_exported(lib):
    syms = header_symbols()
    assert len(syms) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gr_[a-z_0-9]+)", out))
    missing = [s for s in syms if s not in exported]
    assert not missing, missing
    for s in syms:
        assert hasattr(lib, s)
    assert sorted(B.SYMBOLS) == syms


def test_status_strings(lib):
    for code, name in [(0, "GR_OK"), (-1, "GR_ERR_INVALID_ARG"), (-4, "GR_ERR_STATE"), (-6, "GR_ERR_TIMEOUT"),
                       (-7, "GR_ERR_DEVICE")]:
        assert lib.gr_status_str(code).decode() == name


def _trie_bytes(lib, codes, L, C):
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    n = ctypes.c_size_t()
    st = lib.gr_trie_device_bytes(codes.ctypes.data, codes.shape[0], L, C, ctypes.byref(n))
    return st, n.value


def test_trie_bytes_and_duplicates(lib):
    codes = np.array([[0, 1], [0, 2], [3, 1]])
    st, n = _trie_bytes(lib, codes, 2, 16)
    assert st == 0
    # root + 2 depth-1 nodes, one 16-code mask word each, plus 3 leaves
    assert n >= 3 * 4 + 3 * 4 + 3 * 8
    st, _ = _trie_bytes(lib, np.array([[0, 1], [0, 1]]), 2, 16)
    assert st == B.GR_ERR_INVALID_ARG
    assert "duplicate" in lib.gr_last_error().decode()
    st, _ = _trie_bytes(lib, np.array([[0, 16]]), 2, 16)
    assert st == B.GR_ERR_INVALID_ARG
    st, _ = _trie_bytes(lib, np.array([[0] * 9]), 9, 16)
    assert st == B.GR_ERR_UNSUPPORTED
    st, _ = _trie_bytes(lib, np.array([[0, 1]]), 2, 2000)
    assert st == B.GR_ERR_UNSUPPORTED


def test_trie_create_rejects_bad_buffer(lib):
    codes = np.ascontiguousarray([[0, 1]], dtype=np.int32)
    h = ctypes.c_void_p()
    st = lib.gr_trie_create(codes.ctypes.data, None, 1, 2, 16, None, 0, None, ctypes.byref(h))
    assert st == B.GR_ERR_INVALID_ARG and not h.value
    st = lib.gr_trie_create(codes.ctypes.data, None, 1, 2, 16, ctypes.c_void_p(0x1001), 4096, None, ctypes.byref(h))
    assert st == B.GR_ERR_INVALID_ARG


def _cfg(**over):
    c = dict(n_layers=28, n_q_heads=16, n_kv_heads=8, head_dim=128, vocab=151936,
             code_base=151936 - 768, n_levels=3, codes_per_level=256, pool_tokens=40000)
    c.update(over)
    return B.GrConfig(**c)


@pytest.mark.parametrize("over,code", [
    (dict(head_dim=96), B.GR_ERR_UNSUPPORTED),
    (dict(n_q_heads=24), B.GR_ERR_UNSUPPORTED),
    (dict(n_q_heads=15), B.GR_ERR_INVALID_ARG),
    (dict(code_base=151936 - 700), B.GR_ERR_INVALID_ARG),
    (dict(n_levels=9), B.GR_ERR_UNSUPPORTED),
    (dict(codes_per_level=4096), B.GR_ERR_UNSUPPORTED),
    (dict(pool_tokens=0), B.GR_ERR_INVALID_ARG),
])
def test_workspace_bytes_rejects_config(lib, over, code):
    cfg = _cfg(**over)
    reqs = (B.GrRequest * 1)(B.GrRequest(0, 5000, 256, None))
    n = ctypes.c_size_t()
    assert lib.gr_beam_workspace_bytes(ctypes.byref(cfg), reqs, 1, ctypes.byref(n)) == code


def test_workspace_bytes_rejects_requests(lib):
    cfg = _cfg()
    n = ctypes.c_size_t()
    for req, code in [((0, 5000, 256, None), B.GR_ERR_INVALID_ARG),       # no trie
                      ((39000, 5000, 256, None), B.GR_ERR_INVALID_ARG),   # outside the pool
                      ((0, 5000, 2048, None), B.GR_ERR_CAPACITY),         # beam above 1024
                      ((0, 0, 256, None), B.GR_ERR_INVALID_ARG)]:
        reqs = (B.GrRequest * 1)(B.GrRequest(*req))
        assert lib.gr_beam_workspace_bytes(ctypes.byref(cfg), reqs, 1, ctypes.byref(n)) == code
    assert lib.gr_beam_workspace_bytes(ctypes.byref(cfg), None, 0, ctypes.byref(n)) == B.GR_ERR_INVALID_ARG


def test_null_handles(lib):
    assert lib.gr_beam_advance(None, None) == B.GR_ERR_INVALID_ARG
    assert lib.gr_beam_rewind(None, 1, None) == B.GR_ERR_INVALID_ARG
    assert lib.gr_decode_attn(None, 0, None, None, None) == B.GR_ERR_INVALID_ARG
    assert lib.gr_constrained_topk(None, None, 0, None, None, None, None) == B.GR_ERR_INVALID_ARG
    n = ctypes.c_int()
    assert lib.gr_beam_results(None, 0, None, None, None, ctypes.byref(n), None) == B.GR_ERR_INVALID_ARG
