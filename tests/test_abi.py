"""The C-ABI library loads and exports every symbol include/pkv.h declares.

Runs without a GPU: only host-side calls (versions, status strings, argument
checks that fail before any CUDA work) are made.
"""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


def _declared():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", src)))


def test_header_declares_the_path():
    names = _declared()
    for must in ["pkv_write_kv", "pkv_attn_decode", "pkv_attn_varlen", "pkv_copy_blocks",
                 "pkv_alloc_create", "pkv_seq_append"]:
        assert must in names


def test_library_exports_every_declared_symbol():
    from pagedattention_decode_gb300 import _native
    L = _native.lib()
    names = _declared()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # and the binding knows the signature of each one
    assert set(names) == set(_native.SIGNATURES), set(names) ^ set(_native.SIGNATURES)


def test_version_and_status_strings():
    from pagedattention_decode_gb300 import _native
    L = _native.lib()
    assert L.pkv_abi_version() == 1
    assert L.pkv_status_string(0) == b"PKV_OK"
    assert L.pkv_status_string(5) == b"PKV_ERR_EXHAUSTED"


def test_host_side_argument_checks_need_no_gpu():
    from pagedattention_decode_gb300 import _native
    L = _native.lib()
    st = L.pkv_write_kv(None, None, 0, None, 4, None, None, None)
    assert st == 1 and b"NULL" in L.pkv_last_error()
    c = _native.PkvCache(16, 16, 8, 16, 2, 64, 7)  # bad dtype
    st = L.pkv_attn_decode(None, 0, ctypes.byref(c), None, 0, None, 1, 2, 1.0, None, 2, None, 0, None, None)
    assert st == 2
    c = _native.PkvCache(16, 16, 8, 16, 2, 96, 0)  # head_dim 96 not compiled
    st = L.pkv_attn_decode(16, 192, ctypes.byref(c), 16, 1, 16, 1, 2, 1.0, 16, 2, 16, 0, None, None)
    assert st == 9
    pairs = (ctypes.c_int64 * 4)(1, 2, 2, 3)
    assert L.pkv_check_copy_pairs(pairs, 2, 8) == 1  # 2 is both a dst and a src
    pairs = (ctypes.c_int64 * 4)(1, 2, 3, 4)
    assert L.pkv_check_copy_pairs(pairs, 2, 8) == 0
    pairs = (ctypes.c_int64 * 2)(1, 9)
    assert L.pkv_check_copy_pairs(pairs, 1, 8) == 4


def test_varlen_with_no_query_rows_is_a_host_side_no_op():
    """total_q == 0 (every sequence's row set empty): the call returns PKV_OK
    with NULL q / out before any device work (it needs no GPU); a negative
    total_q is refused."""
    from pagedattention_decode_gb300 import _native
    L = _native.lib()
    c = _native.PkvCache(16, 32, 8, 16, 2, 64, 0)  # fp16 pool geometry; never dereferenced here
    st = L.pkv_attn_varlen(None, 8 * 64, ctypes.byref(c), None, 1, None, None, 3, 0, 0, 8, 0.125, 1, None, 2,
                           None, 0, None, None)
    assert st == 0, L.pkv_last_error()
    st = L.pkv_attn_varlen(None, 8 * 64, ctypes.byref(c), None, 1, None, None, 3, -1, 0, 8, 0.125, 1, None, 2,
                           None, 0, None, None)
    assert st == 1
