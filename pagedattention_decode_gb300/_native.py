"""ctypes declarations of libpkv's C ABI (include/pkv.h).

Loading fails loudly: there is no fallback path.  If the library is missing
or stale it is built in-tree first (nvcc, sm_103a).
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

PKV_OK = 0
STATUS = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_DTYPE", 3: "PKV_ERR_SHAPE",
    4: "PKV_ERR_OUT_OF_RANGE", 5: "PKV_ERR_EXHAUSTED", 6: "PKV_ERR_DOUBLE_FREE",
    7: "PKV_ERR_CUDA", 8: "PKV_ERR_WORKSPACE", 9: "PKV_ERR_UNSUPPORTED",
}
PKV_F16, PKV_BF16, PKV_F32 = 0, 1, 2
PKV_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # the fixed scratch of pkv_attn_decode_noalloc (pkv.h)
DEVERR = {"slot": 0x1, "block": 0x2, "pair": 0x4, "timeout": 0x8, "length": 0x10}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message or STATUS.get(status, str(status)))
        self.status = status


class ExhaustedError(PkvError):
    pass


class DoubleFreeError(PkvError, ValueError):
    pass


class PkvCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class PkvCacheI8(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class PkvCounters(ctypes.Structure):
    _fields_ = [("allocs", ctypes.c_int64), ("frees", ctypes.c_int64),
                ("cow_copies", ctypes.c_int64), ("peak_used", ctypes.c_int64)]


# every symbol of include/pkv.h with (restype, argtypes)
_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_P = ctypes.POINTER
SIGNATURES = {
    "pkv_abi_version": (_i32, []),
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_status_string": (ctypes.c_char_p, [_i32]),
    "pkv_write_kv": (_i32, [_vp, _vp, _i64, _vp, _i32, _P(PkvCache), _vp, _vp]),
    "pkv_attn_decode_workspace_size": (_i32, [_i32, _i32, _i32, _i32, _i32, _P(_sz)]),
    "pkv_attn_decode": (_i32, [_vp, _i64, _P(PkvCache), _vp, _i32, _vp, _i32, _i32, _f32, _vp, _i32,
                               _vp, _sz, _vp, _vp]),
    "pkv_attn_decode_noalloc": (_i32, [_vp, _i64, _P(PkvCache), _vp, _i32, _vp, _i32, _i32, _f32, _vp, _i32,
                                       _vp, _vp]),
    "pkv_attn_varlen_workspace_size": (_i32, [_i32, _i32, _i32, _i32, _i32, _P(_sz)]),
    "pkv_attn_varlen": (_i32, [_vp, _i64, _P(PkvCache), _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                               _f32, _i32, _vp, _i32, _vp, _sz, _vp, _vp]),
    "pkv_attn_decode_window": (_i32, [_vp, _i64, _P(PkvCache), _vp, _i32, _vp, _i32, _i32, _f32, _i32, _vp,
                                      _i32, _vp, _sz, _vp, _vp]),
    "pkv_attn_varlen_window": (_i32, [_vp, _i64, _P(PkvCache), _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                      _f32, _i32, _i32, _vp, _i32, _vp, _sz, _vp, _vp]),
    "pkv_attn_decode_append": (_i32, [_vp, _i64, _vp, _vp, _i64, _P(PkvCache), _vp, _i32, _vp, _i32, _i32, _f32,
                                      _i32, _vp, _i32, _vp, _sz, _vp, _vp]),
    "pkv_write_kv_int8": (_i32, [_vp, _vp, _i64, _vp, _i32, _P(PkvCacheI8), _vp, _vp]),
    "pkv_attn_decode_int8": (_i32, [_vp, _i64, _P(PkvCacheI8), _vp, _i32, _vp, _i32, _i32, _f32, _i32, _vp, _i32,
                                    _vp, _sz, _vp, _vp]),
    "pkv_copy_blocks": (_i32, [_P(PkvCache), _i32, _vp, _i32, _vp, _vp]),
    "pkv_check_copy_pairs": (_i32, [_vp, _i32, _i32]),
    "pkv_alloc_create": (_i32, [_i32, _i32, _P(_vp)]),
    "pkv_alloc_destroy": (None, [_vp]),
    "pkv_alloc_set_free_order": (_i32, [_vp, _vp, _i32]),
    "pkv_alloc_allocate": (_i32, [_vp, _P(_i32)]),
    "pkv_alloc_allocate_for": (_i32, [_vp, _i64, _vp, _i32, _P(_i32)]),
    "pkv_alloc_free": (_i32, [_vp, _i32]),
    "pkv_alloc_free_all": (_i32, [_vp, _vp, _i32]),
    "pkv_alloc_retain": (_i32, [_vp, _i32]),
    "pkv_alloc_refcount": (_i32, [_vp, _i32]),
    "pkv_alloc_num_free": (_i32, [_vp]),
    "pkv_alloc_blocks_needed": (_i64, [_vp, _i64]),
    "pkv_alloc_counters_get": (_i32, [_vp, _P(PkvCounters)]),
    "pkv_seq_create": (_i32, [_vp, _vp, _i32, _i64, _P(_i32)]),
    "pkv_seq_fork": (_i32, [_vp, _i32, _P(_i32)]),
    "pkv_seq_free": (_i32, [_vp, _i32]),
    "pkv_seq_append": (_i32, [_vp, _vp, _vp, _i32, _vp, _i64, _vp, _i32, _P(_i32)]),
    "pkv_seq_len": (_i32, [_vp, _i32, _P(_i64)]),
    "pkv_seq_block_table": (_i32, [_vp, _i32, _vp, _i32, _P(_i32)]),
    "pkv_seq_fill_tables": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp]),
    "pkv_prefix_match": (_i32, [_vp, _vp, _i64, _vp, _i32, _P(_i32)]),
    "pkv_seq_create_prefixed": (_i32, [_vp, _vp, _i64, _P(_i32), _P(_i64)]),
    "pkv_prefix_insert": (_i32, [_vp, _vp, _i64, _vp, _i32]),
    "pkv_prefix_evict": (_i32, [_vp, _i32, _vp, _P(_i32)]),
    "pkv_prefix_num_nodes": (_i32, [_vp]),
}

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libpkv (built first if missing or older than its sources)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                path = _build.build()
                L = ctypes.CDLL(path)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def library_path() -> str:
    return _build.OUT


def check(status: int) -> None:
    if status == PKV_OK:
        return
    msg = lib().pkv_last_error().decode()
    if status == 5:
        raise ExhaustedError(status, msg)
    if status == 6:
        raise DoubleFreeError(status, msg)
    raise PkvError(status, msg)
