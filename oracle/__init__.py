"""CPU oracle for the paged KV cache path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  The product library
(``pagedattention_decode_gb300``) never imports it, and this package never
imports the product: the two share no code.  The only module both sides use
is ``workloads`` (seeded inputs, no arithmetic of the method).

Contents:

* ``pkv_oracle.c``: binary64 slot write, block copy and paged attention
  (gather through the block table, then a plain max-subtracted softmax), built
  into ``liboracle.so`` with gcc by :func:`build`.
* ``allocator.py``: the reference block allocator (free stack + handed-out
  set + refcounts + sequences with fork and copy-on-write).

Pins (the tests under ``tests/test_oracle_*.py``): the 6-block/16-token
allocator trace and the block_size 4 slot trace (``tests/golden/``), ceil
block counts, the memory arithmetic of page 2, closed forms (one key, equal
keys, zero query), torch's CPU scaled_dot_product_attention in float64 on the
gathered tensors, invariance under permutations of physical block ids and
changes of block_size, the GQA head mapping, the causal offset, and brute force
in exact rational arithmetic for the scores.  No function here is unpinned.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F16, BF16 = 0, 1
_lib = None


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``liboracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_decode_f16.restype = ctypes.c_double
        L.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        L.oracle_decode_bf16.restype = ctypes.c_double
        L.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_write_kv.restype = i64
        L.oracle_write_kv.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64]
        L.oracle_copy_blocks.restype = i32
        L.oracle_copy_blocks.argtypes = [vp, vp, i64, i64, vp, i64]
        L.oracle_paged_attention.restype = i32
        L.oracle_paged_attention.argtypes = [vp, i64, vp, vp, i32, i64, i32, i32, i32,
                                             vp, i32, vp, vp, i32, i32,
                                             ctypes.c_double, i32, i32, vp]
        L.oracle_write_kv_int8.restype = i32
        L.oracle_write_kv_int8.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp, vp, vp, vp, i64, i32]
        L.oracle_paged_attention_int8.restype = i32
        L.oracle_paged_attention_int8.argtypes = [vp, i64, i32, vp, vp, vp, vp, i64, i32, i32, i32,
                                                  vp, i32, vp, i32, i32, ctypes.c_double, i32, vp]
        _lib = L
    return _lib


def _bits(a) -> np.ndarray:
    """uint16 bit patterns of a float16 / bfloat16 array (numpy or torch)."""
    if hasattr(a, "detach"):  # torch tensor: take the raw 16-bit patterns
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.view(torch.int16)
        a = t.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    elif a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit float bit patterns, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def dtype_code(name) -> int:
    s = str(name)
    return BF16 if "bf16" in s or "bfloat16" in s else F16


def paged_attention(q, k_cache, v_cache, dtype, block_tables, kv_lens, scale: float,
                    cu_q: Optional[np.ndarray] = None, causal: bool = False, window: int = 0) -> np.ndarray:
    """binary64 paged attention.

    q: [rows, Hq, D]; caches: [num_blocks, block_size, Hkv, D] (16-bit floats
    of ``dtype``); block_tables [B, max_blocks] int32; kv_lens [B] int32;
    cu_q [B+1] int32 or None (one row per sequence); window > 0 keeps only the
    most recent ``window`` keys of each row.  Returns [rows, Hq, D].
    """
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    nb, bs, hkv, d = kb.shape
    rows, hq, d2 = qb.shape
    assert d2 == d and vb.shape == kb.shape
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))
    B = lens.shape[0]
    cu = None if cu_q is None else np.ascontiguousarray(np.asarray(cu_q, dtype=np.int32))
    out = np.zeros((rows, hq, d), dtype=np.float64)
    rc = lib().oracle_paged_attention(_ptr(qb), hq * d, _ptr(kb), _ptr(vb), dtype_code(dtype),
                                      nb, bs, hkv, d, _ptr(tables), tables.shape[1], _ptr(lens),
                                      None if cu is None else _ptr(cu), B, hq,
                                      float(scale), 1 if causal else 0, int(window), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_paged_attention rejected its inputs")
    return out


def write_kv(k, v, slots, k_cache: np.ndarray, v_cache: np.ndarray) -> int:
    """Write rows of k/v [T, Hkv, D] into the caches (uint16 arrays, in place)."""
    kb, vb = _bits(k), _bits(v)
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T = kb.shape[0]
    row = int(np.prod(kb.shape[1:]))
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    nslots = k_cache.shape[0] * k_cache.shape[1]
    n = lib().oracle_write_kv(_ptr(kb), _ptr(vb), T, row, _ptr(sl), _ptr(k_cache),
                              _ptr(v_cache), nslots)
    if n < 0:
        raise ValueError("slot outside the pool")
    return int(n)


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """Copy block src -> dst for each (src, dst) pair (uint16 caches, in place)."""
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    nb = k_cache.shape[0]
    blk = int(np.prod(k_cache.shape[1:]))
    rc = lib().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), nb, blk, _ptr(pr), pr.shape[0])
    if rc != 0:
        raise ValueError("block id outside the pool")


def decode_f16(bits: int) -> float:
    return lib().oracle_decode_f16(bits)


def decode_bf16(bits: int) -> float:
    return lib().oracle_decode_bf16(bits)


def write_kv_int8(k, v, dtype, slots, kq: np.ndarray, vq: np.ndarray, kscale: np.ndarray,
                  vscale: np.ndarray) -> None:
    """Quantised write (in place): int8 pools [nb, bs, Hkv, D], float32 scales [nb, Hkv]."""
    kb, vb = _bits(k), _bits(v)
    for a, dt in ((kq, np.int8), (vq, np.int8), (kscale, np.float32), (vscale, np.float32)):
        assert a.dtype == dt and a.flags.c_contiguous
    T, hkv, d = kb.shape
    nb, bs = kq.shape[:2]
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    rc = lib().oracle_write_kv_int8(_ptr(kb), _ptr(vb), dtype_code(dtype), T, hkv, d, _ptr(sl), _ptr(kq),
                                    _ptr(vq), _ptr(kscale), _ptr(vscale), nb, bs)
    if rc != 0:
        raise ValueError("slot outside the pool")


def paged_attention_int8(q, dtype, kq: np.ndarray, vq: np.ndarray, kscale: np.ndarray, vscale: np.ndarray,
                         block_tables, kv_lens, scale: float, window: int = 0) -> np.ndarray:
    """binary64 decode attention over an int8 cache (values = code * scale)."""
    qb = _bits(q)
    B, hq, d = qb.shape
    nb, bs, hkv, d2 = kq.shape
    assert d2 == d
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))
    out = np.zeros((B, hq, d), dtype=np.float64)
    rc = lib().oracle_paged_attention_int8(_ptr(qb), hq * d, dtype_code(dtype), _ptr(np.ascontiguousarray(kq)),
                                           _ptr(np.ascontiguousarray(vq)), _ptr(np.ascontiguousarray(kscale)),
                                           _ptr(np.ascontiguousarray(vscale)), nb, bs, hkv, d, _ptr(tables),
                                           tables.shape[1], _ptr(lens), B, hq, float(scale), int(window), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_paged_attention_int8 rejected its inputs")
    return out
