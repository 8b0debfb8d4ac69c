"""GB300-native paged KV cache attention: Python binding of libpkv.

The functions here only marshal torch tensors into the C ABI of
``include/pkv.h`` (pointers, sizes, the current CUDA stream); every step of
the path runs in libpkv's CUDA kernels or its C++ allocator.  There is no CPU
or PyTorch fallback: a missing library or a non-CUDA tensor is an error.

Calls (names as in the C ABI, without the ``pkv_`` prefix):

* :func:`write_kv` -- scatter new K/V rows into their slots;
* :func:`attn_decode` -- one query row per sequence over its paged keys;
* :func:`attn_varlen` -- packed prefill chunks and decode rows, causal offset;
* :func:`copy_blocks` -- block copies for copy-on-write;
* :class:`BlockAllocator` -- host allocator producing tables, slots and pairs;
* :class:`StepGraph` -- a CUDA graph of a step built from these calls.
"""

from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import torch

from ._native import (DEVERR, PKV_BF16, PKV_F16, PKV_F32, DoubleFreeError, ExhaustedError, PkvCache,
                      PkvCacheI8, PkvCounters, PkvError, check, lib, library_path)

__all__ = [
    "write_kv", "attn_decode", "attn_varlen", "copy_blocks", "decode_workspace_size",
    "varlen_workspace_size", "check_copy_pairs", "BlockAllocator", "PkvError", "ExhaustedError",
    "DoubleFreeError", "DEVERR", "library_path", "StepGraph", "write_kv_int8", "attn_decode_int8",
]

_DT = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.float32: PKV_F32}


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cache(k_cache: torch.Tensor, v_cache: torch.Tensor) -> PkvCache:
    _cuda(k_cache, "k_cache")
    _cuda(v_cache, "v_cache")
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must both be [num_blocks, block_size, kv_heads, head_dim]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if k_cache.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("caches must be float16 or bfloat16")
    nb, bs, hkv, d = k_cache.shape
    return PkvCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, d, _DT[k_cache.dtype])


def _row_stride(t: torch.Tensor, name: str) -> int:
    """Elements between rows of a [rows, heads, dim] tensor with heads/dims packed."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name} must be [rows, heads, head_dim] with heads and dims contiguous")
    return t.stride(0)


def _check_i32(t: torch.Tensor, name: str) -> None:
    _cuda(t, name)
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")


def write_kv(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
             v_cache: torch.Tensor, err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Rows k[t], v[t] ([T, Hkv, D]) go to slot slot_mapping[t] (int64; < 0 skips)."""
    c = _cache(k_cache, v_cache)
    _cuda(k, "k")
    _cuda(v, "v")
    _cuda(slot_mapping, "slot_mapping")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous():
        raise TypeError("slot_mapping must be contiguous int64")
    if k.shape != v.shape or k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or k.stride() != v.stride():
        raise ValueError("k and v must match each other and the cache dtype")
    if k.shape[1:] != k_cache.shape[2:] or k.shape[0] != slot_mapping.numel():
        raise ValueError("k is [T, kv_heads, head_dim] with T = slot_mapping.numel()")
    check(lib().pkv_write_kv(_ptr(k), _ptr(v), _row_stride(k, "k"), _ptr(slot_mapping), k.shape[0],
                             ctypes.byref(c), _ptr(err), _stream(stream)))


def decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          device: Optional[int] = None) -> int:
    n = ctypes.c_size_t(0)
    dev = torch.cuda.current_device() if device is None else device
    check(lib().pkv_attn_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, dev,
                                               ctypes.byref(n)))
    return n.value


def varlen_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          device: Optional[int] = None) -> int:
    n = ctypes.c_size_t(0)
    dev = torch.cuda.current_device() if device is None else device
    check(lib().pkv_attn_varlen_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, dev,
                                               ctypes.byref(n)))
    return n.value


def _workspace(size_fn, workspace: Optional[torch.Tensor], device) -> torch.Tensor:
    """The caller's workspace as given (the library checks its size), or a new one."""
    if workspace is not None:
        return workspace
    return torch.empty(max(size_fn(), 1), dtype=torch.uint8, device=device)


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                seq_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                out_dtype: torch.dtype = torch.float32, workspace: Optional[torch.Tensor] = None,
                err: Optional[torch.Tensor] = None, stream=None, window: int = 0,
                k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None) -> torch.Tensor:
    """q [B, Hq, D]; tables [B, max_blocks] int32; seq_lens [B] int32 -> out [B, Hq, D].

    window > 0 attends only each sequence's most recent ``window`` keys.
    With k_new / v_new [B, Hkv, D], row s is first written to the slot of
    position seq_lens[s] - 1 (from the block table) in the same kernel
    (pkv_attn_decode_append)."""
    c = _cache(k_cache, v_cache)
    _cuda(q, "q")
    _check_i32(block_tables, "block_tables")
    _check_i32(seq_lens, "seq_lens")
    if q.dtype != k_cache.dtype:
        raise TypeError("q must have the cache dtype")
    B, hq, d = q.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=q.device)
    elif not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous [B, Hq, D]")
    ws = _workspace(lambda: decode_workspace_size(B, hq, c.num_kv_heads, d, q.device.index), workspace, q.device)
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _cuda(t, n)
            if t.dtype != k_cache.dtype or t.shape != (B, c.num_kv_heads, d):
                raise ValueError(f"{n} must be [B, Hkv, D] of the cache dtype")
        if k_new.stride() != v_new.stride() or k_new.stride(1) != d or k_new.stride(2) != 1:
            raise ValueError("k_new / v_new: rows of contiguous heads, the same stride")
        check(lib().pkv_attn_decode_append(_ptr(q), _row_stride(q, "q"), _ptr(k_new), _ptr(v_new), k_new.stride(0),
                                           ctypes.byref(c), _ptr(block_tables), mb, _ptr(seq_lens), B, hq,
                                           float(scale), int(window), _ptr(out), _DT[out.dtype], _ptr(ws),
                                           ws.numel() * ws.element_size(), _ptr(err), _stream(stream)))
    elif window > 0:
        check(lib().pkv_attn_decode_window(_ptr(q), _row_stride(q, "q"), ctypes.byref(c), _ptr(block_tables), mb,
                                           _ptr(seq_lens), B, hq, float(scale), int(window), _ptr(out),
                                           _DT[out.dtype], _ptr(ws), ws.numel() * ws.element_size(), _ptr(err),
                                           _stream(stream)))
    else:
        check(lib().pkv_attn_decode(_ptr(q), _row_stride(q, "q"), ctypes.byref(c), _ptr(block_tables), mb,
                                    _ptr(seq_lens), B, hq, float(scale), _ptr(out), _DT[out.dtype], _ptr(ws),
                                    ws.numel() * ws.element_size(), _ptr(err), _stream(stream)))
    return out


def attn_varlen(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                cu_seqlens_q: torch.Tensor, seq_lens: torch.Tensor, max_q_len: int, scale: float,
                causal: bool = True, out: Optional[torch.Tensor] = None,
                out_dtype: torch.dtype = torch.float32, workspace: Optional[torch.Tensor] = None,
                err: Optional[torch.Tensor] = None, stream=None, window: int = 0) -> torch.Tensor:
    """Packed rows q [total_q, Hq, D]; cu_seqlens_q [B+1]; seq_lens = kv_len [B].

    window > 0 attends only each row's most recent ``window`` keys."""
    c = _cache(k_cache, v_cache)
    _cuda(q, "q")
    _check_i32(block_tables, "block_tables")
    _check_i32(seq_lens, "seq_lens")
    _check_i32(cu_seqlens_q, "cu_seqlens_q")
    if q.dtype != k_cache.dtype:
        raise TypeError("q must have the cache dtype")
    total, hq, d = q.shape
    B = seq_lens.numel()
    if cu_seqlens_q.numel() != B + 1:
        raise ValueError("cu_seqlens_q must have num_seqs + 1 entries")
    if out is None:
        out = torch.empty((total, hq, d), dtype=out_dtype, device=q.device)
    ws = _workspace(lambda: varlen_workspace_size(B, hq, c.num_kv_heads, d, q.device.index), workspace, q.device)
    if window > 0:
        check(lib().pkv_attn_varlen_window(_ptr(q), _row_stride(q, "q"), ctypes.byref(c), _ptr(block_tables),
                                           block_tables.shape[1], _ptr(cu_seqlens_q), _ptr(seq_lens), B, total,
                                           int(max_q_len), hq, float(scale), 1 if causal else 0, int(window),
                                           _ptr(out), _DT[out.dtype], _ptr(ws), ws.numel() * ws.element_size(),
                                           _ptr(err), _stream(stream)))
    else:
        check(lib().pkv_attn_varlen(_ptr(q), _row_stride(q, "q"), ctypes.byref(c), _ptr(block_tables),
                                    block_tables.shape[1], _ptr(cu_seqlens_q), _ptr(seq_lens), B, total,
                                    int(max_q_len), hq, float(scale), 1 if causal else 0, _ptr(out), _DT[out.dtype],
                                    _ptr(ws), ws.numel() * ws.element_size(), _ptr(err), _stream(stream)))
    return out


def _cache_i8(kq: torch.Tensor, vq: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
              dtype: torch.dtype) -> PkvCacheI8:
    for t, name in ((kq, "kq"), (vq, "vq"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _cuda(t, name)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if kq.dtype != torch.int8 or vq.dtype != torch.int8 or kq.shape != vq.shape or kq.dim() != 4:
        raise TypeError("int8 pools must be int8 [num_blocks, block_size, kv_heads, head_dim]")
    nb, bs, hkv, d = kq.shape
    if k_scale.dtype != torch.float32 or k_scale.shape != (nb, hkv) or v_scale.shape != (nb, hkv):
        raise TypeError("scales must be float32 [num_blocks, kv_heads]")
    if dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("the compute dtype must be float16 or bfloat16")
    return PkvCacheI8(kq.data_ptr(), vq.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(), nb, bs, hkv, d,
                      _DT[dtype])


def write_kv_int8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, kq: torch.Tensor, vq: torch.Tensor,
                  k_scale: torch.Tensor, v_scale: torch.Tensor, err: Optional[torch.Tensor] = None,
                  stream=None) -> None:
    """Quantised write of rows k[t], v[t] (fp16/bf16 [T, Hkv, D]) into an int8 cache; the blocks
    written are re-quantised with a new per-block-per-head scale."""
    c = _cache_i8(kq, vq, k_scale, v_scale, k.dtype)
    _cuda(k, "k")
    _cuda(v, "v")
    _cuda(slot_mapping, "slot_mapping")
    if slot_mapping.dtype != torch.int64 or k.shape != v.shape or k.shape[0] != slot_mapping.numel():
        raise ValueError("k, v [T, kv_heads, head_dim] and int64 slot_mapping [T] expected")
    check(lib().pkv_write_kv_int8(_ptr(k), _ptr(v), _row_stride(k, "k"), _ptr(slot_mapping), k.shape[0],
                                  ctypes.byref(c), _ptr(err), _stream(stream)))


def attn_decode_int8(q: torch.Tensor, kq: torch.Tensor, vq: torch.Tensor, k_scale: torch.Tensor,
                     v_scale: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     window: int = 0, out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
                     workspace: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """Decode attention over an int8 cache; q fp16/bf16 [B, Hq, D]."""
    c = _cache_i8(kq, vq, k_scale, v_scale, q.dtype)
    _cuda(q, "q")
    _check_i32(block_tables, "block_tables")
    _check_i32(seq_lens, "seq_lens")
    B, hq, d = q.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=out_dtype, device=q.device)
    ws = _workspace(lambda: decode_workspace_size(B, hq, c.num_kv_heads, d, q.device.index), workspace, q.device)
    check(lib().pkv_attn_decode_int8(_ptr(q), _row_stride(q, "q"), ctypes.byref(c), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(seq_lens), B, hq, float(scale), int(window),
                                     _ptr(out), _DT[out.dtype], _ptr(ws), ws.numel() * ws.element_size(), _ptr(err),
                                     _stream(stream)))
    return out


def copy_blocks(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor], src_dst_pairs: torch.Tensor,
                err: Optional[torch.Tensor] = None, stream=None) -> None:
    """For each (src, dst) row of src_dst_pairs (int64 [N, 2], CUDA): block dst <- block src, every layer."""
    if len(k_caches) != len(v_caches):
        raise ValueError("one v cache per k cache")
    _cuda(src_dst_pairs, "src_dst_pairs")
    if src_dst_pairs.dtype != torch.int64 or not src_dst_pairs.is_contiguous():
        raise TypeError("src_dst_pairs must be contiguous int64")
    arr = (PkvCache * max(1, len(k_caches)))(*[_cache(k, v) for k, v in zip(k_caches, v_caches)])
    n = src_dst_pairs.numel() // 2
    check(lib().pkv_copy_blocks(arr, len(k_caches), _ptr(src_dst_pairs), n, _ptr(err), _stream(stream)))


def check_copy_pairs(pairs: Sequence[Tuple[int, int]], num_blocks: int) -> None:
    flat = [int(x) for p in pairs for x in p]
    buf = (ctypes.c_int64 * max(1, len(flat)))(*flat)
    check(lib().pkv_check_copy_pairs(buf, len(flat) // 2, num_blocks))


class BlockAllocator:
    """Host block allocator and block tables (C++, behind the C ABI)."""

    def __init__(self, num_blocks: int, block_size: int):
        h = ctypes.c_void_p()
        check(lib().pkv_alloc_create(num_blocks, block_size, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib().pkv_alloc_destroy(h)
            self._h = None

    # block level
    @property
    def num_free(self) -> int:
        return lib().pkv_alloc_num_free(self._h)

    def set_free_order(self, order: Sequence[int]) -> None:
        buf = (ctypes.c_int32 * max(1, len(order)))(*order)
        check(lib().pkv_alloc_set_free_order(self._h, buf, len(order)))

    def allocate(self) -> int:
        out = ctypes.c_int32()
        check(lib().pkv_alloc_allocate(self._h, ctypes.byref(out)))
        return out.value

    def blocks_needed(self, num_tokens: int) -> int:
        n = lib().pkv_alloc_blocks_needed(self._h, num_tokens)
        if n < 0:
            raise ValueError("negative token count")
        return n

    def allocate_for(self, num_tokens: int) -> List[int]:
        cap = max(1, self.blocks_needed(num_tokens)) if num_tokens >= 0 else 1
        buf = (ctypes.c_int32 * cap)()
        n = ctypes.c_int32()
        check(lib().pkv_alloc_allocate_for(self._h, num_tokens, buf, cap, ctypes.byref(n)))
        return list(buf[:n.value])

    def free(self, block_id: int) -> None:
        check(lib().pkv_alloc_free(self._h, block_id))

    release = free

    def free_all(self, ids: Sequence[int]) -> None:
        buf = (ctypes.c_int32 * max(1, len(ids)))(*ids)
        check(lib().pkv_alloc_free_all(self._h, buf, len(ids)))

    def retain(self, block_id: int) -> None:
        check(lib().pkv_alloc_retain(self._h, block_id))

    def refcount(self, block_id: int) -> int:
        return lib().pkv_alloc_refcount(self._h, block_id)

    def counters(self) -> dict:
        c = PkvCounters()
        check(lib().pkv_alloc_counters_get(self._h, ctypes.byref(c)))
        return {"allocs": c.allocs, "frees": c.frees, "cow_copies": c.cow_copies, "peak_used": c.peak_used}

    # sequence level
    def create_sequence(self, shared_ids: Sequence[int] = (), shared_tokens: int = 0) -> int:
        buf = (ctypes.c_int32 * max(1, len(shared_ids)))(*shared_ids)
        out = ctypes.c_int32()
        check(lib().pkv_seq_create(self._h, buf, len(shared_ids), shared_tokens, ctypes.byref(out)))
        return out.value

    def fork(self, seq_id: int) -> int:
        out = ctypes.c_int32()
        check(lib().pkv_seq_fork(self._h, seq_id, ctypes.byref(out)))
        return out.value

    def free_sequence(self, seq_id: int) -> None:
        check(lib().pkv_seq_free(self._h, seq_id))

    def append_tokens(self, seq_ids: Sequence[int], counts: Optional[Sequence[int]] = None
                      ) -> Tuple[List[int], List[Tuple[int, int]]]:
        n = len(seq_ids)
        ids = (ctypes.c_int32 * max(1, n))(*seq_ids)
        cnt = None if counts is None else (ctypes.c_int32 * max(1, n))(*counts)
        total = n if counts is None else sum(int(c) for c in counts)
        slots = (ctypes.c_int64 * max(1, total))()
        pairs = (ctypes.c_int64 * max(2, 2 * n))()
        np_ = ctypes.c_int32()
        check(lib().pkv_seq_append(self._h, ids, cnt, n, slots, max(0, total), pairs, n, ctypes.byref(np_)))
        return list(slots[:total]), [(pairs[2 * i], pairs[2 * i + 1]) for i in range(np_.value)]

    def append_tokens_into(self, seq_ids: Sequence[int], slots_out, pairs_out) -> int:
        """One token per sequence, slots written into a caller buffer (e.g. pinned
        int64 host memory); returns the number of copy-on-write pairs written."""
        n = len(seq_ids)
        ids = (ctypes.c_int32 * max(1, n))(*seq_ids)
        np_ = ctypes.c_int32()
        check(lib().pkv_seq_append(self._h, ids, None, n, ctypes.c_void_p(slots_out.data_ptr()), n,
                                   ctypes.c_void_p(pairs_out.data_ptr()), pairs_out.numel() // 2,
                                   ctypes.byref(np_)))
        return np_.value

    def seq_len(self, seq_id: int) -> int:
        n = ctypes.c_int64()
        check(lib().pkv_seq_len(self._h, seq_id, ctypes.byref(n)))
        return n.value

    def block_table(self, seq_id: int) -> List[int]:
        cap = self.blocks_needed(self.seq_len(seq_id)) + 1
        buf = (ctypes.c_int32 * cap)()
        n = ctypes.c_int32()
        check(lib().pkv_seq_block_table(self._h, seq_id, buf, cap, ctypes.byref(n)))
        return list(buf[:n.value])

    # prefix sharing
    def prefix_match(self, tokens: Sequence[int]) -> List[int]:
        """Ids of the whole blocks of ``tokens`` already in the trie (not retained)."""
        n = len(tokens)
        toks = (ctypes.c_int32 * max(1, n))(*tokens)
        cap = n // self.block_size
        out = (ctypes.c_int32 * max(1, cap))()
        m = ctypes.c_int32()
        check(lib().pkv_prefix_match(self._h, toks, n, out, cap, ctypes.byref(m)))
        return list(out[:m.value])

    def create_sequence_prefixed(self, tokens: Sequence[int]) -> Tuple[int, int]:
        """New sequence on the trie's matched whole blocks of ``tokens`` (match and
        create atomically); returns (sequence id, shared token count)."""
        toks = (ctypes.c_int32 * max(1, len(tokens)))(*tokens)
        sid, shared = ctypes.c_int32(), ctypes.c_int64()
        check(lib().pkv_seq_create_prefixed(self._h, toks, len(tokens), ctypes.byref(sid), ctypes.byref(shared)))
        return sid.value, shared.value

    def prefix_insert(self, tokens: Sequence[int], block_ids: Sequence[int]) -> None:
        toks = (ctypes.c_int32 * max(1, len(tokens)))(*tokens)
        ids = (ctypes.c_int32 * max(1, len(block_ids)))(*block_ids)
        check(lib().pkv_prefix_insert(self._h, toks, len(tokens), ids, len(block_ids)))

    def prefix_evict(self, max_blocks: int) -> List[int]:
        out = (ctypes.c_int32 * max(1, max_blocks))()
        n = ctypes.c_int32()
        check(lib().pkv_prefix_evict(self._h, max_blocks, out, ctypes.byref(n)))
        return list(out[:n.value])

    @property
    def prefix_nodes(self) -> int:
        return lib().pkv_prefix_num_nodes(self._h)

    def fill_tables(self, seq_ids: Sequence[int], max_blocks: int, tables_out: torch.Tensor,
                    lens_out: torch.Tensor) -> None:
        """Rows of tables_out [n, max_blocks] int32 and lens_out [n] int32 (CPU tensors)."""
        if tables_out.device.type != "cpu" or lens_out.device.type != "cpu":
            raise TypeError("fill_tables writes host tensors")
        ids = (ctypes.c_int32 * max(1, len(seq_ids)))(*seq_ids)
        check(lib().pkv_seq_fill_tables(self._h, ids, len(seq_ids), ctypes.c_void_p(tables_out.data_ptr()),
                                        max_blocks, ctypes.c_void_p(lens_out.data_ptr())))


class StepGraph:
    """A CUDA graph of one step made of libpkv calls (and any copies between
    pinned host buffers and the device that surround them).

    Every call of the library is asynchronous on the current stream, allocates
    nothing and never synchronises the host, so a whole multi-layer step --
    copy_blocks, write_kv and attn_decode / attn_varlen for every layer -- can
    be captured once on static buffers and replayed: the per-call host work
    (argument checks, tensor-map encoding, launches) is paid once at capture.
    ``fn`` must use the same tensors on every call and pass explicit
    workspaces; the first call of pkv_attn_decode_noalloc on a device must
    come before the capture.
    """

    def __init__(self, fn, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def replay(self) -> None:
        self.graph.replay()
