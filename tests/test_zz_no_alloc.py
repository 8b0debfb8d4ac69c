"""pkv_attn_decode_noalloc: decode attention for callers that cannot allocate.

Some users of this library cannot hand it a workspace: a host program that
embeds libpkv in a process whose device memory belongs to another runtime's
allocator, or a loop that must not call cudaMalloc because that synchronises
the device.  The no-allocation entry point keeps its scratch in a fixed array
inside the library instead.  These tests call it through the C ABI and
compare it with the workspace entry point (bit for bit: the same plan and
kernels) and with the binary64 oracle, twice in a row (the array keeps the
previous call's contents), and check that a call one sequence past the
array's size is refused.

This file is collected last so that a failure here, under -x, comes after
every other test has run.
"""
import ctypes

import pytest
import torch

import pagedattention_decode_gb300 as P
from pagedattention_decode_gb300 import _native
from tests.cases import assert_close, decode_case

pytestmark = pytest.mark.gpu


def _cache(c):
    nb, bs, hkv, d = c.k_cache.shape
    dt = _native.PKV_BF16 if c.k_cache.dtype == torch.bfloat16 else _native.PKV_F16
    return _native.PkvCache(c.k_cache.data_ptr(), c.v_cache.data_ptr(), nb, bs, hkv, d, dt)


def _with_workspace(c):
    L = _native.lib()
    B, hq, d = c.q.shape
    out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(P.decode_workspace_size(B, hq, c.k_cache.shape[2], d), dtype=torch.uint8, device="cuda")
    cache = _cache(c)
    st = L.pkv_attn_decode(c.q.data_ptr(), hq * d, ctypes.byref(cache), c.tables.data_ptr(), c.tables.shape[1],
                           c.lens.data_ptr(), B, hq, c.scale, out.data_ptr(), _native.PKV_F32, ws.data_ptr(),
                           ws.numel(), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.pkv_last_error()
    return out


def _no_alloc(c):
    L = _native.lib()
    B, hq, d = c.q.shape
    out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = _cache(c)
    st = L.pkv_attn_decode_noalloc(c.q.data_ptr(), hq * d, ctypes.byref(cache), c.tables.data_ptr(),
                                   c.tables.shape[1], c.lens.data_ptr(), B, hq, c.scale, out.data_ptr(),
                                   _native.PKV_F32, err.data_ptr(),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.pkv_last_error()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def test_no_alloc_matches_workspace_entry_point_twice():
    # two different calls in a row: many sequences cut by the split (records
    # in the scratch), then another shape and dtype over the same array
    first = decode_case(901, [1, 700, 64, 3000, 17, 0, 2048, 5] * 12, 32, 8, 128, 16, "f16")
    second = decode_case(902, [40000, 9, 333], 24, 12, 64, 32, "bf16", sigma=0.5)
    for c in (first, second):
        dc = c.to("cuda")
        want = _with_workspace(dc)
        got = _no_alloc(dc)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
        assert_close(got, c.oracle(), what="no-allocation decode")


def test_no_alloc_refuses_oversize_call():
    """The scratch holds the split-K records (they grow with the device's SM
    count, the query heads and head_dim) and 4 bytes per sequence.  At head_dim
    64 the size query's answer is the 16-bit plan the call checks: the
    smallest batch whose need passes the array's size is refused on the host,
    before anything is launched."""
    hq, hkv, d = 32, 4, 64
    limit = _native.PKV_NOALLOC_SCRATCH_BYTES
    need = lambda b: P.decode_workspace_size(b, hq, hkv, d)
    lo, hi = 1, 1 << 26          # need(lo) <= limit < need(hi)
    assert need(lo) <= limit < need(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= limit else (lo, mid)
    c = decode_case(903, [20, 30], hq, hkv, d, 16, "f16").to("cuda")
    L = _native.lib()
    cache = _cache(c)
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    st = L.pkv_attn_decode_noalloc(c.q.data_ptr(), hq * d, ctypes.byref(cache), c.tables.data_ptr(),
                                   c.tables.shape[1], c.lens.data_ptr(), hi, hq, c.scale, out.data_ptr(),
                                   _native.PKV_F32, None, None)
    msg = L.pkv_last_error()   # read before the next library call replaces it
    assert st == 8 and b"fixed array" in msg
    assert str(need(hi)).encode() in msg
