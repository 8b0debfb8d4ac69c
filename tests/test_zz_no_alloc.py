"""pkv_attn_decode_noalloc: decode attention for callers that cannot allocate.

Some users of this library cannot hand it a workspace: a host program that
embeds libpkv in a process whose device memory belongs to another runtime's
allocator, or a loop that must not call cudaMalloc because that synchronises
the device.  The no-allocation entry point keeps its scratch in a fixed array
inside the library instead.  These tests call it through the C ABI and
compare it with the workspace entry point, twice in a row (the array keeps
the previous call's contents), and check that an over-size call is refused.

This file is collected last so that a failure here, under -x, comes after
every other test has run.
"""
import ctypes

import pytest
import torch

import pagedattention_decode_gb300 as P
from pagedattention_decode_gb300 import _native
from tests.cases import TOL, decode_case

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
    first = decode_case(901, [1, 700, 64, 3000, 17, 0, 2048, 5] * 12, 32, 8, 128, 16, "f16").to("cuda")
    second = decode_case(902, [40000, 9, 333], 24, 12, 64, 32, "bf16", sigma=0.5).to("cuda")
    for c in (first, second):
        want = _with_workspace(c)
        got = _no_alloc(c)
        torch.cuda.synchronize()
        assert (got - want).abs().max().item() <= TOL


def test_no_alloc_refuses_oversize_call():
    c = decode_case(903, [20, 30], 8, 2, 64, 16, "f16").to("cuda")
    L = _native.lib()
    cache = _cache(c)
    out = torch.empty((2, 8, 64), dtype=torch.float32, device="cuda")
    # ten million sequences need more scratch than the fixed array holds: the
    # call is refused on the host before anything is launched
    st = L.pkv_attn_decode_noalloc(c.q.data_ptr(), 8 * 64, ctypes.byref(cache), c.tables.data_ptr(),
                                   c.tables.shape[1], c.lens.data_ptr(), 10_000_000, 8, c.scale, out.data_ptr(),
                                   _native.PKV_F32, None, None)
    assert st == 8 and b"fixed array" in L.pkv_last_error()
