"""Pins of the int8 KV cache oracle (quantised write, int8 attention).

Page 4 ("Building a paged inference engine from scratch, and measuring it
honestly", section 02, INT8 KV cache design) calls its own int8 path
unverified, so the oracle is pinned here by the properties its definition
fixes: the quantiser's error bound and closed forms, and int8 attention
reducing to the 16-bit attention oracle when every scale is 1.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle.allocator import RefAllocator


def _pool(nb, bs, hkv, d):
    return (np.zeros((nb, bs, hkv, d), np.int8), np.zeros((nb, bs, hkv, d), np.int8),
            np.zeros((nb, hkv), np.float32), np.zeros((nb, hkv), np.float32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_fresh_block_round_trip_within_half_step(dtype):
    nb, bs, hkv, d = 4, 16, 2, 64
    kq, vq, ks, vs = _pool(nb, bs, hkv, d)
    g = W.generator(1)
    k = W.normal(g, (bs, hkv, d), 1.0, dtype)
    v = W.normal(g, (bs, hkv, d), 1.0, dtype)
    oracle.write_kv_int8(k, v, dtype, list(range(2 * bs, 3 * bs)), kq, vq, ks, vs)  # block 2
    for x, q, sc in ((k, kq, ks), (v, vq, vs)):
        xf = x.float().numpy()
        for h in range(hkv):
            s = sc[2, h]
            assert s == np.float32(np.abs(xf[:, h]).max()) / np.float32(127)
            err = np.abs(q[2, :, h].astype(np.float64) * s - xf[:, h])
            # half a step, plus the binary32 rounding of x / s (|x / s| <= 127)
            assert (err <= s * (0.5 + 1e-5)).all()
            assert np.abs(q[2, :, h]).max() == 127
    assert not kq[[0, 1, 3]].any() and not ks[[0, 1, 3]].any()


def test_constant_and_zero_blocks():
    nb, bs, hkv, d = 2, 4, 1, 8
    kq, vq, ks, vs = _pool(nb, bs, hkv, d)
    c = torch.full((bs, hkv, d), -3.5, dtype=torch.float16)
    z = torch.zeros((bs, hkv, d), dtype=torch.float16)
    oracle.write_kv_int8(c, z, "f16", [0, 1, 2, 3], kq, vq, ks, vs)
    assert (kq[0] == -127).all() and ks[0, 0] == np.float32(3.5) / np.float32(127)
    assert (vq[0] == 0).all() and vs[0, 0] == 0.0


def test_appends_requantise_the_block():
    """Decode appends one token at a time: each write re-scales the block over
    its earlier (dequantised) rows and the new one."""
    nb, bs, hkv, d = 4, 8, 1, 16
    kq, vq, ks, vs = _pool(nb, bs, hkv, d)
    a = RefAllocator(nb, bs)
    s = a.create_sequence()
    g = W.generator(2)
    prev = 0.0
    for t in range(bs):
        (slot,), _ = a.append_tokens([s])
        x = W.normal(g, (1, hkv, d), 1.0 + t, "f16")  # growing magnitudes
        oracle.write_kv_int8(x, x, "f16", [slot], kq, vq, ks, vs)
        blk = slot // bs
        assert ks[blk, 0] >= prev * (1 - 1e-6)
        prev = ks[blk, 0]
        row = kq[blk, slot % bs, 0].astype(np.float64) * ks[blk, 0]
        assert np.abs(row - x[0, 0].double().numpy()).max() <= ks[blk, 0] * (0.5 + 1e-5)
        assert np.abs(kq[blk, :t + 1]).max() == 127


def test_int8_attention_unit_scales_equals_16bit_oracle():
    rng = np.random.default_rng(3)
    nb, bs, hkv, d, hq = 6, 16, 2, 32, 8
    kq = rng.integers(-127, 128, (nb, bs, hkv, d), dtype=np.int64).astype(np.int8)
    vq = rng.integers(-127, 128, (nb, bs, hkv, d), dtype=np.int64).astype(np.int8)
    ones = np.ones((nb, hkv), np.float32)
    q = W.normal(W.generator(4), (3, hq, d), 0.05, "f16")
    tables = np.array([[4, 1, -1], [0, 5, 2], [3, -1, -1]], np.int32)
    lens = [20, 40, 16]
    got = oracle.paged_attention_int8(q, "f16", kq, vq, ones, ones, tables, lens, 0.1)
    kf = torch.from_numpy(kq.astype(np.float32)).half()  # integers |x| <= 127 are exact in fp16
    vf = torch.from_numpy(vq.astype(np.float32)).half()
    want = oracle.paged_attention(q, kf, vf, "f16", tables, lens, 0.1)
    assert np.array_equal(got, want)
    # and a window of w equals the 16-bit oracle's window
    got_w = oracle.paged_attention_int8(q, "f16", kq, vq, ones, ones, tables, lens, 0.1, window=7)
    assert np.array_equal(got_w, oracle.paged_attention(q, kf, vf, "f16", tables, lens, 0.1, window=7))
