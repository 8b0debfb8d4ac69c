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


def _int8_case(seed, nb=7, bs=16, hkv=3, d=32):
    rng = np.random.default_rng(seed)
    kq = rng.integers(-127, 128, (nb, bs, hkv, d), dtype=np.int64).astype(np.int8)
    vq = rng.integers(-127, 128, (nb, bs, hkv, d), dtype=np.int64).astype(np.int8)
    # distinct power-of-two scales per (block, KV head), different for K and V:
    # code * 2^-k is exact in fp16 for |code| <= 127 and 2 <= k <= 9
    ek = rng.permutation(np.arange(nb * hkv) % 8 + 2).reshape(nb, hkv)
    ev = rng.permutation(np.arange(nb * hkv) % 8 + 2).reshape(nb, hkv)
    ks = np.ldexp(np.float32(1), -ek).astype(np.float32)
    vs = np.ldexp(np.float32(1), -ev).astype(np.float32)
    return kq, vq, ks, vs


def _premultiplied(codes, scales):
    """code * scale[block, head] as an fp16 pool: exact, since each scale is 2^-k."""
    x = codes.astype(np.float64) * scales[:, None, :, None].astype(np.float64)
    h = x.astype(np.float16)
    assert np.array_equal(h.astype(np.float64), x)
    return torch.from_numpy(h)


def test_int8_attention_applies_each_blocks_own_scales():
    """The scale of physical block b and KV head g multiplies exactly the codes
    of that block and head, K's scales for K and V's for V: with power-of-two
    scales the dequantised pool is exact in fp16, so the int8 oracle must equal
    the 16-bit oracle on the pre-multiplied pools bit for bit."""
    nb, bs, hkv, d, hq = 7, 16, 3, 32, 6
    kq, vq, ks, vs = _int8_case(5, nb, bs, hkv, d)
    q = W.normal(W.generator(6), (4, hq, d), 0.5, "f16")
    # scattered tables, partial tails, one sequence ending on a block edge
    tables = np.array([[6, 2, 0], [3, 5, -1], [1, -1, -1], [4, 0, 2]], np.int32)
    lens = [37, 32, 9, 45]
    kf, vf = _premultiplied(kq, ks), _premultiplied(vq, vs)
    want = oracle.paged_attention(q, kf, vf, "f16", tables, lens, 0.3)
    got = oracle.paged_attention_int8(q, "f16", kq, vq, ks, vs, tables, lens, 0.3)
    assert np.array_equal(got, want)
    got_w = oracle.paged_attention_int8(q, "f16", kq, vq, ks, vs, tables, lens, 0.3, window=11)
    assert np.array_equal(got_w, oracle.paged_attention(q, kf, vf, "f16", tables, lens, 0.3, window=11))


def test_int8_scale_pin_rejects_misapplied_scales():
    """The pin above is sharp: K and V scales swapped, scales indexed
    [head][block], or a block's scale taken from its logical position in the
    table instead of its physical id each change the output."""
    nb, bs, hkv, d, hq = 7, 16, 3, 32, 6
    kq, vq, ks, vs = _int8_case(5, nb, bs, hkv, d)
    q = W.normal(W.generator(6), (4, hq, d), 0.5, "f16")
    tables = np.array([[6, 2, 0], [3, 5, -1], [1, -1, -1], [4, 0, 2]], np.int32)
    lens = [37, 32, 9, 45]
    want = oracle.paged_attention(q, _premultiplied(kq, ks), _premultiplied(vq, vs), "f16",
                                  tables, lens, 0.3)
    swapped = oracle.paged_attention_int8(q, "f16", kq, vq, vs, ks, tables, lens, 0.3)
    assert np.abs(swapped - want).max() > 1e-2
    # [head][block] order: the same floats read with the wrong strides
    transposed = np.ascontiguousarray(ks.T).reshape(nb, hkv)
    wrong = oracle.paged_attention_int8(q, "f16", kq, vq, transposed, vs, tables, lens, 0.3)
    assert np.abs(wrong - want).max() > 1e-2
    # scale rows in logical order: row j holds the scale of the j-th block of sequence 0
    logical = ks.copy()
    for j, b in enumerate(tables[0]):
        logical[j] = ks[b]
    wrong = oracle.paged_attention_int8(q, "f16", kq, vq, logical, vs, tables, lens, 0.3)
    assert np.abs(wrong - want).max() > 1e-2


def test_append_requantises_earlier_rows_exact_case():
    """A block holding rows at scale 2^-7 receives a row whose max-abs is
    127 * 2^-5: the new scale is 2^-5 and every earlier code c becomes
    round_half_even(c * 2^-7 / 2^-5) = round_half_even(c / 4), ties included."""
    nb, bs, hkv, d = 2, 8, 1, 16
    kq, vq, ks, vs = _pool(nb, bs, hkv, d)
    old = np.array([127, 126, 122, 10, 6, 2, -2, -6, -10, -122, -126, -127, 0, 1, 3, 5],
                   np.float64)
    rows = np.stack([np.roll(old, r) for r in range(3)])        # 3 earlier rows
    x0 = torch.from_numpy((rows * 2.0 ** -7).astype(np.float16)).view(3, 1, d)
    oracle.write_kv_int8(x0, x0, "f16", [8, 9, 10], kq, vq, ks, vs)   # block 1, rows 0..2
    assert ks[1, 0] == np.float32(2.0 ** -7)
    assert np.array_equal(kq[1, :3, 0].astype(np.float64), rows)
    new = np.zeros(d)
    new[3] = 127 * 2.0 ** -5
    new[7] = -40 * 2.0 ** -5
    x1 = torch.from_numpy(new.astype(np.float16)).view(1, 1, d)
    oracle.write_kv_int8(x1, x1, "f16", [11], kq, vq, ks, vs)
    assert ks[1, 0] == np.float32(2.0 ** -5) and vs[1, 0] == np.float32(2.0 ** -5)
    want = np.round(rows / 4.0)            # numpy rounds half to even
    assert np.array_equal(want[0, :3], [32, 32, 30])  # 31.75, 31.5, 30.5
    assert np.array_equal(kq[1, :3, 0].astype(np.float64), want)
    assert np.array_equal(vq[1, :3, 0].astype(np.float64), want)
    assert kq[1, 3, 0, 3] == 127 and kq[1, 3, 0, 7] == -40
    assert not kq[1, 4:].any() and not kq[0].any()   # rows past the write untouched


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_append_requantises_earlier_rows_general(dtype):
    """General case in binary32: after an append with a larger max-abs, each
    earlier code c (old scale s0) becomes clamp(rint(f32(c * s0) / s1), ±127)
    with s1 = max(|new row|, |c * s0|) / 127 over the block, per KV head."""
    nb, bs, hkv, d = 3, 16, 2, 64
    kq, vq, ks, vs = _pool(nb, bs, hkv, d)
    g = W.generator(9)
    x0 = W.normal(g, (5, hkv, d), 0.5, dtype)
    oracle.write_kv_int8(x0, x0, dtype, [32, 33, 34, 35, 36], kq, vq, ks, vs)   # block 2
    c0, s0 = kq[2, :5].copy(), ks[2].copy()
    x1 = W.normal(g, (1, hkv, d), 4.0, dtype)
    oracle.write_kv_int8(x1, x1, dtype, [37], kq, vq, ks, vs)
    f32 = np.float32
    for h in range(hkv):
        deq = c0[:, h].astype(f32) * f32(s0[h])
        new = x1[0, h].float().numpy()
        s1 = f32(max(np.abs(deq).max(), np.abs(new).max())) / f32(127)
        assert ks[2, h] == s1 and s1 > s0[h]
        want = np.clip(np.rint(deq / s1), -127, 127)
        assert np.array_equal(kq[2, :5, h].astype(f32), want)
        assert np.array_equal(kq[2, 5, h].astype(f32), np.clip(np.rint(new / s1), -127, 127))
        # keeping the old codes under the new scale would differ somewhere
        assert not np.array_equal(c0[:, h], kq[2, :5, h])
