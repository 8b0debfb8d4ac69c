"""Pins of the oracle's slot write and block copy.

Page 2 ("How to Implement Paged Attention in PyTorch and vLLM", section "Test
and benchmark paged attention against a contiguous KV cache") asks for
write-read round trips within a block, at a block boundary and across
non-contiguous blocks; page 1's copy-on-write paragraph asks that the
diverging block be duplicated.  The read-back here goes through block slicing,
not through the slot formula.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.allocator import RefAllocator
import workloads as W


def _pool(nb, bs, hkv, d):
    return (np.zeros((nb, bs, hkv, d), dtype=np.uint16), np.zeros((nb, bs, hkv, d), dtype=np.uint16))


@pytest.mark.parametrize("n_tokens", [5, 16, 17, 40])
def test_write_read_round_trip(n_tokens):
    nb, bs, hkv, d = 12, 16, 3, 8
    a = RefAllocator(nb, bs)
    g = W.generator(n_tokens)
    a.set_free_order(W.permutation(g, nb))  # non-contiguous blocks
    s = a.create_sequence()
    slots, _ = a.append_tokens([s], [n_tokens])
    k = W.normal(g, (n_tokens, hkv, d), 1.0, "f16")
    v = W.normal(g, (n_tokens, hkv, d), 1.0, "f16")
    kc, vc = _pool(nb, bs, hkv, d)
    assert oracle.write_kv(k, v, slots, kc, vc) == n_tokens
    kb = k.view(torch.int16).numpy().view(np.uint16)
    vb = v.view(torch.int16).numpy().view(np.uint16)
    table = a.block_table(s)
    for j, phys in enumerate(table):
        rows = slice(j * bs, min((j + 1) * bs, n_tokens))
        n = rows.stop - rows.start
        assert np.array_equal(kc[phys, :n], kb[rows])
        assert np.array_equal(vc[phys, :n], vb[rows])
        assert not kc[phys, n:].any()  # nothing beyond the sequence was touched
    untouched = [b for b in range(nb) if b not in table]
    assert not kc[untouched].any() and not vc[untouched].any()


def test_negative_slot_skips_and_bad_slot_rejected():
    kc, vc = _pool(2, 4, 1, 8)
    g = W.generator(3)
    k = W.normal(g, (3, 1, 8), 1.0, "f16")
    assert oracle.write_kv(k, k, [0, -1, 7], kc, vc) == 2
    assert not kc.reshape(8, 8)[1].any()
    with pytest.raises(ValueError):
        oracle.write_kv(k, k, [0, 1, 8], kc, vc)


def test_copy_blocks_duplicates_and_leaves_src():
    nb, bs, hkv, d = 8, 4, 2, 8
    g = W.generator(4)
    kc = W.normal(g, (nb, bs, hkv, d), 1.0, "f16").view(torch.int16).numpy().view(np.uint16).copy()
    vc = W.normal(g, (nb, bs, hkv, d), 1.0, "f16").view(torch.int16).numpy().view(np.uint16).copy()
    k0, v0 = kc.copy(), vc.copy()
    pairs = [(1, 5), (1, 6), (3, 0)]
    oracle.copy_blocks(kc, vc, pairs)
    for s, dd in pairs:
        assert np.array_equal(kc[dd], k0[s]) and np.array_equal(vc[dd], v0[s])
        assert np.array_equal(kc[s], k0[s])
    for b in (1, 2, 3, 4, 7):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
    with pytest.raises(ValueError):
        oracle.copy_blocks(kc, vc, [(0, 8)])
