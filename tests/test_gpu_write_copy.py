"""Slot write and block copy on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_gb300 as P
import workloads as W
from oracle.allocator import RefAllocator

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,hkv,d,bs", [("f16", 12, 64, 16), ("bf16", 8, 128, 32), ("f16", 8, 128, 16),
                                            ("f16", 1, 64, 64)])
def test_write_kv_bit_exact(dtype, hkv, d, bs):
    g = W.generator(100 + hkv + d + bs)
    nb = 40
    kc = W.normal(g, (nb, bs, hkv, d), 1.0, dtype)
    vc = W.normal(g, (nb, bs, hkv, d), 1.0, dtype)
    # slots from the reference allocator: several sequences, scattered blocks,
    # within a block, at boundaries and across non-contiguous blocks
    a = RefAllocator(nb, bs)
    a.set_free_order(W.permutation(g, nb))
    seqs = [a.create_sequence() for _ in range(5)]
    a.append_tokens(seqs, [3, bs - 1, bs, 2 * bs + 5, 1])
    slots, _ = a.append_tokens(seqs, [1, 1, 2, bs + 3, 0])
    slots = slots + [-1, -5]  # negative slots are skipped
    T = len(slots)
    k = W.normal(g, (T, hkv, d), 1.0, dtype)
    v = W.normal(g, (T, hkv, d), 1.0, dtype)
    kw, vw = _u16(kc).copy(), _u16(vc).copy()
    oracle.write_kv(k, v, slots, kw, vw)
    dk, dv = kc.cuda(), vc.cuda()
    P.write_kv(k.cuda(), v.cuda(), torch.tensor(slots, dtype=torch.int64, device="cuda"), dk, dv)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(dk), kw) and np.array_equal(_u16(dv), vw)


def test_write_kv_strided_rows_and_bad_slot_flag():
    g = W.generator(7)
    nb, bs, hkv, d = 8, 16, 2, 64
    kc = torch.zeros(nb, bs, hkv, d, dtype=torch.float16)
    vc = torch.zeros_like(kc)
    qkv = W.normal(g, (5, 3, hkv, d), 1.0, "f16")  # k and v are views into a packed buffer
    k, v = qkv[:, 1], qkv[:, 2]
    slots = [0, 17, 127, 128, 5]  # 128 is outside the pool of 128 slots
    kw, vw = _u16(kc).copy(), _u16(vc).copy()
    oracle.write_kv(k, v, [s if s < 128 else -1 for s in slots], kw, vw)
    dq = qkv.cuda()
    dk, dv = kc.cuda(), vc.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.write_kv(dq[:, 1], dq[:, 2], torch.tensor(slots, device="cuda"), dk, dv, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & P.DEVERR["slot"]
    assert np.array_equal(_u16(dk), kw) and np.array_equal(_u16(dv), vw)


@pytest.mark.parametrize("layers,bs,hkv,d", [(1, 16, 8, 128), (3, 32, 8, 128), (12, 16, 12, 64), (40, 16, 2, 64)])
def test_copy_blocks_bit_exact(layers, bs, hkv, d):
    g = W.generator(200 + layers)
    nb = 24
    ks = [W.normal(g, (nb, bs, hkv, d), 1.0, "f16") for _ in range(layers)]
    vs = [W.normal(g, (nb, bs, hkv, d), 1.0, "f16") for _ in range(layers)]
    pairs = [(3, 10), (3, 11), (5, 0), (23, 7)]
    P.check_copy_pairs(pairs, nb)
    want = []
    for kk, vv in zip(ks, vs):
        kw, vw = _u16(kk).copy(), _u16(vv).copy()
        oracle.copy_blocks(kw, vw, pairs)
        want.append((kw, vw))
    dks = [x.cuda() for x in ks]
    dvs = [x.cuda() for x in vs]
    P.copy_blocks(dks, dvs, torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    for (kw, vw), dk, dv in zip(want, dks, dvs):
        assert np.array_equal(_u16(dk), kw) and np.array_equal(_u16(dv), vw)


def test_copy_blocks_bad_pair_flagged_and_skipped():
    g = W.generator(9)
    kc = W.normal(g, (4, 16, 1, 64), 1.0, "f16")
    vc = W.normal(g, (4, 16, 1, 64), 1.0, "f16")
    kw, vw = _u16(kc).copy(), _u16(vc).copy()
    oracle.copy_blocks(kw, vw, [(1, 2)])
    dk, dv = kc.cuda(), vc.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.copy_blocks([dk], [dv], torch.tensor([[1, 2], [0, 4]], dtype=torch.int64, device="cuda"), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & P.DEVERR["pair"]
    assert np.array_equal(_u16(dk), kw) and np.array_equal(_u16(dv), vw)
