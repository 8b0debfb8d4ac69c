"""A whole mixed step, small: shared prefix, prefill chunks and decode rows in
one packed call, then a width-4 beam split with copy-on-write.

GPU side: the product allocator (C++) -> copy_blocks -> write_kv ->
attn_varlen / attn_decode.  Oracle side: the reference allocator -> oracle
copy / write -> binary64 attention.  Pools are compared bit for bit, outputs
within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_gb300 as P
import workloads as W
from oracle.allocator import RefAllocator
from tests.cases import assert_close

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS, NB = 32, 8, 128, 32, 160


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Both:
    """Runs each allocator call on both allocators and checks they agree."""

    def __init__(self, order):
        self.n = P.BlockAllocator(NB, BS)
        self.r = RefAllocator(NB, BS)
        self.n.set_free_order(order)
        self.r.set_free_order(order)

    def __getattr__(self, name):
        def call(*a, **k):
            x = getattr(self.n, name)(*a, **k)
            y = getattr(self.r, name)(*a, **k)
            assert x == y, (name, x, y)
            return x
        return call


def test_mixed_step_with_prefix_and_cow():
    g = W.generator(55)
    al = Both(W.permutation(g, NB))
    kc = torch.zeros(NB, BS, HKV, D, dtype=torch.float16)
    vc = torch.zeros_like(kc)
    dk, dv = kc.cuda(), vc.cuda()
    ok, ov = _u16(kc).copy(), _u16(vc).copy()   # oracle pools
    scale = D ** -0.5

    def write(slots):
        k = W.normal(g, (len(slots), HKV, D), 1.0, "f16")
        v = W.normal(g, (len(slots), HKV, D), 1.0, "f16")
        oracle.write_kv(k, v, slots, ok, ov)
        P.write_kv(k.cuda(), v.cuda(), torch.tensor(slots, dtype=torch.int64, device="cuda"), dk, dv)

    # a 96-token common prefix (3 whole blocks), written once
    owner = al.create_sequence()
    slots, _ = al.append_tokens([owner], [96])
    write(slots)
    prefix = al.block_table(owner)

    # step 1: two prefill chunks over the prefix, three decode sequences
    chunks = [al.create_sequence(prefix, 96) for _ in range(2)]
    decs = []
    for L in (40, 130, 97):  # cached context before this step
        shared = min(3, (L - 1) // BS)
        s = al.create_sequence(prefix[:shared], shared * BS)
        sl, _ = al.append_tokens([s], [L - shared * BS])
        write(sl)
        decs.append(s)
    q_lens = [50, 64, 1, 1, 1]
    seqs = chunks + decs
    slots, pairs = al.append_tokens(seqs, q_lens)
    assert pairs == []
    write(slots)
    kv_lens = [al.seq_len(s) for s in seqs]
    mb = max(len(al.block_table(s)) for s in seqs) + 1
    tables = torch.full((len(seqs), mb), -1, dtype=torch.int32)
    for i, s in enumerate(seqs):
        t = al.block_table(s)
        tables[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    q = W.normal(g, (int(cu[-1]), HQ, D), 1.0, "f16")
    lens = torch.tensor(kv_lens, dtype=torch.int32)
    out = P.attn_varlen(q.cuda(), dk, dv, tables.cuda(), cu.cuda(), lens.cuda(), max(q_lens), scale)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(dk), ok) and np.array_equal(_u16(dv), ov)
    want = oracle.paged_attention(q, ok.view(np.float16), ov.view(np.float16), "f16", tables.numpy(),
                                  lens.numpy(), scale, cu_q=cu.numpy(), causal=True)
    assert_close(out, want, what="step 1")

    # step 2: every decode sequence forks to width 4; each beam appends a token
    beams = []
    for s in decs:
        beams += [s] + [al.fork(s) for _ in range(3)]
    slots, pairs = al.append_tokens(beams)
    assert len(pairs) == 3 * sum(1 for L in kv_lens[2:] if L % BS != 0)
    if pairs:
        P.check_copy_pairs(pairs, NB)
        oracle.copy_blocks(ok, ov, pairs)
        P.copy_blocks([dk], [dv], torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    write(slots)
    mb = max(len(al.block_table(s)) for s in beams)
    tables = torch.full((len(beams), mb), -1, dtype=torch.int32)
    for i, s in enumerate(beams):
        t = al.block_table(s)
        tables[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    lens = torch.tensor([al.seq_len(s) for s in beams], dtype=torch.int32)
    q = W.normal(g, (len(beams), HQ, D), 1.0, "f16")
    out = P.attn_decode(q.cuda(), dk, dv, tables.cuda(), lens.cuda(), scale)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(dk), ok) and np.array_equal(_u16(dv), ov)
    want = oracle.paged_attention(q, ok.view(np.float16), ov.view(np.float16), "f16", tables.numpy(),
                                  lens.numpy(), scale)
    assert_close(out, want, what="step 2")
    for s in list(beams) + chunks + [owner]:
        al.free_sequence(s)
    assert al.n.num_free == NB
