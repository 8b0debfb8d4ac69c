"""Prefix trie and LRU reclaim feeding the kernels.

"Build a paged KV cache manager from scratch", Step 4 (prefix tree: a new
request reuses the whole blocks of a cached prompt prefix) and Step 2 (LRU
reclaim of blocks only the cache still holds).  The block tables here are
produced by the trie (``create_sequence_prefixed`` / ``prefix_insert``), by
fork + copy-on-write, and after an eviction by the reuse of the freed ids;
every kernel launch is checked against the binary64 oracle on host pools that
the reference allocator's replay of the same calls wrote.

A token's K/V row is a fixed function of the token prefix it ends (as in a
model, where position p's keys depend on tokens 0..p only), so a sequence
that reuses cached blocks must see exactly the rows it would have written
itself: the outputs are also compared with the oracle on a private,
unshared layout of every sequence's rows.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_gb300 as P
import workloads as W
from oracle.allocator import RefAllocator
from tests.cases import assert_close

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS, NB = 16, 4, 128, 16, 64


class Both:
    """Each allocator call on the product allocator and the reference one; they must agree."""

    def __init__(self, order):
        self.n = P.BlockAllocator(NB, BS)
        self.r = RefAllocator(NB, BS)
        self.n.set_free_order(order)
        self.r.set_free_order(order)

    @property
    def prefix_nodes(self):
        assert self.n.prefix_nodes == self.r.nodes
        return self.r.nodes

    def __getattr__(self, name):
        def call(*a, **k):
            x = getattr(self.n, name)(*a, **k)
            y = getattr(self.r, name)(*a, **k)
            assert x == y, (name, x, y)
            return x
        return call


class Model:
    """Host pools (oracle side), device pools (kernel side), token ids per sequence."""

    def __init__(self, dtype):
        self.dtype = dtype
        tdt = torch.float16 if dtype == "f16" else torch.bfloat16
        nan = torch.full((NB, BS, HKV, D), float("nan"), dtype=tdt)
        self.dk, self.dv = nan.cuda(), nan.clone().cuda()
        self.ok = nan.view(torch.int16).numpy().view(np.uint16).copy()
        self.ov = self.ok.copy()
        self.tokens = {}
        self._rows = {}
        self.g = W.generator(71)

    def row(self, prefix):
        key = tuple(prefix)
        if key not in self._rows:
            g = W.generator(zlib.crc32(np.asarray(key, np.int32).tobytes()))
            self._rows[key] = W.normal(g, (2, HKV, D), 1.0, self.dtype)
        return self._rows[key]

    def write(self, seq, slots, first_pos):
        """Rows of positions first_pos .. first_pos + len(slots) - 1 of seq."""
        toks = self.tokens[seq]
        kv = torch.stack([self.row(toks[:p + 1]) for p in range(first_pos, first_pos + len(slots))])
        k, v = kv[:, 0].contiguous(), kv[:, 1].contiguous()
        oracle.write_kv(k, v, slots, self.ok, self.ov)
        P.write_kv(k.cuda(), v.cuda(), torch.tensor(slots, dtype=torch.int64, device="cuda"), self.dk, self.dv)

    def pools_match(self):
        torch.cuda.synchronize()
        for d, o in ((self.dk, self.ok), (self.dv, self.ov)):
            assert np.array_equal(d.cpu().view(torch.int16).numpy().view(np.uint16), o)

    def private_expectation(self, seqs, q, cu=None, causal=True):
        """Oracle on a layout where every sequence owns fresh blocks holding its own rows."""
        lens = [len(self.tokens[s]) for s in seqs]
        nblk = sum(W.blocks_for(L, BS) for L in lens)
        kp = torch.zeros(nblk, BS, HKV, D, dtype=self.dk.dtype)
        vp = torch.zeros_like(kp)
        mb = max(W.blocks_for(L, BS) for L in lens)
        tables = np.full((len(seqs), mb), -1, np.int32)
        nxt = 0
        for i, s in enumerate(seqs):
            toks = self.tokens[s]
            for p in range(len(toks)):
                j = p // BS
                if p % BS == 0:
                    tables[i, j] = nxt
                    nxt += 1
                kv = self.row(toks[:p + 1])
                kp[tables[i, j], p % BS] = kv[0]
                vp[tables[i, j], p % BS] = kv[1]
        return oracle.paged_attention(q, kp, vp, self.dtype, tables, np.array(lens, np.int32), D ** -0.5,
                                      cu_q=cu, causal=causal)

    def check(self, al, seqs, q_lens, what):
        """One packed varlen call (prefill chunks + decode rows) on the trie's tables."""
        lens = torch.tensor([al.seq_len(s) for s in seqs], dtype=torch.int32)
        assert lens.tolist() == [len(self.tokens[s]) for s in seqs]
        mb = max(len(al.block_table(s)) for s in seqs) + 1
        tables = torch.full((len(seqs), mb), -1, dtype=torch.int32)
        for i, s in enumerate(seqs):
            t = al.block_table(s)
            tables[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
        q = W.normal(self.g, (int(cu[-1]), HQ, D), 1.0, self.dtype)
        if max(q_lens) == 1:
            out = P.attn_decode(q.cuda(), self.dk, self.dv, tables.cuda(), lens.cuda(), D ** -0.5)
            cu_np = None
        else:
            out = P.attn_varlen(q.cuda(), self.dk, self.dv, tables.cuda(), cu.cuda(), lens.cuda(), max(q_lens),
                                D ** -0.5)
            cu_np = cu.numpy()
        self.pools_match()
        want = oracle.paged_attention(q, self.ok, self.ov, self.dtype, tables.numpy(),
                                      lens.numpy(), D ** -0.5, cu_q=cu_np, causal=True)
        assert_close(out, want, what=what)
        # the shared tables reach exactly the rows a private layout holds
        assert np.array_equal(want, self.private_expectation(seqs, q, cu_np))
        return tables


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefix_trie_tables_through_the_kernels(dtype):
    g = W.generator(70)
    al = Both(W.permutation(g, NB))
    m = Model(dtype)
    tok = lambda n, base: [base + int(x) for x in torch.randint(0, 1000, (n,), generator=g)]

    # prompt A: 80 tokens (5 whole blocks) prefilled from scratch, then cached
    A = tok(80, 0)
    a, shared = al.create_sequence_prefixed(A)
    assert shared == 0
    m.tokens[a] = list(A)
    slots, _ = al.append_tokens([a], [80])
    m.write(a, slots, 0)
    m.check(al, [a], [80], "prefill A")
    al.prefix_insert(A, al.block_table(a))
    assert al.prefix_nodes == 5

    # B shares A's first 3 blocks (and 5 tokens more, inside block 3: not
    # shared); C shares 2; D nothing; A decodes one token (a fresh block)
    B = A[:53] + tok(35, 2000)
    C = A[:32] + tok(20, 4000)
    Dp = tok(30, 6000)
    b, sb = al.create_sequence_prefixed(B)
    c, sc = al.create_sequence_prefixed(C)
    d, sd = al.create_sequence_prefixed(Dp)
    assert (sb, sc, sd) == (48, 32, 0)
    tb, ta = al.block_table(b), al.block_table(a)
    assert tb == ta[:3] and al.block_table(c) == ta[:2]
    assert [al.n.refcount(x) for x in ta] == [4, 4, 3, 2, 2]   # owner + trie + sharers
    for s, toks in ((b, B), (c, C), (d, Dp)):
        m.tokens[s] = list(toks)
    m.tokens[a].append(999)
    seqs, q_lens = [b, c, d, a], [88 - 48, 52 - 32, 30, 1]
    slots, pairs = al.append_tokens(seqs, q_lens)
    assert pairs == []
    pos = 0
    for s, n in zip(seqs, q_lens):
        m.write(s, slots[pos:pos + n], len(m.tokens[s]) - n)
        pos += n
    m.check(al, seqs, q_lens, "chunks on shared prefixes + decode row")

    # beams: B and C fork to width 3 and each beam appends a token; their
    # tails are partial, so every beam but the last copies its tail first
    beams = []
    for s in (b, c):
        beams += [s] + [al.fork(s) for _ in range(2)]
    for bm in beams:
        parent = b if bm in (beams[:3]) else c
        m.tokens[bm] = list(m.tokens[parent])
    for i, bm in enumerate(beams):
        m.tokens[bm].append(7000 + i)
    slots, pairs = al.append_tokens(beams)
    assert len(pairs) == 4
    P.check_copy_pairs(pairs, NB)
    oracle.copy_blocks(m.ok, m.ov, pairs)
    P.copy_blocks([m.dk], [m.dv], torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    for bm, sl in zip(beams, slots):
        m.write(bm, [sl], len(m.tokens[bm]) - 1)
    m.check(al, beams, [1] * len(beams), "beams after copy-on-write")

    # everyone but C's beams finishes; B's blocks beyond the shared prefix go
    # back to the stack at once, A's stay cached in the trie
    for s in [a, d] + beams[:3]:
        al.free_sequence(s)
    for s in [a, d] + beams[:3]:
        del m.tokens[s]
    cached_only = [x for x in ta if al.n.refcount(x) == 1]
    assert cached_only == ta[2:]        # blocks 0, 1 are still held by C's beams
    evicted = al.prefix_evict(2)
    assert evicted == [ta[4], ta[3]]    # least recently used leaf first, then its parent
    assert al.prefix_nodes == 3

    # E reuses the freed ids (the stack is LIFO: the evicted ids come back first);
    # F still finds A's first 3 blocks in the trie
    E = tok(40, 8000)
    e, se = al.create_sequence_prefixed(E)
    F = A[:48] + tok(17, 9000)
    f, sf = al.create_sequence_prefixed(F)
    assert (se, sf) == (0, 48) and al.block_table(f) == ta[:3]
    m.tokens[e], m.tokens[f] = list(E), list(F)
    slots, pairs = al.append_tokens([e, f], [40, 17])
    assert pairs == []
    m.write(e, slots[:40], 0)
    m.write(f, slots[40:], 48)
    assert set(evicted) <= set(al.block_table(e)) | set(al.block_table(f))
    live = [e, f] + beams[3:]
    for bm in beams[3:]:
        m.tokens[bm].append(7100 + bm)
    slots, pairs = al.append_tokens(beams[3:])
    for bm, sl in zip(beams[3:], slots):
        m.write(bm, [sl], len(m.tokens[bm]) - 1)
    if pairs:
        P.check_copy_pairs(pairs, NB)
        oracle.copy_blocks(m.ok, m.ov, pairs)
        P.copy_blocks([m.dk], [m.dv], torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    m.check(al, live, [40, 17, 1, 1, 1], "after eviction and reuse of the freed ids")
    for s in live:
        al.free_sequence(s)
    al.prefix_evict(NB)
    assert al.n.num_free == NB and al.prefix_nodes == 0
