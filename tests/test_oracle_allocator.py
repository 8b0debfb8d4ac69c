"""Pins of the reference allocator (oracle/allocator.py) against the pages."""
import json
import os
import random

import pytest

from oracle.allocator import DoubleFree, Exhausted, RefAllocator
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_six_block_trace():
    """nanoserve day 14, 'What I learned': the 6-block / 16-token trace."""
    g = _golden("allocator_trace_6x16.json")
    a = RefAllocator(g["num_blocks"], g["block_size"])
    assert a.num_free == g["num_blocks"]
    for st in g["steps"]:
        if st["op"] == "allocate_for":
            if "error" in st:
                with pytest.raises(Exhausted):
                    a.allocate_for(st["tokens"])
            else:
                assert a.allocate_for(st["tokens"]) == st["ids"], st
        elif st["op"] == "free_all":
            a.free_all(st["ids"])
        assert a.num_free == st["num_free"], st
        a.check_invariants(exact=False)


def test_block_counts_ceil():
    g = _golden("allocator_trace_6x16.json")["block_counts"]
    a = RefAllocator(1024, g["block_size"])
    for tokens, blocks in g["tokens_to_blocks"]:
        assert a.blocks_needed(tokens) == blocks
    assert a.blocks_needed(0) == 0
    assert a.allocate_for(0) == []


def test_allocate_for_is_atomic():
    a = RefAllocator(4, 16)
    a.allocate_for(33)  # 3 blocks
    before = (list(a.free_stack), dict(a.refcount))
    with pytest.raises(Exhausted):
        a.allocate_for(17)  # needs 2, 1 free
    assert (a.free_stack, a.refcount) == before


def test_double_free_and_foreign_id_rejected():
    a = RefAllocator(4, 16)
    ids = a.allocate_for(32)
    a.free(ids[0])
    with pytest.raises(DoubleFree):
        a.free(ids[0])
    with pytest.raises(DoubleFree):
        a.free(3)  # never handed out
    before = (list(a.free_stack), dict(a.refcount))
    with pytest.raises(DoubleFree):
        a.free_all([ids[1], ids[1]])  # held once, freed twice: nothing moves
    assert (a.free_stack, a.refcount) == before


def test_slot_trace_block_size_4():
    """Page 2, 'Trace a block-table lookup during one decode step'."""
    g = _golden("slot_trace_bs4.json")
    bs = g["block_size"]
    a = RefAllocator(16, bs)
    # make the pool hand out 5, 2, then 9 (the page's "say physical block 9")
    rest = [i for i in range(16) if i not in (5, 2, 9)]
    a.set_free_order([5, 2, 9] + rest)
    s = a.create_sequence()
    slots, pairs = a.append_tokens([s], [g["seq_len"]])
    assert a.block_table(s) == g["table"] and a.seq_len(s) == g["seq_len"] and pairs == []
    for lk in g["lookups"]:
        assert slots[lk["pos"]] == lk["slot"]
        assert lk["pos"] // bs == lk["logical_block"] and lk["pos"] % bs == lk["offset"]
        assert a.block_table(s)[lk["logical_block"]] == lk["phys"]
    for ap in g["appends"]:
        (slot,), pairs = a.append_tokens([s])
        assert slot == ap["slot"] and pairs == []
        assert a.block_table(s) == ap["table_after"] and a.seq_len(s) == ap["len_after"]
        assert slot == ap["phys"] * bs + ap["offset"]
    nb = g["next_block_trace"]
    assert nb["pos"] // nb["block_size"] == nb["logical_block"]
    assert nb["pos"] % nb["block_size"] == nb["offset"]


def test_fork_doubles_refcounts():
    """Page 1, test_copy_on_write_via_fork: refcounts double on fork."""
    a = RefAllocator(8, 16)
    p = a.create_sequence()
    a.append_tokens([p], [48])
    before = [a.get_refcount(b) for b in a.block_table(p)]
    c = a.fork(p)
    after = [a.get_refcount(b) for b in a.block_table(p)]
    assert after == [2 * r for r in before]
    a.check_invariants()
    a.free_sequence(p)
    a.free_sequence(c)
    a.free_sequence(c)  # second finish is harmless (page 1, test_no_double_free)
    assert a.num_free == 8
    a.check_invariants()


def test_copy_on_write_beams():
    """Width-4 beam split of a non-full tail: three copies, last holder in place."""
    a = RefAllocator(32, 16)
    p = a.create_sequence()
    a.append_tokens([p], [40])  # tail holds 8 of 16
    tail = a.block_table(p)[-1]
    beams = [p] + [a.fork(p) for _ in range(3)]
    assert a.get_refcount(tail) == 4
    slots, pairs = a.append_tokens(beams)
    assert [s for s, _ in pairs] == [tail] * 3
    dsts = [d for _, d in pairs]
    assert len(set(dsts)) == 3 and tail not in dsts
    # beams 0..2 moved to their copies; beam 3 (last holder) writes in place
    for b, d in zip(beams[:3], dsts):
        assert a.block_table(b)[-1] == d
    assert a.block_table(beams[3])[-1] == tail
    assert slots == [d * 16 + 8 for d in dsts] + [tail * 16 + 8]
    assert a.get_refcount(tail) == 1
    a.check_invariants()


def test_full_tail_needs_no_copy():
    a = RefAllocator(32, 16)
    p = a.create_sequence()
    a.append_tokens([p], [32])  # tail full
    beams = [p, a.fork(p)]
    slots, pairs = a.append_tokens(beams)
    assert pairs == []
    t0, t1 = a.block_table(beams[0]), a.block_table(beams[1])
    assert t0[:2] == t1[:2] and t0[2] != t1[2]
    a.check_invariants()


def test_append_batch_atomic_on_exhaustion():
    a = RefAllocator(5, 16)
    p = a.create_sequence()
    a.append_tokens([p], [20])  # 2 blocks, tail 4/16
    beams = [p] + [a.fork(p) for _ in range(3)]
    q = a.create_sequence()
    a.append_tokens([q], [1])  # takes one block: 2 free left, 3 copies needed
    snapshot = (list(a.free_stack), dict(a.refcount), {k: list(v) for k, v in a.tables.items()},
                dict(a.lens))
    with pytest.raises(Exhausted):
        a.append_tokens(beams)
    assert snapshot == (a.free_stack, a.refcount, a.tables, a.lens)


def test_prefix_share_retains_once():
    a = RefAllocator(16, 4)
    owner = a.create_sequence()
    a.append_tokens([owner], [8])
    shared = a.block_table(owner)
    s = a.create_sequence(shared, 8)
    assert [a.get_refcount(b) for b in shared] == [2, 2]
    with pytest.raises(ValueError):
        a.create_sequence(shared, 7)  # only whole blocks are shared
    (slot,), pairs = a.append_tokens([s])
    assert pairs == [] and a.block_table(s)[:2] == shared and len(a.block_table(s)) == 3
    a.check_invariants()


def test_random_ops_keep_invariants():
    rng = random.Random(7)
    a = RefAllocator(64, 8)
    live = []
    for _ in range(3000):
        op = rng.random()
        try:
            if op < 0.3 or not live:
                s = a.create_sequence()
                a.append_tokens([s], [rng.randint(0, 30)])
                live.append(s)
            elif op < 0.55:
                batch = rng.sample(live, min(len(live), rng.randint(1, 5)))
                a.append_tokens(batch)
            elif op < 0.7:
                live.append(a.fork(rng.choice(live)))
            else:
                s = live.pop(rng.randrange(len(live)))
                a.free_sequence(s)
        except Exhausted:
            pass
        a.check_invariants()
    for s in live:
        a.free_sequence(s)
    assert a.num_free == 64 and not a.refcount


def test_prefix_sharing_first_block():
    """Page 1, test_prefix_sharing: two prompts that agree on their first 16
    tokens share the first block id."""
    a = RefAllocator(16, 16)
    p1 = list(range(1, 17)) + [99]
    p2 = list(range(1, 17)) + [100]
    s1 = a.create_sequence()
    a.append_tokens([s1], [len(p1)])
    a.prefix_insert(p1, a.block_table(s1))
    shared = a.prefix_match(p2)
    assert shared == a.block_table(s1)[:1]
    s2 = a.create_sequence(shared, len(shared) * 16)
    a.append_tokens([s2], [len(p2) - 16])
    assert a.block_table(s1)[0] == a.block_table(s2)[0]
    # one retain per holder: s1, the trie and s2 (page 1 would count it twice for s2)
    assert a.get_refcount(shared[0]) == 3
    a.check_invariants()
    a.free_sequence(s1)
    a.free_sequence(s2)
    a.check_invariants()


def test_prefix_demo_prompts_share_leading_block():
    """Page 1's demo: 'The capital of France is' and '... is Paris' share their
    leading 16-token block; 'The capital of Germany is' shares none at bs 16."""
    a = RefAllocator(16, 16)
    prompts = ["The capital of France is", "The capital of France is Paris", "The capital of Germany is"]
    firsts = []
    for p in prompts:
        toks = [ord(c) for c in p]
        shared = a.prefix_match(toks)
        s = a.create_sequence(shared, len(shared) * 16)
        a.append_tokens([s], [len(toks) - len(shared) * 16])
        a.prefix_insert(toks, a.block_table(s))
        firsts.append(a.block_table(s)[0])
        a.free_sequence(s)
    assert firsts[0] == firsts[1] and firsts[2] != firsts[0]
    assert a.num_free > 0
    a.check_invariants()


def test_lru_eviction_order_and_reuse():
    """Page 1, Step 2 (reclaim) and test_eviction_recycles_zero_refcount: once no
    sequence holds a block, the least recently used one is reclaimed first."""
    a = RefAllocator(4, 4)
    sA, sB = a.create_sequence(), a.create_sequence()
    a.append_tokens([sA, sB], [4, 4])
    tA, tB = [1, 2, 3, 4], [5, 6, 7, 8]
    bA, bB = a.block_table(sA)[0], a.block_table(sB)[0]
    a.prefix_insert(tA, [bA])
    a.prefix_insert(tB, [bB])
    a.free_sequence(sA)
    a.free_sequence(sB)
    assert a.num_free == 2          # the trie still holds both blocks
    assert a.prefix_match(tA) == [bA]  # A becomes the most recently used
    assert a.prefix_evict(1) == [bB]
    assert a.prefix_match(tB) == [] and a.prefix_match(tA) == [bA]
    assert a.num_free == 3
    assert a.prefix_evict(5) == [bA] and a.num_free == 4
    a.check_invariants()


def test_evict_takes_leaves_first_and_skips_blocks_in_use():
    a = RefAllocator(8, 4)
    s = a.create_sequence()
    a.append_tokens([s], [8])
    b0, b1 = a.block_table(s)
    a.prefix_insert(list(range(8)), [b0, b1])
    assert a.prefix_evict(4) == []  # s still holds both
    a.free_sequence(s)
    assert a.prefix_evict(4) == [b1, b0]  # the leaf goes first, then its parent
    assert a.num_free == 8
    a.check_invariants()
