"""The product's C++ allocator (through the C ABI) against the pinned oracle
allocator, op by op, plus the 6-block trace and a threaded stress test."""
import json
import os
import random
import threading

import pytest

import pagedattention_decode_gb300 as P
from oracle.allocator import DoubleFree, Exhausted, RefAllocator
from tests.conftest import GOLDEN


def test_six_block_trace_native():
    g = json.load(open(os.path.join(GOLDEN, "allocator_trace_6x16.json")))
    a = P.BlockAllocator(g["num_blocks"], g["block_size"])
    for st in g["steps"]:
        if st["op"] == "allocate_for":
            if "error" in st:
                with pytest.raises(P.ExhaustedError):
                    a.allocate_for(st["tokens"])
            else:
                assert a.allocate_for(st["tokens"]) == st["ids"]
        else:
            a.free_all(st["ids"])
        assert a.num_free == st["num_free"]
    for tokens, blocks in g["block_counts"]["tokens_to_blocks"]:
        assert a.blocks_needed(tokens) == blocks


def test_double_free_native():
    a = P.BlockAllocator(4, 16)
    ids = a.allocate_for(32)
    a.free(ids[0])
    with pytest.raises(P.DoubleFreeError):
        a.free(ids[0])
    with pytest.raises(P.DoubleFreeError):
        a.free_all([ids[1], ids[1]])
    assert a.refcount(ids[1]) == 1 and a.num_free == 3


def _same_state(n, r, live):
    assert n.num_free == r.num_free
    for b in range(r.num_blocks):
        assert n.refcount(b) == r.get_refcount(b), b
    for s in live:
        assert n.block_table(s) == r.block_table(s)
        assert n.seq_len(s) == r.seq_len(s)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_differential_random_ops(seed):
    rng = random.Random(seed)
    nb, bs = 48, rng.choice([4, 8, 16])
    n, r = P.BlockAllocator(nb, bs), RefAllocator(nb, bs)
    order = list(range(nb))
    rng.shuffle(order)
    n.set_free_order(order)
    r.set_free_order(order)
    live = []
    for step in range(1500):
        op = rng.random()
        args = None
        try:
            if op < 0.25 or not live:
                k = rng.randint(0, 2)
                donor = rng.choice(live) if live and k else None
                shared = []
                if donor is not None:
                    full = r.seq_len(donor) // bs
                    shared = r.block_table(donor)[:rng.randint(0, full)]
                ref_exc = None
                try:
                    sr = r.create_sequence(shared, len(shared) * bs)
                except Exception as e:  # noqa: BLE001
                    ref_exc = e
                if ref_exc is None:
                    sn = n.create_sequence(shared, len(shared) * bs)
                    assert sn == sr
                    live.append(sr)
                    cnt = rng.randint(0, 3 * bs)
                    args = ([sr], [cnt])
                    try:
                        want = r.append_tokens(*args)
                    except Exhausted:
                        with pytest.raises(P.ExhaustedError):
                            n.append_tokens(*args)
                    else:
                        assert n.append_tokens(*args) == want
            elif op < 0.55:
                batch = rng.sample(live, min(len(live), rng.randint(1, 6)))
                try:
                    want = r.append_tokens(batch)
                except Exhausted:
                    with pytest.raises(P.ExhaustedError):
                        n.append_tokens(batch)
                else:
                    assert n.append_tokens(batch) == want
            elif op < 0.7:
                s = rng.choice(live)
                c = r.fork(s)
                assert n.fork(s) == c
                live.append(c)
            elif op < 0.9:
                s = live.pop(rng.randrange(len(live)))
                r.free_sequence(s)
                n.free_sequence(s)
                n.free_sequence(s)  # second free is a no-op
            else:
                k = rng.randint(0, 40)
                try:
                    want = r.allocate_for(k)
                except Exhausted:
                    with pytest.raises(P.ExhaustedError):
                        n.allocate_for(k)
                else:
                    got = n.allocate_for(k)
                    assert got == want
                    r.free_all(want)
                    n.free_all(got)
        finally:
            pass
        if step % 50 == 0:
            _same_state(n, r, live)
            r.check_invariants()
    _same_state(n, r, live)
    for s in live:
        r.free_sequence(s)
        n.free_sequence(s)
    assert n.num_free == nb == r.num_free
    c = n.counters()
    assert c["allocs"] == r.stats["allocs"] and c["frees"] == r.stats["frees"]
    assert c["cow_copies"] == r.stats["cow_copies"] and c["peak_used"] == r.stats["peak_used"]


def test_cow_pairs_native_match_oracle():
    for a in (P.BlockAllocator(64, 16), RefAllocator(64, 16)):
        p = a.create_sequence()
        a.append_tokens([p], [40])
        beams = [p] + [a.fork(p) for _ in range(3)]
        slots, pairs = a.append_tokens(beams)
        if isinstance(a, RefAllocator):
            assert (slots, pairs) == want
        else:
            want = (slots, pairs)
            assert len(pairs) == 3


def test_threaded_stress():
    """Many threads create, extend, fork and free sequences concurrently
    ('Build a paged KV cache manager from scratch', roadmap item 5); at the end
    every block is back on the free stack and the counters balance."""
    nb = 512
    a = P.BlockAllocator(nb, 16)
    errors = []

    def worker(seed):
        rng = random.Random(seed)
        mine = []
        try:
            for _ in range(400):
                op = rng.random()
                try:
                    if op < 0.3 or not mine:
                        s = a.create_sequence()
                        mine.append(s)
                        a.append_tokens([s], [rng.randint(1, 40)])
                    elif op < 0.6:
                        a.append_tokens(rng.sample(mine, min(len(mine), 3)))
                    elif op < 0.75:
                        mine.append(a.fork(rng.choice(mine)))
                    else:
                        a.free_sequence(mine.pop(rng.randrange(len(mine))))
                except P.ExhaustedError:
                    pass
            for s in mine:
                a.free_sequence(s)
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(16)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    assert a.num_free == nb
    assert all(a.refcount(b) == 0 for b in range(nb))
    c = a.counters()
    assert c["allocs"] == c["frees"]


def test_prefix_trie_differential():
    """Prompts drawn from a few shared system prefixes: match -> create ->
    append -> insert -> finish, with LRU evictions, op by op against the
    reference allocator."""
    rng = random.Random(11)
    nb, bs = 96, 4
    n, r = P.BlockAllocator(nb, bs), RefAllocator(nb, bs)
    prefixes = [[rng.randint(0, 5) for _ in range(rng.randint(4, 16))] for _ in range(4)]
    live = []
    for step in range(600):
        op = rng.random()
        if op < 0.45:
            toks = rng.choice(prefixes) + [rng.randint(0, 5) for _ in range(rng.randint(0, 9))]
            if rng.random() < 0.5:
                shared = r.prefix_match(toks)
                assert n.prefix_match(toks) == shared
                sid = r.create_sequence(shared, len(shared) * bs)
                assert n.create_sequence(shared, len(shared) * bs) == sid
            else:
                sid, stoks = r.create_sequence_prefixed(toks)
                assert n.create_sequence_prefixed(toks) == (sid, stoks)
                shared = r.block_table(sid)
            rest = len(toks) - len(shared) * bs
            try:
                want = r.append_tokens([sid], [rest])
            except Exhausted:
                with pytest.raises(P.ExhaustedError):
                    n.append_tokens([sid], [rest])
                r.free_sequence(sid)
                n.free_sequence(sid)
                continue
            assert n.append_tokens([sid], [rest]) == want
            r.prefix_insert(toks, r.block_table(sid))
            n.prefix_insert(toks, n.block_table(sid))
            live.append(sid)
        elif op < 0.75 and live:
            sid = live.pop(rng.randrange(len(live)))
            r.free_sequence(sid)
            n.free_sequence(sid)
        else:
            k = rng.randint(0, 6)
            assert n.prefix_evict(k) == r.prefix_evict(k)
        if step % 25 == 0:
            _same_state(n, r, live)
            assert n.prefix_nodes == r.nodes
            r.check_invariants()
    for sid in live:
        r.free_sequence(sid)
        n.free_sequence(sid)
    assert n.prefix_evict(nb) == r.prefix_evict(nb)
    assert n.num_free == r.num_free == nb and n.prefix_nodes == 0


def test_prefix_threaded_stress():
    """'Build a paged KV cache manager from scratch', roadmap item 5: many
    threads share prefixes, fork, finish and evict concurrently; at the end,
    after a full eviction, every block is free again."""
    nb, bs = 1024, 8
    a = P.BlockAllocator(nb, bs)
    base = [[t % 7 for t in range(64)], [t % 5 for t in range(40)]]
    errors = []

    def worker(seed):
        rng = random.Random(seed)
        mine = []
        try:
            for _ in range(300):
                op = rng.random()
                try:
                    if op < 0.4:
                        toks = rng.choice(base)[:rng.randint(8, 40)] + [rng.randint(0, 9) for _ in range(5)]
                        s, shared = a.create_sequence_prefixed(toks)
                        mine.append(s)
                        a.append_tokens([s], [len(toks) - shared])
                        a.prefix_insert(toks, a.block_table(s))
                    elif op < 0.55 and mine:
                        mine.append(a.fork(rng.choice(mine)))
                    elif op < 0.85 and mine:
                        a.free_sequence(mine.pop(rng.randrange(len(mine))))
                    else:
                        a.prefix_evict(rng.randint(1, 8))
                except P.ExhaustedError:
                    pass
            for s in mine:
                a.free_sequence(s)
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(16)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    a.prefix_evict(nb)
    assert a.prefix_nodes == 0 and a.num_free == nb
