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
