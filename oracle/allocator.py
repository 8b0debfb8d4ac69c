"""Reference block allocator and sequence bookkeeping (pure Python).

TEST INFRASTRUCTURE ONLY: used by the tests to check the product's C++
allocator (exported through the C ABI) op by op.  It shares no code with it.

What it follows:

* "nanoserve day 14: the block allocator" (page 3), section "What I learned":
  free ids live on a stack, handed-out ids in a set; every id is in exactly
  one of the two; freeing an id that is not handed out is an error;
  ``allocate_for(n)`` needs ceil(n / block_size) blocks and reserves all of
  them or none; reuse is last-in-first-out.  The worked 6-block trace on that
  page pins this class.
* "How to Implement Paged Attention in PyTorch and vLLM" (page 2), section
  "Build the block allocator and block tables in PyTorch": the free stack
  starts as ids num_blocks-1 .. 0 so that the first pop returns 0; a new block
  is taken when pos % block_size == 0; a token lands at offset pos %
  block_size of table[pos // block_size]; freeing a sequence pushes its ids in
  table order.
* "Build a paged KV cache manager from scratch" (page 1), Steps 2 and 3 and
  the copy-on-write paragraph of its Architecture Overview: a block carries a
  refcount (1 on allocation, +1 per retain, -1 per release); a fork shares
  every id and retains each; a shared block is copied on the first divergent
  write.

Readings where the pages are silent or at odds:

* refcounts and the free stack meet as follows: releasing the last reference
  pushes the id back on the stack (page 1 parks zero-ref blocks until an LRU
  reclaim, which is out of scope);
* block-level double free is an error; freeing a sequence twice is a no-op;
* shared prefix blocks are retained once per new holder (page 1 retains
  twice, once in the trie lookup and once in add_request: a bug);
* copy-on-write: appending into a non-full tail whose refcount is > 1 takes a
  new block ``dst``, records the pair (tail, dst), releases the tail and writes
  into ``dst``; the last holder (refcount 1) writes in place; a full tail
  needs no copy.  Page 1's listing never copies (a bug).
* prefix trie (page 1, Step 4, and the LRU reclaim of Step 2): children are
  keyed by a whole block of token ids; ``prefix_match`` walks whole blocks and
  returns their ids without retaining them (the new sequence retains each
  once when it is created -- page 1 retains twice); ``prefix_insert``
  publishes a sequence's whole blocks, the trie holding one reference to each
  node's block (first writer wins on an existing key); ``prefix_evict``
  removes least recently used leaves whose block only the trie still holds
  and releases them.  Recency is a logical clock bumped by every match or
  insert that touches a node.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class Exhausted(Exception):
    """The pool cannot cover the request (page 3's KVCacheExhausted)."""


class DoubleFree(ValueError):
    """An id that is not handed out was freed (page 3's ValueError)."""


class _Node:
    __slots__ = ("children", "block", "last_used", "parent", "key", "serial")

    def __init__(self, parent=None, key=None, block=-1, serial=0):
        self.children = {}
        self.block = block
        self.last_used = 0
        self.parent = parent
        self.key = key
        self.serial = serial


class RefAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_stack: List[int] = list(range(num_blocks - 1, -1, -1))  # top = end
        self.refcount: Dict[int, int] = {}  # handed-out ids only
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.freed: set = set()
        self.next_seq = 0
        self.stats = {"allocs": 0, "frees": 0, "cow_copies": 0, "peak_used": 0}
        self.root = _Node()
        self.clock = 0
        self.node_serial = 0
        self.nodes = 0

    # ---- block level -------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self.free_stack)

    def set_free_order(self, order: Sequence[int]) -> None:
        """Make the next pops return ``order`` (a permutation of the free ids)."""
        if sorted(order) != sorted(self.free_stack):
            raise ValueError("order must be a permutation of the free ids")
        self.free_stack = list(reversed(list(order)))

    def _pop(self) -> int:
        bid = self.free_stack.pop()
        self.refcount[bid] = 1
        self.stats["allocs"] += 1
        used = self.num_blocks - len(self.free_stack)
        self.stats["peak_used"] = max(self.stats["peak_used"], used)
        return bid

    def allocate(self) -> int:
        if not self.free_stack:
            raise Exhausted("all blocks allocated")
        return self._pop()

    def blocks_needed(self, num_tokens: int) -> int:
        if num_tokens < 0:
            raise ValueError("negative token count")
        return (num_tokens + self.block_size - 1) // self.block_size

    def allocate_for(self, num_tokens: int) -> List[int]:
        need = self.blocks_needed(num_tokens)
        if need > len(self.free_stack):
            raise Exhausted(f"need {need} blocks, {len(self.free_stack)} free")
        return [self._pop() for _ in range(need)]

    def retain(self, bid: int) -> None:
        if bid not in self.refcount:
            raise DoubleFree(f"block {bid} is not allocated")
        self.refcount[bid] += 1

    def release(self, bid: int) -> None:
        if bid not in self.refcount:
            raise DoubleFree(f"block {bid} is not allocated")
        self.refcount[bid] -= 1
        if self.refcount[bid] == 0:
            del self.refcount[bid]
            self.free_stack.append(bid)
            self.stats["frees"] += 1

    free = release

    def free_all(self, ids: Sequence[int]) -> None:
        counts: Dict[int, int] = {}
        for b in ids:
            counts[b] = counts.get(b, 0) + 1
        for b, c in counts.items():
            if self.refcount.get(b, 0) < c:
                raise DoubleFree(f"block {b} freed more often than it is held")
        for b in ids:
            self.release(b)

    def get_refcount(self, bid: int) -> int:
        return self.refcount.get(bid, 0)

    # ---- sequence level ----------------------------------------------------
    def create_sequence(self, shared_ids: Sequence[int] = (), shared_tokens: int = 0) -> int:
        if shared_tokens != len(shared_ids) * self.block_size:
            raise ValueError("only whole blocks are shared")
        for b in shared_ids:
            if b not in self.refcount:
                raise DoubleFree(f"shared block {b} is not allocated")
        for b in shared_ids:
            self.retain(b)
        sid = self.next_seq
        self.next_seq += 1
        self.tables[sid] = list(shared_ids)
        self.lens[sid] = shared_tokens
        return sid

    def _blocks_for_appends(self, seq_ids: Sequence[int], counts: Sequence[int]) -> int:
        need = 0
        delta: Dict[int, int] = {}
        for sid, n in zip(seq_ids, counts):
            pos = self.lens[sid]
            table = self.tables[sid]
            for k in range(n):
                p = pos + k
                if p % self.block_size == 0:
                    need += 1
                elif k == 0:
                    tail = table[p // self.block_size]
                    rc = self.refcount[tail] + delta.get(tail, 0)
                    if rc > 1:
                        need += 1
                        delta[tail] = delta.get(tail, 0) - 1
        return need

    def append_tokens(self, seq_ids: Sequence[int], counts: Optional[Sequence[int]] = None
                      ) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Reserve slots for new tokens; all or nothing across the whole call.

        Returns (slots in call order, copy-on-write pairs (src, dst) in order).
        """
        if counts is None:
            counts = [1] * len(seq_ids)
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence appears twice")
        for sid, n in zip(seq_ids, counts):
            if sid not in self.tables:
                raise KeyError(f"unknown sequence {sid}")
            if n < 0:
                raise ValueError("negative token count")
        need = self._blocks_for_appends(seq_ids, counts)
        if need > len(self.free_stack):
            raise Exhausted(f"need {need} blocks, {len(self.free_stack)} free")
        slots: List[int] = []
        pairs: List[Tuple[int, int]] = []
        bs = self.block_size
        for sid, n in zip(seq_ids, counts):
            table = self.tables[sid]
            for _ in range(n):
                pos = self.lens[sid]
                off = pos % bs
                if off == 0:
                    table.append(self._pop())
                else:
                    tail = table[pos // bs]
                    if self.refcount[tail] > 1:
                        dst = self._pop()
                        pairs.append((tail, dst))
                        self.stats["cow_copies"] += 1
                        self.release(tail)
                        table[pos // bs] = dst
                slots.append(table[pos // bs] * bs + off)
                self.lens[sid] = pos + 1
        return slots, pairs

    def fork(self, sid: int) -> int:
        if sid not in self.tables:
            raise KeyError(f"unknown sequence {sid}")
        for b in self.tables[sid]:
            self.retain(b)
        child = self.next_seq
        self.next_seq += 1
        self.tables[child] = list(self.tables[sid])
        self.lens[child] = self.lens[sid]
        return child

    def free_sequence(self, sid: int) -> None:
        if sid in self.freed:
            return
        if sid not in self.tables:
            raise KeyError(f"unknown sequence {sid}")
        for b in self.tables.pop(sid):
            self.release(b)
        del self.lens[sid]
        self.freed.add(sid)

    def block_table(self, sid: int) -> List[int]:
        return list(self.tables[sid])

    def seq_len(self, sid: int) -> int:
        return self.lens[sid]

    # ---- prefix trie -------------------------------------------------------
    def _tick(self) -> int:
        self.clock += 1
        return self.clock

    def prefix_match(self, tokens: Sequence[int]) -> List[int]:
        bs = self.block_size
        node, ids = self.root, []
        for j in range(len(tokens) // bs):
            key = tuple(int(t) for t in tokens[j * bs:(j + 1) * bs])
            child = node.children.get(key)
            if child is None:
                break
            node = child
            node.last_used = self._tick()
            ids.append(node.block)
        return ids

    def create_sequence_prefixed(self, tokens: Sequence[int]) -> Tuple[int, int]:
        shared = self.prefix_match(tokens)
        sid = self.create_sequence(shared, len(shared) * self.block_size)
        return sid, len(shared) * self.block_size

    def prefix_insert(self, tokens: Sequence[int], block_ids: Sequence[int]) -> None:
        bs = self.block_size
        n = min(len(block_ids), len(tokens) // bs)
        for j in range(n):
            if block_ids[j] not in self.refcount:
                raise DoubleFree(f"block {block_ids[j]} is not allocated")
        node = self.root
        for j in range(n):
            key = tuple(int(t) for t in tokens[j * bs:(j + 1) * bs])
            child = node.children.get(key)
            if child is None:
                self.node_serial += 1
                child = _Node(node, key, int(block_ids[j]), self.node_serial)
                node.children[key] = child
                self.retain(child.block)
                self.nodes += 1
            node = child
            node.last_used = self._tick()

    def prefix_evict(self, max_blocks: int) -> List[int]:
        evicted: List[int] = []
        while len(evicted) < max_blocks:
            best = None
            stack = list(self.root.children.values())
            while stack:
                nd = stack.pop()
                if nd.children:
                    stack.extend(nd.children.values())
                elif self.refcount.get(nd.block) == 1:
                    if best is None or (nd.last_used, nd.serial) < (best.last_used, best.serial):
                        best = nd
            if best is None:
                break
            del best.parent.children[best.key]
            self.nodes -= 1
            self.release(best.block)
            evicted.append(best.block)
        return evicted

    def check_invariants(self, exact: bool = True) -> None:
        """Every id is in exactly one of {free stack, handed out}; refcounts
        equal (``exact``) or exceed the number of table entries holding the id
        (page 2's four invariants; page 3's one invariant)."""
        free = self.free_stack
        assert len(set(free)) == len(free), "id twice on the free stack"
        assert not (set(free) & set(self.refcount)), "id both free and handed out"
        assert len(free) + len(self.refcount) == self.num_blocks, "an id went missing"
        held: Dict[int, int] = {}
        for t in self.tables.values():
            for b in t:
                held[b] = held.get(b, 0) + 1
        stack = list(self.root.children.values())
        while stack:
            nd = stack.pop()
            stack.extend(nd.children.values())
            held[nd.block] = held.get(nd.block, 0) + 1
        for b, c in held.items():
            rc = self.refcount.get(b, 0)
            assert rc >= c, f"refcount of {b} is {rc}, held {c}"
        if exact:
            for b, rc in self.refcount.items():
                assert held.get(b, 0) == rc, f"refcount of {b} is {rc}, held {held.get(b, 0)}"
