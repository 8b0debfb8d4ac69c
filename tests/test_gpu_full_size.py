"""Full-size workloads, launched as the bench launches them, checked on sampled
outputs the oracle computes one by one.

* the mixed packed step (2048-token shared prefix, 16 prefill chunks of 512
  rows, 240 decode rows, block_size 32) and its width-4 beam split with
  copy-on-write -- built by the bench's own MixedStep;
* the GPT-2-shaped 12-layer decode step (one pool per layer, one shared table,
  write then attend in every layer).

The oracle's copy of each sampled sequence's blocks is taken from the device
before any kernel of this project runs, and the step's writes and copies are
replayed on it by the oracle itself.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_gb300 as P
import workloads as W
from tests.cases import assert_close

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Subset:
    """Host copy of the blocks a few sequences use, with ids renumbered."""

    def __init__(self, k_cache, v_cache, table_rows):
        ids = sorted({int(b) for row in table_rows for b in row if b >= 0})
        self.local = {b: i for i, b in enumerate(ids)}
        idx = torch.tensor(ids, dtype=torch.long, device=k_cache.device)
        self.k = _u16(k_cache[idx]).copy()
        self.v = _u16(v_cache[idx]).copy()
        self.bs = k_cache.shape[1]

    def table(self, row):
        return [self.local[int(b)] for b in row if b >= 0]

    def write(self, slots, k, v):
        keep = [(i, s) for i, s in enumerate(slots) if s // self.bs in self.local]
        if not keep:
            return
        loc = [self.local[s // self.bs] * self.bs + s % self.bs for _, s in keep]
        rows = torch.tensor([i for i, _ in keep])
        oracle.write_kv(k[rows], v[rows], loc, self.k, self.v)

    def copy(self, pairs):
        loc = [(self.local[s], self.local[d]) for s, d in pairs if s in self.local and d in self.local]
        if loc:
            oracle.copy_blocks(self.k, self.v, loc)

    def attend(self, q_rows, table_rows, lens, scale, dtype):
        mb = max(len(t) for t in table_rows)
        tab = np.full((len(table_rows), mb), -1, dtype=np.int32)
        for i, t in enumerate(table_rows):
            tab[i, :len(t)] = t
        kf = self.k.view(np.float16) if dtype == "f16" else self.k
        vf = self.v.view(np.float16) if dtype == "f16" else self.v
        return oracle.paged_attention(q_rows, kf, vf, dtype, tab, np.array(lens, dtype=np.int32), scale)


def test_mixed_step_full_size_sampled():
    import bench
    dev = torch.device("cuda", torch.cuda.current_device())
    m = bench.MixedStep(dev)
    s1, s2 = m.s1, m.s2
    tab1 = s1["tables"].cpu()
    lens1 = m.s1_lens_host
    rng = np.random.default_rng(5)
    chunk_ids = [0, 7, 15]
    dec_ids = sorted(m.nchunk + rng.choice(m.ndec, size=5, replace=False))
    tab2 = s2["tables"].cpu()
    beam_ids = [0, 1, 2, 3, 64, 65, 66, 67, 127]
    rows_needed = [tab1[i].tolist() for i in chunk_ids + dec_ids] + [tab2[i].tolist() for i in beam_ids]
    sub = Subset(m.k_cache, m.v_cache, rows_needed)   # before any of our kernels ran
    k1, v1, slots1 = s1["k"].cpu(), s1["v"].cpu(), s1["slots"].cpu().tolist()
    k2, v2, slots2 = s2["k"].cpu(), s2["v"].cpu(), s2["slots"].cpu().tolist()
    pairs2 = s2["pairs"].cpu().tolist()

    m.step1()
    torch.cuda.synchronize()
    out1 = m.out1.clone()
    m.step2()
    torch.cuda.synchronize()
    out2 = m.out2.clone()
    assert int(m.err.item()) == 0

    # oracle replay of step 1
    sub.write(slots1, k1, v1)
    q1 = s1["q"].cpu()
    cu = s1["cu"].cpu().tolist()
    for i in chunk_ids:
        ql, kv = cu[i + 1] - cu[i], lens1[i]
        for r in (0, 1, 100, ql - 1):
            vis = kv - ql + r + 1  # row r sees keys t <= kv - ql + r
            want = sub.attend(q1[cu[i] + r:cu[i] + r + 1], [sub.table(tab1[i].tolist())], [vis], m.scale, "f16")
            assert_close(out1[cu[i] + r:cu[i] + r + 1], want, what=f"chunk {i} row {r}")
    for i in dec_ids:
        want = sub.attend(q1[cu[i]:cu[i] + 1], [sub.table(tab1[i].tolist())], [lens1[i]], m.scale, "f16")
        assert_close(out1[cu[i]:cu[i] + 1], want, what=f"decode row {i}")
    # oracle replay of step 2: copies, writes, decode of the sampled beams
    sub.copy(pairs2)
    sub.write(slots2, k2, v2)
    q2 = s2["q"].cpu()
    for i in beam_ids:
        want = sub.attend(q2[i:i + 1], [sub.table(tab2[i].tolist())], [m.s2_lens_host[i]], m.scale, "f16")
        assert_close(out2[i:i + 1], want, what=f"beam {i}")


def test_gpt2_shaped_twelve_layers_sampled():
    w = W.gpt2_decode()
    dev = "cuda"
    g = W.generator(w.seed)
    tables, _ = W.scattered_tables(g, [L + 1 for L in w.lengths], w.block_size, w.num_blocks)
    lens = torch.tensor([L + 1 for L in w.lengths], dtype=torch.int32)
    slots = [int(tables[i, L // w.block_size]) * w.block_size + L % w.block_size for i, L in enumerate(w.lengths)]
    pick = [0, 13, 31]
    rows = [tables[i].tolist() for i in pick]
    dt, dtables, dlens = tables.to(dev), tables.to(dev), lens.to(dev)
    dslots = torch.tensor(slots, dtype=torch.int64, device=dev)
    for layer in range(w.layers):
        shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
        kc = W.normal_device(200 + 2 * layer, shape, 1.0, w.dtype, dev)
        vc = W.normal_device(201 + 2 * layer, shape, 1.0, w.dtype, dev)
        sub = Subset(kc, vc, rows)
        q = W.normal(g, (w.batch, w.num_q_heads, w.head_dim), 1.0, w.dtype)
        kn = W.normal(g, (w.batch, w.num_kv_heads, w.head_dim), 1.0, w.dtype)
        vn = W.normal(g, (w.batch, w.num_kv_heads, w.head_dim), 1.0, w.dtype)
        P.write_kv(kn.to(dev), vn.to(dev), dslots, kc, vc)
        out = P.attn_decode(q.to(dev), kc, vc, dtables, dlens, w.scale)
        torch.cuda.synchronize()
        sub.write(slots, kn, vn)
        for j, i in enumerate(pick):
            want = sub.attend(q[i:i + 1], [sub.table(rows[j])], [int(lens[i])], w.scale, "f16")
            assert_close(out[i:i + 1], want, what=f"layer {layer} seq {i}")
        del kc, vc
