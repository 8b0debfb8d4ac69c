"""int8 KV cache on the GPU: quantised writes bit-exact against the oracle's
writer, int8 decode attention within 2e-3 of the binary64 int8 oracle."""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_gb300 as P
import workloads as W
from oracle.allocator import RefAllocator
from tests.cases import assert_close

pytestmark = pytest.mark.gpu


def _pools(nb, bs, hkv, d):
    return (np.zeros((nb, bs, hkv, d), np.int8), np.zeros((nb, bs, hkv, d), np.int8),
            np.zeros((nb, hkv), np.float32), np.zeros((nb, hkv), np.float32))


def _dev(*arrs):
    return [torch.from_numpy(a.copy()).cuda() for a in arrs]


@pytest.mark.parametrize("dtype,bs", [("f16", 16), ("bf16", 32), ("f16", 64)])
def test_int8_write_bit_exact(dtype, bs):
    nb, hkv, d = 48, 8, 128
    g = W.generator(500 + bs)
    a = RefAllocator(nb, bs)
    a.set_free_order(W.permutation(g, nb))
    kq, vq, ks, vs = _pools(nb, bs, hkv, d)
    dk, dv, dks, dvs = _dev(kq, vq, ks, vs)
    seqs = [a.create_sequence() for _ in range(5)]
    # prefill runs, then several decode steps (each re-quantises the tail block)
    for counts in ([37, 1, bs, 2 * bs + 3, 5], [1] * 5, [1] * 5, [3, 1, 0, 1, bs + 1], [1] * 5):
        slots, _ = a.append_tokens(seqs, counts)
        T = len(slots)
        k = W.normal(g, (T, hkv, d), 1.0 + 0.1 * T % 3, dtype)
        v = W.normal(g, (T, hkv, d), 0.7, dtype)
        oracle.write_kv_int8(k, v, dtype, slots, kq, vq, ks, vs)
        P.write_kv_int8(k.cuda(), v.cuda(), torch.tensor(slots, dtype=torch.int64, device="cuda"), dk, dv, dks, dvs)
        torch.cuda.synchronize()
        assert np.array_equal(dk.cpu().numpy(), kq) and np.array_equal(dv.cpu().numpy(), vq)
        assert np.array_equal(dks.cpu().numpy(), ks) and np.array_equal(dvs.cpu().numpy(), vs)


def _int8_case(seed, lens, hq, hkv, bs, dtype, nb=None):
    d = 128
    g = W.generator(seed)
    need = sum(W.blocks_for(L, bs) for L in lens)
    nb = nb or need + 8
    a = RefAllocator(nb, bs)
    a.set_free_order(W.permutation(g, nb))
    kq, vq, ks, vs = _pools(nb, bs, hkv, d)
    seqs = [a.create_sequence() for _ in lens]
    slots, _ = a.append_tokens(seqs, lens)
    k = W.normal(g, (len(slots), hkv, d), 1.0, dtype)
    v = W.normal(g, (len(slots), hkv, d), 1.0, dtype)
    oracle.write_kv_int8(k, v, dtype, slots, kq, vq, ks, vs)
    mb = max(W.blocks_for(L, bs) for L in lens) + 1
    tables = np.full((len(lens), mb), -1, np.int32)
    for i, s in enumerate(seqs):
        t = a.block_table(s)
        tables[i, :len(t)] = t
    q = W.normal(g, (len(lens), hq, d), 1.0, dtype)
    return q, kq, vq, ks, vs, tables, np.array(lens, np.int32)


@pytest.mark.parametrize("hq,hkv,bs,dtype", [(32, 8, 16, "f16"), (32, 8, 32, "bf16"), (32, 4, 16, "f16"),
                                             (8, 8, 16, "bf16"), (16, 8, 16, "f16"), (8, 4, 32, "bf16"),
                                             (32, 16, 16, "f16"), (48, 12, 16, "bf16")])
@pytest.mark.parametrize("window", [0, 100])
def test_int8_decode_matches_oracle(hq, hkv, bs, dtype, window):
    lens = [1, 15, 16, 17, 33, 300, 1000, 2500] + [0]
    q, kq, vq, ks, vs, tables, L = _int8_case(600 + hq + bs, lens, hq, hkv, bs, dtype)
    scale = 128 ** -0.5
    dk, dv, dks, dvs = _dev(kq, vq, ks, vs)
    out = P.attn_decode_int8(q.cuda(), dk, dv, dks, dvs, torch.from_numpy(tables).cuda(),
                             torch.from_numpy(L).cuda(), scale, window=window)
    torch.cuda.synchronize()
    want = oracle.paged_attention_int8(q, dtype, kq, vq, ks, vs, tables, L, scale, window=window)
    assert_close(out, want, what=f"int8 {hq}/{hkv}/{bs}/{dtype}/w{window}")


def test_int8_decode_every_sequence_empty():
    """Every sequence of length 0 over an int8 pool: zero rows, nothing flagged."""
    lens = [0, 0, 0]
    q, kq, vq, ks, vs, tables, L = _int8_case(610, lens, 32, 8, 16, "f16")
    dk, dv, dks, dvs = _dev(kq, vq, ks, vs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.attn_decode_int8(q.cuda(), dk, dv, dks, dvs, torch.from_numpy(tables).cuda(), torch.from_numpy(L).cuda(),
                             128 ** -0.5, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.paged_attention_int8(q, "f16", kq, vq, ks, vs, tables, L, 128 ** -0.5)
    assert_close(out, want, what="int8 every sequence empty")
    assert torch.all(out == 0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_int8_decode_rising_and_jumping_scores(dtype):
    """Key scales that grow block by block, so the scores keep rising along
    each sequence and the running max moves on many tiles (split sequences
    included), and one late block whose scores jump far above all others."""
    lens = [5000, 700, 33, 16, 2100]
    q, kq, vq, ks, vs, tables, L = _int8_case(720, lens, 32, 8, 16, dtype)
    ks = ks.copy()
    for i, n in enumerate(lens):
        nblk = W.blocks_for(n, 16)
        for j in range(nblk):
            ks[tables[i, j], :] = 0.002 * (1 + j)
        if nblk > 20:
            ks[tables[i, nblk - 10], :] = 1.0
    dk, dv, dks, dvs = _dev(kq, vq, ks, vs)
    out = P.attn_decode_int8(q.cuda(), dk, dv, dks, dvs, torch.from_numpy(tables).cuda(), torch.from_numpy(L).cuda(),
                             128 ** -0.5)
    torch.cuda.synchronize()
    want = oracle.paged_attention_int8(q, dtype, kq, vq, ks, vs, tables, L, 128 ** -0.5)
    assert_close(out, want, what=f"int8 rising {dtype}")


def test_int8_decode_long_split_and_16bit_out():
    lens = [30000, 5, 4000]
    q, kq, vq, ks, vs, tables, L = _int8_case(700, lens, 32, 8, 16, "f16")
    dk, dv, dks, dvs = _dev(kq, vq, ks, vs)
    out = P.attn_decode_int8(q.cuda(), dk, dv, dks, dvs, torch.from_numpy(tables).cuda(), torch.from_numpy(L).cuda(),
                             0.088, out_dtype=torch.float16)
    torch.cuda.synchronize()
    want = oracle.paged_attention_int8(q, "f16", kq, vq, ks, vs, tables, L, 0.088)
    assert_close(out, want, what="int8 long")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_int8_full_size_workload_every_sequence(dtype):
    """The int8 row at the bench's shapes (GQA 32/8, 256 sequences of 512-4096
    tokens, random codes and per-block-per-head scales as the bench makes
    them), launched as the bench launches it: every sequence against the int8
    oracle, those cut over several CTAs (merged) included (bf16: the same
    codes with bf16 queries)."""
    w = W.gqa_decode()
    dev = "cuda"
    B, hq, hkv, d, bs = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 100 + 77)
    shape = (w.num_blocks, bs, hkv, d)
    kq = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8, device=dev)
    vq = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8, device=dev)
    ks = torch.rand((w.num_blocks, hkv), generator=g, device=dev) * 0.03 + 0.01
    vs = torch.rand((w.num_blocks, hkv), generator=g, device=dev) * 0.03 + 0.01
    gh = W.generator(w.seed)
    q = W.normal(gh, (B, hq, d), w.sigma, dtype)
    tables, _ = W.scattered_tables(gh, w.lengths, bs, w.num_blocks)
    lens = torch.tensor(w.lengths, dtype=torch.int32)
    # host copy of the blocks the sequences use, ids renumbered (before any kernel of ours runs)
    ids = sorted({int(b) for b in tables.flatten().tolist() if b >= 0})
    local = {b: i for i, b in enumerate(ids)}
    idx = torch.tensor(ids, dtype=torch.long, device=dev)
    kq_h, vq_h = kq[idx].cpu().numpy(), vq[idx].cpu().numpy()
    ks_h, vs_h = ks[idx].cpu().numpy(), vs[idx].cpu().numpy()
    tab_l = np.full(tables.shape, -1, np.int32)
    for i in range(B):
        row = [local[int(b)] for b in tables[i].tolist() if b >= 0]
        tab_l[i, :len(row)] = row
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = P.attn_decode_int8(q.to(dev), kq, vq, ks, vs, tables.to(dev), lens.to(dev), w.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    del kq, vq
    want = oracle.paged_attention_int8(q, dtype, kq_h, vq_h, ks_h, vs_h, tab_l, lens.numpy(), w.scale)
    assert_close(out, want, what=f"{w.name} int8 {dtype}")
