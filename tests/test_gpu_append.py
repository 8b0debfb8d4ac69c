"""pkv_attn_decode_append: the step's new key / value written by the decode
kernel itself, against pkv_write_kv followed by pkv_attn_decode (bit for bit)
and against the binary64 oracle (pools written by the oracle's slot write on
host copies, then binary64 attention)."""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_gb300 as P
import workloads as W
from tests.cases import Subset, assert_close, decode_case

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().contiguous().view(torch.int16)


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _oracle_pools(case, kn, vn):
    ok, ov = _u16(case.k_cache).copy(), _u16(case.v_cache).copy()
    oracle.write_kv(kn, vn, _slots(case).tolist(), ok, ov)
    return ok, ov


def _new_rows(case, seed):
    B = case.lens.numel()
    hkv, d = case.k_cache.shape[2], case.k_cache.shape[3]
    g = W.generator(seed)
    return (W.normal(g, (B, hkv, d), 1.0, case.dtype), W.normal(g, (B, hkv, d), 1.0, case.dtype))


def _slots(case):
    bs = case.k_cache.shape[1]
    out = []
    for s, L in enumerate(case.lens.tolist()):
        if L == 0:
            out.append(-1)
        else:
            out.append(int(case.tables[s, (L - 1) // bs]) * bs + (L - 1) % bs)
    return torch.tensor(out, dtype=torch.int64)


def _both(case, kn, vn, window=0):
    """(out, k, v) of the fused call and of write-then-decode, on copies of the pools."""
    dev = "cuda"
    q, t, lens = case.q.to(dev), case.tables.to(dev), case.lens.to(dev)
    k1, v1 = case.k_cache.to(dev), case.v_cache.to(dev)
    k2, v2 = k1.clone(), v1.clone()
    out1 = P.attn_decode(q, k1, v1, t, lens, case.scale, window=window, k_new=kn.to(dev), v_new=vn.to(dev))
    P.write_kv(kn.to(dev), vn.to(dev), _slots(case).to(dev), k2, v2)
    out2 = P.attn_decode(q, k2, v2, t, lens, case.scale, window=window)
    torch.cuda.synchronize()
    return (out1, k1, v1), (out2, k2, v2)


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [(32, 8, 128, 16, "f16"), (12, 12, 64, 32, "bf16"),
                                                (32, 16, 128, 16, "f16"), (8, 2, 64, 64, "bf16")])
def test_append_equals_write_then_decode(hq, hkv, d, bs, dtype):
    """Empty and one-key sequences, block-boundary lengths, and a long
    sequence cut over many CTAs (its new row sits in its last part); with 16
    KV heads the heads are split over two head groups, each writing its own."""
    lens = [0, 1, 15, 16, 17, 33, 300, 1000, 40000, 2500]
    case = decode_case(170 + hkv + bs, lens, hq, hkv, d, bs, dtype)
    kn, vn = _new_rows(case, 171 + hkv)
    (o1, k1, v1), (o2, k2, v2) = _both(case, kn, vn)
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    assert torch.equal(o1, o2)
    # and the oracle: the new rows written into host copies of the pools by
    # the oracle's own slot write, then binary64 attention over them
    ok, ov = _oracle_pools(case, kn, vn)
    assert np.array_equal(_u16(k1), ok) and np.array_equal(_u16(v1), ov)
    want = oracle.paged_attention(case.q, ok, ov, case.dtype, case.tables.numpy(), case.lens.numpy(), case.scale)
    assert_close(o1, want, what=f"append {hq}/{hkv}/{d}/{bs}/{dtype}")


@pytest.mark.parametrize("window", [1, 17, 4096])
def test_append_with_window(window):
    lens = [1, 15, 16, 17, 0, 33, 300, 9000]
    case = decode_case(180 + window, lens, 32, 8, 128, 16, "f16")
    kn, vn = _new_rows(case, 181)
    (o1, k1, v1), (o2, k2, v2) = _both(case, kn, vn, window=window)
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    assert torch.equal(o1, o2)
    ok, ov = _oracle_pools(case, kn, vn)
    assert np.array_equal(_u16(k1), ok) and np.array_equal(_u16(v1), ov)
    want = oracle.paged_attention(case.q, ok, ov, case.dtype, case.tables.numpy(), case.lens.numpy(), case.scale,
                                  window=window)
    assert_close(o1, want, what=f"append, window {window}")


def test_append_bad_block_is_flagged_and_not_written():
    lens = [40, 20]
    case = decode_case(190, lens, 8, 2, 64, 16, "f16")
    kn, vn = _new_rows(case, 191)
    t = case.tables.clone()
    t[1, (20 - 1) // 16] = case.k_cache.shape[0] + 5  # the new row's block: out of range
    dev = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    k1, v1 = case.k_cache.to(dev), case.v_cache.to(dev)
    before = _bits(k1).clone()
    P.attn_decode(case.q.to(dev), k1, v1, t.to(dev), case.lens.to(dev), case.scale, err=err,
                  k_new=kn.to(dev), v_new=vn.to(dev))
    torch.cuda.synchronize()
    assert int(err.item()) & P.DEVERR["block"]
    # sequence 0's row was written, nothing else changed
    slot0 = int(case.tables[0, (40 - 1) // 16]) * 16 + (40 - 1) % 16
    changed = (_bits(k1) != before).view(-1, 2 * 64).any(dim=1).nonzero().view(-1).tolist()
    assert changed == [slot0] or changed == []
    assert torch.equal(k1.view(-1, 2, 64)[slot0].cpu(), kn[0])


def test_append_full_size_workload_every_sequence():
    """The GQA 32/8 workload (256 sequences of 512-4096 tokens) with each
    sequence's new row written by the decode kernel: outputs and pools bit
    for bit those of pkv_write_kv + pkv_attn_decode, and every output within
    2e-3 of the oracle's slot write followed by binary64 attention."""
    w = W.gqa_decode()
    dev = "cuda"
    bs = w.block_size
    shape = (w.num_blocks, bs, w.num_kv_heads, w.head_dim)
    k1 = W.normal_device(w.seed * 10 + 1, shape, w.sigma, w.dtype, dev)
    v1 = W.normal_device(w.seed * 10 + 2, shape, w.sigma, w.dtype, dev)
    g = W.generator(w.seed)
    q = W.normal(g, (w.batch, w.num_q_heads, w.head_dim), w.sigma, w.dtype)
    tables, _ = W.scattered_tables(g, w.lengths, bs, w.num_blocks)
    kn = W.normal(g, (w.batch, w.num_kv_heads, w.head_dim), w.sigma, w.dtype)
    vn = W.normal(g, (w.batch, w.num_kv_heads, w.head_dim), w.sigma, w.dtype)
    lens = torch.tensor(w.lengths, dtype=torch.int32)
    slots = [int(tables[i, (L - 1) // bs]) * bs + (L - 1) % bs for i, L in enumerate(w.lengths)]
    rows = [tables[i].tolist() for i in range(w.batch)]
    sub = Subset(k1, v1, rows)   # before any kernel of ours runs
    k2, v2 = k1.clone(), v1.clone()
    qd, td, ld = q.to(dev), tables.to(dev), lens.to(dev)
    out1 = P.attn_decode(qd, k1, v1, td, ld, w.scale, k_new=kn.to(dev), v_new=vn.to(dev))
    P.write_kv(kn.to(dev), vn.to(dev), torch.tensor(slots, dtype=torch.int64, device=dev), k2, v2)
    out2 = P.attn_decode(qd, k2, v2, td, ld, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    del k1, v1, k2, v2
    sub.write(slots, kn, vn)
    want = sub.attend(q, [sub.table(r) for r in rows], w.lengths, w.scale, w.dtype)
    assert_close(out1, want, what=w.name + " append")
