"""Decode attention on the GPU against the binary64 oracle (max-abs 2e-3)."""
import math

import numpy as np
import pytest
import torch

import pagedattention_decode_gb300 as P
import workloads as W
from tests.cases import TOL, Subset, assert_close, decode_case

pytestmark = pytest.mark.gpu


def run(case, out_dtype=torch.float32, err=None):
    c = case.to("cuda")
    out = P.attn_decode(c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, out_dtype=out_dtype, err=err)
    torch.cuda.synchronize()
    return out


def test_tiny_workload_exact_lengths():
    """1 layer, 12/12 heads, D 64, bs 16, fp16, 64-block pool, L = 40/20/16/30."""
    w = W.tiny_decode()
    case = decode_case(w.seed, w.lengths, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                       w.dtype, num_blocks=w.num_blocks)
    assert_close(run(case), case.oracle(), what="tiny")


SHAPES = [
    # hq, hkv, d, bs, dtype
    (32, 8, 128, 16, "f16"),
    (32, 8, 128, 32, "bf16"),
    (12, 12, 64, 16, "f16"),
    (16, 2, 128, 16, "f16"),   # 8 query heads per KV head
    (4, 2, 64, 32, "bf16"),    # 2 per KV head
    (8, 8, 128, 64, "bf16"),
    (24, 24, 64, 16, "f16"),   # two KV-head groups per sequence
    (2, 1, 128, 128, "f16"),
    (16, 8, 128, 16, "bf16"),  # 2 per KV head, both parts of P in one MMA
    (64, 16, 128, 16, "f16"),  # 4 per KV head, two head groups of 8 KV heads
]


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", SHAPES)
def test_ragged_lengths(hq, hkv, d, bs, dtype):
    lens = [1, 15, 16, 17, 0, 33, 300, 1000, 127, 2]
    case = decode_case(11 + hq + bs, lens, hq, hkv, d, bs, dtype, sigma=1.0 if dtype == "f16" else 0.5)
    got = run(case)
    assert_close(got, case.oracle(), what=f"{hq}/{hkv}/{d}/{bs}/{dtype}")
    assert torch.all(got[4] == 0)  # empty sequence -> zero row


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_many_sequences_split_across_ctas(dtype):
    g = W.generator(5)
    lens = W.uniform_lengths(g, 300, 1, 700)
    case = decode_case(6, lens, 32, 8, 128, 16, dtype)
    assert_close(run(case), case.oracle(), what="300 seqs")


def test_one_long_sequence_spans_every_cta():
    case = decode_case(8, [40000], 8, 2, 128, 16, "bf16", sigma=0.5)
    assert_close(run(case), case.oracle(), what="40k")


def test_skewed_lengths():
    lens = [1024 << k for k in range(5)] + [3, 5000]
    case = decode_case(9, lens, 32, 8, 128, 16, "bf16", sigma=0.5)
    assert_close(run(case), case.oracle(), what="skew")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_16bit_output(dtype):
    lens = [5, 64, 100, 1000]
    case = decode_case(10, lens, 32, 8, 128, 16, dtype)
    got = run(case, out_dtype=W.DTYPES[dtype])
    assert got.dtype == W.DTYPES[dtype]
    assert_close(got, case.oracle(), what="16-bit out")


def test_block_permutation_gives_identical_bits():
    """The arithmetic order depends only on logical positions: relocating the
    physical blocks does not change a single output bit."""
    lens = [700, 3, 48, 1500]
    a = decode_case(12, lens, 32, 8, 128, 16, "f16")
    nb = a.k_cache.shape[0]
    perm = torch.tensor(W.permutation(W.generator(13), nb))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    k2 = torch.empty_like(a.k_cache)
    v2 = torch.empty_like(a.v_cache)
    k2[perm] = a.k_cache
    v2[perm] = a.v_cache
    t2 = a.tables.clone()
    m = t2 >= 0
    t2[m] = perm[t2[m].long()].int()
    b = type(a)(a.q, k2, v2, t2, a.lens, a.scale, a.dtype)
    assert torch.equal(run(a), run(b))


def test_block_size_change_within_tolerance():
    lens = [333, 64, 1]
    a = decode_case(14, lens, 16, 4, 64, 16, "f16", poison=False)
    # same logical K/V re-laid out in 32-token blocks
    g = W.generator(15)
    tabs, _ = W.scattered_tables(g, lens, 32, 40)
    k2 = torch.zeros(40, 32, 4, 64, dtype=torch.float16)
    v2 = torch.zeros_like(k2)
    for i, L in enumerate(lens):
        for t in range(L):
            src = int(a.tables[i, t // 16]), t % 16
            dst = int(tabs[i, t // 32]), t % 32
            k2[dst] = a.k_cache[src]
            v2[dst] = a.v_cache[src]
    b = type(a)(a.q, k2, v2, tabs, a.lens, a.scale, a.dtype)
    want = a.oracle()
    assert np.array_equal(want, b.oracle())
    assert_close(run(a), want)
    assert_close(run(b), want)


def test_bad_table_entry_is_flagged_not_trapped():
    case = decode_case(16, [40, 20], 8, 2, 64, 16, "f16")
    case.tables[1, 0] = case.k_cache.shape[0] + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run(case, err=err)
    assert int(err.item()) & P.DEVERR["block"]


def test_length_beyond_table_is_flagged():
    case = decode_case(17, [40, 20], 8, 2, 64, 16, "f16", extra_table_cols=0)
    case.lens[1] = 10000
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(case, err=err)
    assert int(err.item()) & P.DEVERR["length"]
    assert torch.all(out[1] == 0)


def test_gqa_mapping_contiguous_groups():
    hq, hkv, d, L = 32, 8, 128, 50
    case = decode_case(18, [L], hq, hkv, d, 16, "f16", poison=False)
    # V of KV head j is the constant j: output head h must read h // 4
    case.v_cache[:] = torch.arange(hkv, dtype=torch.float16).view(1, 1, hkv, 1)
    got = run(case)
    want = (torch.arange(hq) // (hq // hkv)).float().view(hq, 1).expand(hq, d)
    assert torch.allclose(got[0].cpu(), want, atol=1e-6)


@pytest.mark.parametrize("lens", [[16, 32] * 16,            # 32 sequences, 48 sub-blocks: whole
                                  [32] * 31 + [33],         # 32 sequences, exactly 64 + 1: even split
                                  [16] * 40,                # 40 sequences, 40 sub-blocks: even split
                                  [32] * 32,                # 32 sequences, exactly 64: whole
                                  [5, 0, 40]])              # the even split would cut the third
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (12, 12, 64)])
def test_small_calls_one_cta_per_sequence(lens, hq, hkv, d):
    """Calls of at most 32 sequences and 64 sub-blocks give each sequence a
    CTA of its own (no cut, nothing to merge); just past either bound the
    even split takes over.  Both sides of the bounds against the oracle."""
    case = decode_case(97 + len(lens) + d, lens, hq, hkv, d, 16, "f16")
    assert_close(run(case), case.oracle(), what=f"{len(lens)} sequences, {sum(-(-L // 16) for L in lens)} sub-blocks")


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (12, 12, 64)])
@pytest.mark.parametrize("window", [0, 16])
def test_every_sequence_empty(hq, hkv, d, window):
    """A batch whose sequences all have length 0: there is nothing to split,
    every output row is zero, nothing is flagged, and the pool (NaN in every
    slot, since no sequence holds one) is never read."""
    case = decode_case(91 + d, [0, 0, 0, 0, 0], hq, hkv, d, 16, "f16")
    assert torch.isnan(case.k_cache.float()).all()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = case.to("cuda")
    got = P.attn_decode(c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, window=window, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got, case.oracle(), what="every sequence empty")
    assert torch.all(got == 0)


@pytest.mark.parametrize("wl", [W.gqa_decode, W.long_skewed_decode])
def test_full_size_workload_every_sequence(wl):
    """The full-size workloads, launched as the bench launches them; every
    sequence checked against the oracle, those the even split of sub-blocks
    cuts over several CTAs (their outputs come from the merge) included."""
    import bench
    w = wl()
    dev = "cuda"
    kc = W.normal_device(w.seed * 10 + 1, (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim), w.sigma,
                         w.dtype, dev)
    vc = W.normal_device(w.seed * 10 + 2, kc.shape, w.sigma, w.dtype, dev)
    g = W.generator(w.seed)
    q = W.normal(g, (w.batch, w.num_q_heads, w.head_dim), w.sigma, w.dtype)
    tables, _ = W.scattered_tables(g, w.lengths, w.block_size, w.num_blocks)
    lens = torch.tensor(w.lengths, dtype=torch.int32)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert bench.split_records(w.lengths, sms) > 0   # some sequences are cut
    rows = [tables[i].tolist() for i in range(w.batch)]
    sub = Subset(kc, vc, rows)   # before any kernel of ours runs
    out = P.attn_decode(q.to(dev), kc, vc, tables.to(dev), lens.to(dev), w.scale)
    torch.cuda.synchronize()
    del kc, vc
    want = sub.attend(q, [sub.table(r) for r in rows], w.lengths, w.scale, w.dtype)
    assert_close(out, want, what=w.name)


def test_full_size_window_every_sequence():
    """The GQA 32/8 workload (256 sequences of 512-4096 tokens) with a
    1,024-token window, launched as the bench's window block launches it:
    every sequence against the oracle (sequences shorter than the window see
    all their keys; the others start mid-block)."""
    w = W.gqa_decode()
    window = 1024
    dev = "cuda"
    kc = W.normal_device(w.seed * 10 + 1, (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim), w.sigma,
                         w.dtype, dev)
    vc = W.normal_device(w.seed * 10 + 2, kc.shape, w.sigma, w.dtype, dev)
    g = W.generator(w.seed)
    q = W.normal(g, (w.batch, w.num_q_heads, w.head_dim), w.sigma, w.dtype)
    tables, _ = W.scattered_tables(g, w.lengths, w.block_size, w.num_blocks)
    lens = torch.tensor(w.lengths, dtype=torch.int32)
    assert min(w.lengths) < window < max(w.lengths)
    rows = [tables[i].tolist() for i in range(w.batch)]
    sub = Subset(kc, vc, rows)   # before any kernel of ours runs
    out = P.attn_decode(q.to(dev), kc, vc, tables.to(dev), lens.to(dev), w.scale, window=window)
    torch.cuda.synchronize()
    del kc, vc
    want = sub.attend(q, [sub.table(r) for r in rows], w.lengths, w.scale, w.dtype, window=window)
    assert_close(out, want, what=f"{w.name} window {window}")


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 4096])
@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [(32, 8, 128, 16, "f16"), (12, 12, 64, 32, "bf16")])
def test_sliding_window_decode(window, hq, hkv, d, bs, dtype):
    lens = [1, 15, 16, 17, 0, 33, 300, 1000, 2500]
    case = decode_case(60 + window, lens, hq, hkv, d, bs, dtype, sigma=1.0 if dtype == "f16" else 0.5)
    c = case.to("cuda")
    got = P.attn_decode(c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, window=window)
    torch.cuda.synchronize()
    want = oracle_window(case, window)
    assert_close(got, want, what=f"window {window}")


def oracle_window(case, window):
    import oracle
    return oracle.paged_attention(case.q, case.k_cache, case.v_cache, case.dtype, case.tables.numpy(),
                                  case.lens.numpy(), case.scale, window=window)


def test_sliding_window_long_sequence_split():
    case = decode_case(70, [40000, 7, 9000], 32, 8, 128, 16, "bf16", sigma=0.5)
    c = case.to("cuda")
    got = P.attn_decode(c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale, window=4097)
    torch.cuda.synchronize()
    assert_close(got, oracle_window(case, 4097), what="window 4097")


def test_decode_sees_inputs_rewritten_by_another_kernel_just_before_it():
    """Every kernel of the library is a programmatic dependent of the work before
    it on the stream and waits for that grid before reading: tables, lengths,
    queries and a cache row rewritten by another library's kernels immediately
    before the call are seen -- eagerly and inside a captured graph."""
    import dataclasses
    case = decode_case(71, [300, 17, 1000, 64], 32, 8, 128, 16)
    # the last token of sequence 2 gets new K/V values (written by a torch kernel)
    g = W.generator(72)
    k_new = W.normal(g, (8, 128), 1.0, "f16")
    v_new = W.normal(g, (8, 128), 1.0, "f16")
    L = int(case.lens[2])
    phys, off = int(case.tables[2, (L - 1) // 16]), (L - 1) % 16
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    kc[phys, off] = k_new
    vc[phys, off] = v_new
    want = dataclasses.replace(case, k_cache=kc, v_cache=vc).oracle()

    c = case.to("cuda")
    src = dict(tables=c.tables.clone(), lens=c.lens.clone(), q=c.q.clone(), k=k_new.cuda(), v=v_new.cuda())
    dst = dict(tables=torch.zeros_like(c.tables), lens=torch.ones_like(c.lens), q=torch.zeros_like(c.q))
    out = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(P.decode_workspace_size(4, 32, 8, 128), dtype=torch.uint8, device="cuda")

    def step():
        # elementwise kernels (not copies) write every input of the call
        for name in ("tables", "lens", "q"):
            torch.mul(src[name], 1, out=dst[name])
        torch.mul(src["k"], 1, out=c.k_cache[phys, off])
        torch.mul(src["v"], 1, out=c.v_cache[phys, off])
        P.attn_decode(dst["q"], c.k_cache, c.v_cache, dst["tables"], dst["lens"], c.scale, out=out, workspace=ws)

    def scramble():
        for t in dst.values():
            t.zero_()
        c.k_cache[phys, off].zero_()
        c.v_cache[phys, off].zero_()

    for _ in range(3):
        scramble()
        step()
        torch.cuda.synchronize()
        assert_close(out, want, what="eager")
    graph = P.StepGraph(step)
    for _ in range(3):
        scramble()
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_close(out, want, what="graph")
