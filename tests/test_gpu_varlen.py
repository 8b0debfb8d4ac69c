"""Packed varlen prefill + decode on the GPU against the binary64 oracle."""
import numpy as np
import pytest
import torch

import pagedattention_decode_gb300 as P
import workloads as W
from tests.cases import assert_close, varlen_case

pytestmark = pytest.mark.gpu


def run(case, causal=True, out_dtype=torch.float32, err=None):
    c = case.to("cuda")
    ql = (case.cu_q[1:] - case.cu_q[:-1])
    out = P.attn_varlen(c.q, c.k_cache, c.v_cache, c.tables, c.cu_q, c.lens, int(ql.max()), c.scale,
                        causal=causal, out_dtype=out_dtype, err=err)
    torch.cuda.synchronize()
    return out


SHAPES = [(32, 8, 128, 16, "f16"), (32, 8, 128, 32, "bf16"), (12, 12, 64, 16, "f16"), (16, 2, 128, 16, "bf16"),
          (4, 2, 64, 32, "f16")]


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_mixed_prefill_and_decode(hq, hkv, d, bs, dtype, causal):
    # chunks of several tiles with ragged tails, a chunk equal to its context,
    # decode rows, an empty row set and a q_len 2 chunk
    q_lens = [77, 1, 300, 1, 0, 2, 40, 1]
    kv_lens = [77 + 200, 50, 300, 1, 5, 2, 40 + 1000, 700]
    case = varlen_case(31 + hq + bs, q_lens, kv_lens, hq, hkv, d, bs, dtype,
                       sigma=1.0 if dtype == "f16" else 0.5)
    assert_close(run(case, causal), case.oracle(causal), what=f"varlen {hq}/{hkv}/{d}/{bs}/{dtype}/{causal}")


def test_decode_rows_equal_decode_kernel():
    """A q_len = 1 row sees every key (page 4's decode-mask bug made it see only the first)."""
    q_lens = [1, 1, 1]
    kv_lens = [37, 900, 16]
    case = varlen_case(41, q_lens, kv_lens, 32, 8, 128, 16)
    got = run(case)
    c = case.to("cuda")
    dec = P.attn_decode(c.q, c.k_cache, c.v_cache, c.tables, c.lens, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(got, dec)
    assert_close(got, case.oracle())


def test_square_chunk_is_plain_causal():
    case = varlen_case(42, [513], [513], 32, 8, 128, 16)
    assert_close(run(case), case.oracle())


def test_16bit_output_varlen():
    case = varlen_case(43, [129, 1, 64], [1000, 77, 64], 32, 8, 128, 16, "bf16", sigma=0.5)
    got = run(case, out_dtype=torch.bfloat16)
    assert_close(got, case.oracle())


@pytest.mark.parametrize("q_lens", [[0, 0, 0], []])
def test_no_query_rows_is_a_no_op(q_lens):
    """total_q = 0 (every sequence's row set empty) or no sequences at all:
    the call succeeds, returns an empty output and flags nothing."""
    kv_lens = [5, 0, 70][:len(q_lens)]
    if q_lens:
        case = varlen_case(46, q_lens, kv_lens, 8, 2, 64, 16)
        c = case.to("cuda")
        q, kc, vc, tab, cu, lens = c.q, c.k_cache, c.v_cache, c.tables, c.cu_q, c.lens
    else:
        kc = torch.zeros((4, 16, 2, 64), dtype=torch.float16, device="cuda")
        vc = torch.zeros_like(kc)
        q = torch.empty((0, 8, 64), dtype=torch.float16, device="cuda")
        tab = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
        cu = torch.zeros(1, dtype=torch.int32, device="cuda")
        lens = torch.zeros(0, dtype=torch.int32, device="cuda")
    assert q.shape[0] == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.attn_varlen(q, kc, vc, tab, cu, lens, 0, 0.125, err=err)
    torch.cuda.synchronize()
    assert out.shape == (0, 8, 64)
    assert int(err.item()) == 0


def test_q_len_beyond_kv_len_is_flagged():
    case = varlen_case(44, [40, 1], [30, 20], 8, 2, 64, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run(case, err=err)
    assert int(err.item()) & P.DEVERR["length"]


@pytest.mark.parametrize("window", [1, 33, 64, 200])
@pytest.mark.parametrize("causal", [True, False])
def test_sliding_window_varlen(window, causal):
    import oracle
    q_lens = [77, 1, 300, 1, 2, 130]
    kv_lens = [77 + 200, 50, 300, 1, 2, 1000]
    case = varlen_case(80 + window, q_lens, kv_lens, 32, 8, 128, 16)
    c = case.to("cuda")
    out = P.attn_varlen(c.q, c.k_cache, c.v_cache, c.tables, c.cu_q, c.lens, max(q_lens), c.scale, causal=causal,
                        window=window)
    torch.cuda.synchronize()
    want = oracle.paged_attention(case.q, case.k_cache, case.v_cache, case.dtype, case.tables.numpy(),
                                  case.lens.numpy(), case.scale, cu_q=case.cu_q.numpy(), causal=causal, window=window)
    assert_close(out, want, what=f"varlen window {window} causal {causal}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("q_sigma", [2.0, 4.0])
def test_peaked_attention_prefill(dtype, q_sigma):
    """Large query magnitudes concentrate each row's softmax on a few keys, where
    the rounding of P to a 16-bit operand of the P V MMA weighs most: the 2e-3
    gate must still hold (fp16 P keeps 11 significant bits, bf16 a hi + lo pair)."""
    import dataclasses
    q_lens = [300, 1, 129]
    kv_lens = [300 + 700, 900, 129]
    case = varlen_case(90 + int(q_sigma), q_lens, kv_lens, 32, 8, 128, 16, dtype)
    g = W.generator(95 + int(q_sigma))
    case = dataclasses.replace(case, q=W.normal(g, tuple(case.q.shape), q_sigma, dtype))
    for causal in (True, False):
        assert_close(run(case, causal), case.oracle(causal), what=f"peaked {dtype} q_sigma {q_sigma} causal {causal}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("factor", [4.0, 8.0])
def test_scores_jump_after_the_first_tiles(dtype, factor):
    """The keys of the later half of every context are scaled up, so a row's
    top scores rise by ~13 (factor 4) or ~30 (factor 8) log2 units after its
    first tiles.  The prefill kernel takes its running max from a row's first
    tile with a visible key: with factor 4 most rows keep that max and carry p
    of up to ~2^13 as 16-bit operands; with factor 8 a step's p would pass
    2^15, so the row moves its max, rescales O and its sum, and writes P
    again."""
    import dataclasses
    q_lens = [300, 1, 129, 520]
    kv_lens = [300 + 700, 900, 129 + 300, 520]
    bs = 16
    case = varlen_case(130 + int(factor), q_lens, kv_lens, 32, 8, 128, bs, dtype)
    k = case.k_cache.clone()
    for s, L in enumerate(kv_lens):
        nblk = W.blocks_for(L, bs)
        for j in range(nblk // 2, nblk):
            phys = int(case.tables[s, j])
            k[phys] = (k[phys].float() * factor).to(k.dtype)
    case = dataclasses.replace(case, k_cache=k)
    for causal in (True, False):
        assert_close(run(case, causal), case.oracle(causal), what=f"jump x{factor} {dtype} causal {causal}")


def _spread_lens(n, chunks, seed):
    """q_len / kv_len of n sequences: prefill chunks at the given indices,
    decode rows and empty row sets elsewhere."""
    g = np.random.default_rng(seed)
    q_lens, kv_lens = [], []
    for i in range(n):
        if i in chunks:
            q = chunks[i]
            q_lens.append(q)
            kv_lens.append(q + int(g.integers(0, 300)))
        elif i % 7 == 3:
            q_lens.append(0)
            kv_lens.append(int(g.integers(1, 200)))
        else:
            q_lens.append(1)
            kv_lens.append(int(g.integers(1, 200)))
    return q_lens, kv_lens


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_chunks_spread_over_many_sequences(causal):
    """The prefill kernel is persistent: each CTA walks work items (pairs of q
    tiles x KV heads) found by scanning cu_seqlens_q 32 sequences at a time.
    Chunks at indices past 32 and 64, between decode rows and empty row sets,
    with more items (20 pairs x 8 KV heads) than SMs, so some CTAs take two."""
    chunks = {3: 130, 37: 65, 38: 2, 64: 200, 70: 300, 99: 257}
    q_lens, kv_lens = _spread_lens(100, chunks, 5)
    case = varlen_case(150, q_lens, kv_lens, 32, 8, 128, 16)
    assert_close(run(case, causal), case.oracle(causal), what=f"spread causal {causal}")


def test_bad_sequence_is_flagged_and_others_still_right():
    """A chunk with q_len > kv_len (index 50) is flagged and skipped; every
    other sequence's rows still match the oracle."""
    chunks = {2: 70, 50: 40, 80: 129}
    q_lens, kv_lens = _spread_lens(90, chunks, 6)
    kv_lens[50] = 20
    case = varlen_case(151, q_lens, kv_lens, 32, 8, 128, 16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run(case, err=err)
    assert int(err.item()) & P.DEVERR["length"]
    # expected rows from the oracle on a copy whose sequence 50 is made valid
    # (it reads sequence 2's blocks); no other row depends on it
    import dataclasses
    tables, lens = case.tables.clone(), case.lens.clone()
    tables[50] = tables[2]
    lens[50] = 40
    want = dataclasses.replace(case, tables=tables, lens=lens).oracle(True)
    cu = case.cu_q.tolist()
    rows = [r for s in range(90) if s != 50 for r in range(cu[s], cu[s + 1])]
    assert_close(got[rows], want[rows], what="rows of the good sequences")


@pytest.mark.parametrize("bs", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_large_blocks_use_tall_tma_boxes(bs, dtype):
    """The prefill kernel loads K/V with the tallest TMA box (16, 32, 64 or 128
    rows) that divides block_size; blocks of 64-256 tokens take the 64- and
    128-row boxes, with ragged sequence tails inside a box."""
    q_lens = [300, 1, 77, 129]
    kv_lens = [300 + 500, 700, 77, 129 + 64]
    case = varlen_case(110 + bs, q_lens, kv_lens, 32, 8, 128, bs, dtype, sigma=1.0 if dtype == "f16" else 0.5)
    for causal in (True, False):
        assert_close(run(case, causal), case.oracle(causal), what=f"bs {bs} {dtype} causal {causal}")
