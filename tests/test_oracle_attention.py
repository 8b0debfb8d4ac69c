"""Pins of the binary64 attention oracle (oracle/pkv_oracle.c).

Each test fixes the oracle to something other than itself: exact format
decoding checked against numpy/torch casts, closed forms, torch's own CPU
scaled_dot_product_attention (float64, enable_gqa for the head grouping,
is_causal for the square causal case), invariances the definition implies,
and high-precision brute force with Python's decimal module.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W


def build_pool(seqs_k, seqs_v, block_size, num_blocks, seed, dtype=torch.float16):
    """Place contiguous per-sequence K/V ([L, Hkv, D]) into a scattered pool.

    Block j of a sequence gets rows j*bs .. j*bs+bs-1 of its contiguous
    tensor (slicing, not the slot formula).  Unused slots are NaN poison and
    unused table entries are -1.
    """
    hkv, d = seqs_k[0].shape[1], seqs_k[0].shape[2]
    lens = [k.shape[0] for k in seqs_k]
    g = W.generator(seed)
    tables, _ = W.scattered_tables(g, lens, block_size, num_blocks)
    kc = torch.full((num_blocks, block_size, hkv, d), float("nan"), dtype=dtype)
    vc = kc.clone()
    for i, (k, v) in enumerate(zip(seqs_k, seqs_v)):
        for j in range(tables.shape[1]):
            phys = int(tables[i, j])
            if phys < 0:
                continue
            rows = k[j * block_size:(j + 1) * block_size]
            kc[phys, :rows.shape[0]] = rows
            vc[phys, :rows.shape[0]] = v[j * block_size:(j + 1) * block_size]
    return kc, vc, tables


def rand_case(seed, lens, hq, hkv, d, bs, nb, dtype="f16", sigma=1.0):
    g = W.generator(seed)
    ks = [W.normal(g, (L, hkv, d), sigma, dtype) for L in lens]
    vs = [W.normal(g, (L, hkv, d), sigma, dtype) for L in lens]
    q = W.normal(g, (len(lens), hq, d), sigma, dtype)
    kc, vc, tables = build_pool(ks, vs, bs, nb, seed + 1000, W.DTYPES[dtype])
    return q, ks, vs, kc, vc, tables


# ---------------------------------------------------------------------------
def test_decoders_exact_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    want16 = bits.view(np.float16).astype(np.float64)
    wantbf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for b in range(0, 65536, 1):
        got = oracle.decode_f16(int(b))
        w = want16[b]
        assert (math.isnan(got) and math.isnan(w)) or got == w, b
        got = oracle.decode_bf16(int(b))
        w = wantbf[b]
        assert (math.isnan(got) and math.isnan(w)) or got == w, b


def test_sdpa_equivalence_gqa():
    """Torch CPU SDPA (float64, enable_gqa) on the contiguous tensors."""
    lens = [40, 20, 16, 30, 1]
    hq, hkv, d, bs = 8, 2, 32, 16
    q, ks, vs, kc, vc, tables = rand_case(11, lens, hq, hkv, d, bs, 64)
    out = oracle.paged_attention(q, kc, vc, "f16", tables, lens, 1 / math.sqrt(d))
    for i, L in enumerate(lens):
        qq = q[i].double().unsqueeze(1)                 # [Hq, 1, D]
        kk = ks[i].double().permute(1, 0, 2)            # [Hkv, L, D]
        vv = vs[i].double().permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(qq.unsqueeze(0), kk.unsqueeze(0), vv.unsqueeze(0),
                                             scale=1 / math.sqrt(d), enable_gqa=True)[0, :, 0]
        np.testing.assert_allclose(out[i], ref.numpy(), rtol=0, atol=1e-12)


def test_sdpa_equivalence_bf16_mha():
    lens = [33, 7]
    q, ks, vs, kc, vc, tables = rand_case(12, lens, 4, 4, 16, 8, 16, dtype="bf16", sigma=0.5)
    out = oracle.paged_attention(q, kc, vc, "bf16", tables, lens, 0.3)
    for i in range(len(lens)):
        ref = F.scaled_dot_product_attention(q[i].double().unsqueeze(1).unsqueeze(0),
                                             ks[i].double().permute(1, 0, 2).unsqueeze(0),
                                             vs[i].double().permute(1, 0, 2).unsqueeze(0),
                                             scale=0.3)[0, :, 0]
        np.testing.assert_allclose(out[i], ref.numpy(), rtol=0, atol=1e-12)


def test_single_key_returns_v():
    q, ks, vs, kc, vc, tables = rand_case(13, [1, 1], 4, 2, 8, 4, 8)
    out = oracle.paged_attention(q, kc, vc, "f16", tables, [1, 1], 0.7)
    for i in range(2):
        want = vs[i][0].double().repeat_interleave(2, dim=0).numpy()
        assert np.array_equal(out[i], want)


def test_equal_keys_zero_query_zero_scale_give_mean_of_v():
    g = W.generator(14)
    L, hq, hkv, d = 37, 4, 4, 8
    k1 = W.normal(g, (1, hkv, d), 1.0, "f16").expand(L, hkv, d).contiguous()
    v = W.normal(g, (L, hkv, d), 1.0, "f16")
    q = W.normal(g, (1, hq, d), 1.0, "f16")
    kc, vc, tables = build_pool([k1], [v], 8, 8, 15)
    mean = v.double().mean(0).numpy()
    out = oracle.paged_attention(q, kc, vc, "f16", tables, [L], 0.5)
    np.testing.assert_allclose(out[0], mean, rtol=0, atol=1e-14)
    # zero query or zero scale with distinct keys: also the mean of V
    k = W.normal(g, (L, hkv, d), 1.0, "f16")
    kc, vc, tables = build_pool([k], [v], 8, 8, 16)
    out0 = oracle.paged_attention(torch.zeros_like(q), kc, vc, "f16", tables, [L], 0.5)
    np.testing.assert_allclose(out0[0], mean, rtol=0, atol=1e-14)
    out1 = oracle.paged_attention(q, kc, vc, "f16", tables, [L], 0.0)
    np.testing.assert_allclose(out1[0], mean, rtol=0, atol=1e-14)


def test_gqa_mapping_is_contiguous_groups():
    """Query head h reads KV head h // (Hq/Hkv) (page 2's unsqueeze/expand/reshape)."""
    hq, hkv, d, L = 12, 3, 4, 5
    g = W.generator(17)
    k = W.normal(g, (L, hkv, d), 1.0, "f16")
    v = torch.arange(hkv, dtype=torch.float16).view(1, hkv, 1).expand(L, hkv, d).contiguous()
    q = W.normal(g, (1, hq, d), 1.0, "f16")
    kc, vc, tables = build_pool([k], [v], 4, 4, 18)
    out = oracle.paged_attention(q, kc, vc, "f16", tables, [L], 1.0)
    for h in range(hq):
        assert np.all(out[0, h] == h // (hq // hkv)), h


def test_block_permutation_and_block_size_invariance():
    lens = [45, 3, 32]
    hq, hkv, d = 4, 2, 16
    g = W.generator(19)
    ks = [W.normal(g, (L, hkv, d), 1.0, "f16") for L in lens]
    vs = [W.normal(g, (L, hkv, d), 1.0, "f16") for L in lens]
    q = W.normal(g, (3, hq, d), 1.0, "f16")
    outs = []
    for bs, nb, seed in [(16, 12, 1), (16, 12, 2), (16, 40, 3), (4, 64, 4), (32, 8, 5), (1, 90, 6)]:
        kc, vc, tables = build_pool(ks, vs, bs, nb, seed)
        outs.append(oracle.paged_attention(q, kc, vc, "f16", tables, lens, 0.25))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_poison_in_unused_slots_is_never_read():
    lens = [21, 5]
    q, ks, vs, kc, vc, tables = rand_case(20, lens, 2, 2, 8, 16, 10)
    assert torch.isnan(kc).any()  # tails and unused blocks hold NaN
    out = oracle.paged_attention(q, kc, vc, "f16", tables, lens, 0.5)
    assert np.isfinite(out).all()


def test_empty_sequence_gives_zeros():
    lens = [0, 9]
    q, ks, vs, kc, vc, tables = rand_case(21, [1, 9], 2, 1, 8, 4, 8)
    out = oracle.paged_attention(q, kc, vc, "f16", tables, lens, 0.5)
    assert np.all(out[0] == 0.0) and np.isfinite(out[1]).all()


def test_causal_square_matches_sdpa_is_causal():
    """q_len == kv_len: the causal offset reduces to the usual causal mask."""
    L, hq, hkv, d = 19, 4, 2, 8
    g = W.generator(22)
    k = W.normal(g, (L, hkv, d), 1.0, "f16")
    v = W.normal(g, (L, hkv, d), 1.0, "f16")
    q = W.normal(g, (L, hq, d), 1.0, "f16")
    kc, vc, tables = build_pool([k], [v], 4, 8, 23)
    out = oracle.paged_attention(q, kc, vc, "f16", tables, [L], 0.4, cu_q=[0, L], causal=True)
    ref = F.scaled_dot_product_attention(q.double().permute(1, 0, 2).unsqueeze(0),
                                         k.double().permute(1, 0, 2).unsqueeze(0),
                                         v.double().permute(1, 0, 2).unsqueeze(0),
                                         scale=0.4, is_causal=True, enable_gqa=True)
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_causal_offset_rows_equal_truncated_decode():
    """Row i of a chunk of q_len rows over kv_len keys equals a one-row decode
    over the first kv_len - q_len + i + 1 keys; a q_len = 1 row sees every key
    (the decode-mask bug on page 4 made it see only the first)."""
    L, ql, hq, hkv, d = 23, 6, 4, 2, 8
    g = W.generator(24)
    k = W.normal(g, (L, hkv, d), 1.0, "f16")
    v = W.normal(g, (L, hkv, d), 1.0, "f16")
    q = W.normal(g, (ql, hq, d), 1.0, "f16")
    kc, vc, tables = build_pool([k], [v], 4, 8, 25)
    chunk = oracle.paged_attention(q, kc, vc, "f16", tables, [L], 0.4, cu_q=[0, ql], causal=True)
    for i in range(ql):
        vis = L - ql + i + 1
        one = oracle.paged_attention(q[i:i + 1], kc, vc, "f16", tables, [vis], 0.4)
        assert np.array_equal(chunk[i], one[0])
    last = oracle.paged_attention(q[-1:], kc, vc, "f16", tables, [L], 0.4, cu_q=[0, 1], causal=True)
    full = oracle.paged_attention(q[-1:], kc, vc, "f16", tables, [L], 0.4)
    assert np.array_equal(last, full)


def test_brute_force_decimal():
    """Integer-valued q/K/V (exact in fp16): 60-digit decimal softmax."""
    getcontext().prec = 60
    rng = np.random.default_rng(26)
    for trial in range(6):
        L, d, hq, hkv = int(rng.integers(1, 9)), int(rng.integers(1, 9)), 2, 1
        k = torch.tensor(rng.integers(-3, 4, (L, hkv, d)), dtype=torch.float16)
        v = torch.tensor(rng.integers(-3, 4, (L, hkv, d)), dtype=torch.float16)
        q = torch.tensor(rng.integers(-3, 4, (1, hq, d)), dtype=torch.float16)
        scale = 0.25
        kc, vc, tables = build_pool([k], [v], 4, 4, 27 + trial)
        out = oracle.paged_attention(q, kc, vc, "f16", tables, [L], scale)
        for h in range(hq):
            sc = [Decimal(int(sum(int(q[0, h, j]) * int(k[t, 0, j]) for j in range(d)))) * Decimal(scale)
                  for t in range(L)]
            m = max(sc)
            w = [(s - m).exp() for s in sc]
            z = sum(w)
            for j in range(d):
                want = sum(w[t] * Decimal(int(v[t, 0, j])) for t in range(L)) / z
                assert abs(out[0, h, j] - float(want)) <= 1e-13, (trial, h, j)


def test_rejects_bad_table_entry():
    q, ks, vs, kc, vc, tables = rand_case(28, [20], 2, 2, 8, 16, 4)
    bad = tables.clone()
    bad[0, 1] = 99
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kc, vc, "f16", bad, [20], 0.5)


def test_window_pins():
    """Sliding window ('How to Implement Paged Attention in PyTorch and vLLM',
    section 'PagedAttention vs sliding-window attention...'): a row attends only
    to the most recent w tokens, its own included."""
    lens = [45, 64, 7]
    bs = 16
    q, ks, vs, kc, vc, tables = rand_case(40, lens, 4, 2, 16, bs, 16)
    full = oracle.paged_attention(q, kc, vc, "f16", tables, lens, 0.3)
    # a window at least as long as the context changes nothing
    assert np.array_equal(oracle.paged_attention(q, kc, vc, "f16", tables, lens, 0.3, window=64), full)
    # window 1: the last key only
    one = oracle.paged_attention(q, kc, vc, "f16", tables, lens, 0.3, window=1)
    for i, L in enumerate(lens):
        assert np.array_equal(one[i], vs[i][L - 1].double().repeat_interleave(2, dim=0).numpy())
    # a window starting on a block boundary equals full attention over the
    # table shifted by whole blocks (a different path through the oracle)
    w = 29  # 45 - 29 = 16: the window starts at block 1 of sequence 0
    win = oracle.paged_attention(q[:1], kc, vc, "f16", tables[:1], lens[:1], 0.3, window=w)
    shifted = tables[:1, 1:].clone()
    alt = oracle.paged_attention(q[:1], kc, vc, "f16", shifted, [w], 0.3)
    assert np.array_equal(win, alt)
    # causal chunk rows with a window: row i equals a windowed one-row decode
    ql, L = 6, 45
    qq = W.normal(W.generator(41), (ql, 4, 16), 1.0, "f16")
    chunk = oracle.paged_attention(qq, kc, vc, "f16", tables[:1], [L], 0.3, cu_q=[0, ql], causal=True, window=10)
    for i in range(ql):
        one_row = oracle.paged_attention(qq[i:i + 1], kc, vc, "f16", tables[:1], [L - ql + i + 1], 0.3, window=10)
        assert np.array_equal(chunk[i], one_row[0])
