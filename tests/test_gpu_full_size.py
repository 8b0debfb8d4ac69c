"""Full-size workloads, launched as the bench launches them, every output row
checked against the oracle.

* the mixed packed step (2048-token shared prefix, 16 prefill chunks of 512
  rows, 240 decode rows, block_size 32) and its width-4 beam split with
  copy-on-write -- built by the bench's own MixedStep;
* the GPT-2-shaped 12-layer decode step (one pool per layer, one shared table,
  write then attend in every layer).

The oracle's copy of the blocks the step's sequences use is taken from the device
before any kernel of this project runs, and the step's writes and copies are
replayed on it by the oracle itself.
"""
import pytest
import torch

import pagedattention_decode_gb300 as P
import workloads as W
from tests.cases import Subset, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_mixed_step_full_size_every_row(dtype):
    """Every output row of both steps: the 16 x 512 prefill rows and 240
    decode rows of the packed step, then all 128 beams after the split (bf16:
    the same step over a bf16 cache, P entering P V as a hi + lo pair)."""
    import bench
    dev = torch.device("cuda", torch.cuda.current_device())
    m = bench.MixedStep(dev, dtype)
    s1, s2 = m.s1, m.s2
    tab1, tab2 = s1["tables"].cpu(), s2["tables"].cpu()
    rows1 = [tab1[i].tolist() for i in range(tab1.shape[0])]
    rows2 = [tab2[i].tolist() for i in range(tab2.shape[0])]
    sub = Subset(m.k_cache, m.v_cache, rows1 + rows2)   # before any of our kernels ran
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

    # oracle replay of step 1: the writes, then the whole packed call (causal rows)
    sub.write(slots1, k1, v1)
    cu = s1["cu"].cpu().numpy()
    want1 = sub.attend(s1["q"].cpu(), [sub.table(r) for r in rows1], m.s1_lens_host, m.scale, dtype, cu_q=cu)
    n_pf = m.nchunk * m.chunk
    assert_close(out1[:n_pf], want1[:n_pf], what=f"step 1 prefill rows ({dtype})")
    assert_close(out1[n_pf:], want1[n_pf:], what=f"step 1 decode rows ({dtype})")
    # oracle replay of step 2: copies, writes, decode of every beam
    sub.copy(pairs2)
    sub.write(slots2, k2, v2)
    want2 = sub.attend(s2["q"].cpu(), [sub.table(r) for r in rows2], m.s2_lens_host, m.scale, dtype)
    assert_close(out2, want2, what=f"step 2 beams ({dtype})")


def test_mixed_step_full_size_window_every_row():
    """Step 1 of the mixed workload with a 1,024-key sliding window: the
    prefill chunks skip the tiles before each row's window and mask inside
    the first tile they read; every row against the oracle."""
    import bench
    dev = torch.device("cuda", torch.cuda.current_device())
    m = bench.MixedStep(dev)
    s1 = m.s1
    tab1 = s1["tables"].cpu()
    rows1 = [tab1[i].tolist() for i in range(tab1.shape[0])]
    sub = Subset(m.k_cache, m.v_cache, rows1)   # before any of our kernels ran
    k1, v1, slots1 = s1["k"].cpu(), s1["v"].cpu(), s1["slots"].cpu().tolist()
    window = 1024
    P.write_kv(s1["k"], s1["v"], s1["slots"], m.k_cache, m.v_cache, err=m.err)
    out = P.attn_varlen(s1["q"], m.k_cache, m.v_cache, s1["tables"], s1["cu"], s1["lens"], s1["max_q"], m.scale,
                        workspace=m.ws, err=m.err, window=window)
    torch.cuda.synchronize()
    assert int(m.err.item()) == 0
    sub.write(slots1, k1, v1)
    cu = s1["cu"].cpu().numpy()
    want = sub.attend(s1["q"].cpu(), [sub.table(r) for r in rows1], m.s1_lens_host, m.scale, "f16", cu_q=cu,
                      window=window)
    n_pf = m.nchunk * m.chunk
    assert_close(out[:n_pf], want[:n_pf], what="window prefill rows")
    assert_close(out[n_pf:], want[n_pf:], what="window decode rows")


def test_gpt2_shaped_twelve_layers_every_sequence():
    w = W.gpt2_decode()
    dev = "cuda"
    g = W.generator(w.seed)
    tables, _ = W.scattered_tables(g, [L + 1 for L in w.lengths], w.block_size, w.num_blocks)
    lens = torch.tensor([L + 1 for L in w.lengths], dtype=torch.int32)
    slots = [int(tables[i, L // w.block_size]) * w.block_size + L % w.block_size for i, L in enumerate(w.lengths)]
    rows = [tables[i].tolist() for i in range(w.batch)]
    dtables, dlens = tables.to(dev), lens.to(dev)
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
        want = sub.attend(q, [sub.table(r) for r in rows], lens.tolist(), w.scale, "f16")
        assert_close(out, want, what=f"layer {layer}")
        del kc, vc
