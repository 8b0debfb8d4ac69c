"""A multi-layer decode step captured as one CUDA graph replays to the same
bits as the eager calls (the graph only removes the per-call host work), and
its outputs and pools match the binary64 oracle's write-then-attend on host
copies of the pools."""
import numpy as np
import pytest
import torch

import oracle

import pagedattention_decode_gb300 as P
import workloads as W
from tests.cases import assert_close, decode_case

pytestmark = pytest.mark.gpu


def test_captured_multi_layer_step_matches_eager():
    layers = 3
    host = [decode_case(300 + l, [37, 700, 1, 64, 2000], 32, 8, 128, 16, "f16", poison=False)
            for l in range(layers)]
    cases = [h.to("cuda") for h in host]
    g = W.generator(310)
    B = 5
    k_new = W.normal(g, (B, 8, 128), 1.0, "f16").cuda()
    v_new = W.normal(g, (B, 8, 128), 1.0, "f16").cuda()
    c0 = cases[0]
    lens = c0.lens.clone()
    slots = torch.tensor([int(c0.tables[i, (int(L) - 1) // 16]) * 16 + (int(L) - 1) % 16 for i, L in
                          enumerate(lens.tolist())], dtype=torch.int64, device="cuda")
    ws = torch.empty(P.decode_workspace_size(B, 32, 8, 128), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((B, 32, 128), dtype=torch.float32, device="cuda") for _ in range(layers)]
    kc0 = [c.k_cache.clone() for c in cases]
    vc0 = [c.v_cache.clone() for c in cases]

    def step():
        for l, c in enumerate(cases):
            P.write_kv(k_new, v_new, slots, c.k_cache, c.v_cache)
            P.attn_decode(c.q, c.k_cache, c.v_cache, c0.tables, c0.lens, c.scale, out=outs[l], workspace=ws)

    # eager reference from the original pools
    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for l, c in enumerate(cases):
        c.k_cache.copy_(kc0[l])
        c.v_cache.copy_(vc0[l])
    graph = P.StepGraph(step)
    for o in outs:
        o.zero_()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, eager):
            assert torch.equal(a, b)
    # the oracle: each layer's pools written on the host, then attended
    slots_h = slots.cpu().tolist()
    for l, h in enumerate(host):
        ok = h.k_cache.view(torch.int16).numpy().view(np.uint16).copy()
        ov = h.v_cache.view(torch.int16).numpy().view(np.uint16).copy()
        oracle.write_kv(k_new.cpu(), v_new.cpu(), slots_h, ok, ov)
        assert np.array_equal(cases[l].k_cache.cpu().view(torch.int16).numpy().view(np.uint16), ok)
        assert np.array_equal(cases[l].v_cache.cpu().view(torch.int16).numpy().view(np.uint16), ov)
        want = oracle.paged_attention(h.q, ok, ov, "f16", host[0].tables.numpy(), host[0].lens.numpy(), h.scale)
        assert_close(outs[l], want, what=f"graph replay, layer {l}")
