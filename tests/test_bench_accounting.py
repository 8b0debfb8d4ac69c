"""The bench's byte accounting, pinned to the pages' memory arithmetic and to a
brute-force replay of the even split of sub-blocks over CTAs."""
import json
import os
import random

import bench
from tests.conftest import GOLDEN


def test_kv_bytes_match_page_memory_math():
    """'How to Implement Paged Attention in PyTorch and vLLM': 512 MB per
    sequence at 4096 tokens (32 layers, 8 KV heads, head_dim 128, FP16) and
    128 GB for 256 such sequences."""
    g = json.load(open(os.path.join(GOLDEN, "kv_memory_math.json")))
    per_tok = bench.kv_bytes_per_token(g["kv_heads"], g["head_dim"], g["dtype_bytes"], layers=g["layers"])
    assert per_tok * g["max_tokens"] == g["bytes_per_sequence"] == 512 * 2 ** 20
    assert per_tok * g["max_tokens"] * g["sequences"] == g["bytes_total"] == 128 * 2 ** 30


def test_split_records_brute_force():
    rng = random.Random(3)
    for _ in range(200):
        lens = [rng.choice([0, rng.randint(1, 40), rng.randint(1, 3000)]) for _ in range(rng.randint(1, 40))]
        ctas_max = rng.randint(1, 160)
        n = [-(-L // 16) for L in lens]
        total = sum(n)
        want = 0
        whole = len(lens) <= 32 and total <= 64 and len(lens) <= ctas_max  # a CTA per sequence
        if total and not whole:
            ctas = min(ctas_max, -(-total // 4))
            owner = []
            for c in range(ctas):
                lo, hi = c * total // ctas, (c + 1) * total // ctas
                owner += [c] * (hi - lo)
            assert len(owner) == total
            start = 0
            for k in n:
                cs = set(owner[start:start + k])
                if len(cs) > 1:
                    want += len(cs)
                start += k
        assert bench.split_records(lens, ctas_max) == want


def test_window_keeps_each_sequences_last_keys():
    """A window of w keys counts min(L, w) keys per sequence (all of them when
    there is no window), as the windowed decode attends them."""
    lens = [0, 1, 15, 1023, 1024, 1025, 4096]
    assert bench.windowed(lens, 0) == lens
    assert bench.windowed(lens, 1024) == [0, 1, 15, 1023, 1024, 1024, 1024]
    assert bench.windowed(lens, 1) == [0, 1, 1, 1, 1, 1, 1]
    # the windowed decode's bytes are those of a call over the kept lengths
    kept = bench.windowed(lens, 1024)
    assert bench.decode_bytes(kept, 32, 8, 128, 2, 4, 152) == bench.decode_bytes(
        [min(L, 1024) for L in lens], 32, 8, 128, 2, 4, 152)
    assert sum(kept) * bench.kv_bytes_per_token(8, 128, 2) < sum(lens) * bench.kv_bytes_per_token(8, 128, 2)
