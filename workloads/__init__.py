"""Seeded synthetic inputs for the paged KV cache attention path.

This module is shared by the CPU oracle (``oracle/``), the CUDA path's tests
and ``bench.py``.  It only draws numbers and lays them out as inputs: it holds
none of the attention, softmax, slot or allocator arithmetic.

Recipe (the shapes follow the synthetic workloads built from the paged-attention
pages; "How to Implement Paged Attention in PyTorch and vLLM", section "Size the
paged KV cache and choose a block size", gives the pool layout and 16-token
blocks):

* one ``torch.Generator`` seeded with an integer per workload;
* lengths drawn with ``torch.randint(lo, hi + 1)``;
* values drawn as fp32 normals with a given sigma and rounded once,
  round-to-nearest-even, to fp16 or bf16;
* block tables drawn by taking a seeded permutation of all pool ids and
  handing each sequence the next ids of that permutation ("scattered"
  placement); unused table entries are ``-1``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform_lengths(g: torch.Generator, n: int, lo: int, hi: int) -> List[int]:
    """``n`` integers uniform on the closed range [lo, hi]."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def normal(g: torch.Generator, shape: Sequence[int], sigma: float, dtype: str) -> torch.Tensor:
    """fp32 N(0, sigma^2) rounded once (RNE) to ``dtype`` ("f16" or "bf16"), CPU."""
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(DTYPES[dtype])


def normal_device(seed: int, shape: Sequence[int], sigma: float, dtype: str,
                  device: str = "cuda", chunk: int = 1 << 26) -> torch.Tensor:
    """Like :func:`normal` but drawn on ``device`` in chunks (for multi-GB pools).

    The values depend on the seed and the device generator; they are inputs
    only, drawn by torch, never by this project's kernels.
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(tuple(shape), dtype=DTYPES[dtype], device=device)
    flat = out.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        t = torch.randn(n, generator=g, dtype=torch.float32, device=device)
        if sigma != 1.0:
            t.mul_(sigma)
        flat[i:i + n].copy_(t)
    return out


def permutation(g: torch.Generator, n: int) -> List[int]:
    return [int(x) for x in torch.randperm(n, generator=g)]


def blocks_for(length: int, block_size: int) -> int:
    """How many whole blocks hold ``length`` tokens (sizing the inputs only)."""
    return -(-int(length) // int(block_size))


def scattered_tables(g: torch.Generator, lengths: Sequence[int], block_size: int,
                     num_blocks: int, max_blocks: Optional[int] = None):
    """Hand each sequence the next ids of a seeded permutation of the pool.

    Returns ``(tables, order)``: ``tables`` is an int32 ``[B, max_blocks]``
    tensor, -1 where a sequence holds no block; ``order`` is the permutation.
    """
    need = [blocks_for(L, block_size) for L in lengths]
    if sum(need) > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {sum(need)}")
    mb = max(need + [1]) if max_blocks is None else max_blocks
    order = permutation(g, num_blocks)
    tables = torch.full((len(lengths), mb), -1, dtype=torch.int32)
    pos = 0
    for i, n in enumerate(need):
        if n:
            tables[i, :n] = torch.tensor(order[pos:pos + n], dtype=torch.int32)
        pos += n
    return tables, order


# ---------------------------------------------------------------------------
# The five synthetic workloads, restated with their sizes.
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    sigma: float
    lengths: List[int]
    num_blocks: int
    scale: float

    @property
    def batch(self) -> int:
        return len(self.lengths)


def tiny_decode() -> Workload:
    """1 layer, 12/12 heads, D 64, bs 16, fp16 N(0,1), 64-block pool, L = 40/20/16/30."""
    return Workload("tiny_decode_mha12_d64_bs16", 1, 1, 12, 12, 64, 16, "f16", 1.0,
                    [40, 20, 16, 30], 64, 1.0 / math.sqrt(64))


def gpt2_decode() -> Workload:
    """12 layers, 12/12 heads, D 64, bs 16, fp16, 8192 blocks/layer, B 32, L ~ U[64,1024]."""
    g = generator(2)
    lens = uniform_lengths(g, 32, 64, 1024)
    return Workload("gpt2s_decode_b32_l64_1024", 2, 12, 12, 12, 64, 16, "f16", 1.0,
                    lens, 8192, 1.0 / math.sqrt(64))


def gqa_decode() -> Workload:
    """GQA 32/8, D 128, bs 16, fp16, B 256, L ~ U[512,4096], pool = 1.1 x needed."""
    g = generator(3)
    lens = uniform_lengths(g, 256, 512, 4096)
    need = sum(blocks_for(L, 16) for L in lens)
    return Workload("gqa32_8_d128_bs16_b256_l512_4096", 3, 1, 32, 8, 128, 16, "f16", 1.0,
                    lens, int(math.ceil(1.1 * need)), 1.0 / math.sqrt(128))


def long_skewed_decode() -> Workload:
    """GQA 32/8, D 128, bs 16, bf16 N(0,0.5), B 8, L = 1024 * 2^k for k = 0..7."""
    lens = [1024 << k for k in range(8)]
    need = sum(blocks_for(L, 16) for L in lens)
    return Workload("gqa32_8_d128_bs16_bf16_skew_1k_128k", 4, 1, 32, 8, 128, 16, "bf16", 0.5,
                    lens, int(math.ceil(1.1 * need)), 1.0 / math.sqrt(128))


def first_sequences(w: Workload, n: int) -> Workload:
    """The same workload cut to its first n sequences, pool resized to 1.1x."""
    lens = list(w.lengths[:n])
    need = sum(blocks_for(L, w.block_size) for L in lens)
    return dataclasses.replace(w, name=f"{w.name}_first{n}", lengths=lens,
                               num_blocks=max(1, int(math.ceil(1.1 * need))))


def mixed_step_decode_lengths() -> List[int]:
    """Total contexts of the 240 decode sequences of the mixed step, U[256, 8192]."""
    g = generator(5)
    return uniform_lengths(g, 240, 256, 8192)


ALL = {
    1: tiny_decode,
    2: gpt2_decode,
    3: gqa_decode,
    4: long_skewed_decode,
}
