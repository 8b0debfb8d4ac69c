"""Builders of paged-attention test cases shared by the GPU parity tests.

Inputs come from ``workloads`` (seeded, CPU); expected values from ``oracle``
(binary64).  Nothing here is computed by the CUDA path.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

import oracle
import workloads as W

TOL = 2e-3  # max-abs error on attention outputs (fp16/bf16 K/V, fp32 accumulate)


@dataclasses.dataclass
class PagedCase:
    q: torch.Tensor           # [rows, Hq, D] CPU
    k_cache: torch.Tensor     # [nb, bs, Hkv, D] CPU
    v_cache: torch.Tensor
    tables: torch.Tensor      # [B, max_blocks] int32 CPU
    lens: torch.Tensor        # [B] int32 CPU
    scale: float
    dtype: str
    cu_q: Optional[torch.Tensor] = None

    def to(self, device):
        return dataclasses.replace(
            self, q=self.q.to(device), k_cache=self.k_cache.to(device), v_cache=self.v_cache.to(device),
            tables=self.tables.to(device), lens=self.lens.to(device),
            cu_q=None if self.cu_q is None else self.cu_q.to(device))

    def oracle(self, causal: bool = True) -> np.ndarray:
        return oracle.paged_attention(self.q, self.k_cache, self.v_cache, self.dtype, self.tables.numpy(),
                                      self.lens.numpy(), self.scale,
                                      cu_q=None if self.cu_q is None else self.cu_q.numpy(), causal=causal)


def poison_unused(k_cache: torch.Tensor, v_cache: torch.Tensor, tables: torch.Tensor, lens: List[int]) -> None:
    """NaN into every slot no sequence holds (tails of last blocks, unused blocks)."""
    nb, bs = k_cache.shape[:2]
    used = torch.zeros(nb, bs, dtype=torch.bool)
    for i, L in enumerate(lens):
        for j in range(W.blocks_for(L, bs)):
            n = min(bs, L - j * bs)
            used[int(tables[i, j]), :n] = True
    k_cache[~used] = float("nan")
    v_cache[~used] = float("nan")


def decode_case(seed: int, lens: List[int], hq: int, hkv: int, d: int, bs: int, dtype: str = "f16",
                sigma: float = 1.0, num_blocks: Optional[int] = None, poison: bool = True,
                scale: Optional[float] = None, extra_table_cols: int = 1) -> PagedCase:
    g = W.generator(seed)
    need = sum(W.blocks_for(L, bs) for L in lens)
    nb = num_blocks or max(4, int(math.ceil(1.25 * need)) + 3)
    kc = W.normal(g, (nb, bs, hkv, d), sigma, dtype)
    vc = W.normal(g, (nb, bs, hkv, d), sigma, dtype)
    q = W.normal(g, (len(lens), hq, d), sigma, dtype)
    mb = max([W.blocks_for(L, bs) for L in lens] + [1]) + extra_table_cols
    tables, _ = W.scattered_tables(g, lens, bs, nb, max_blocks=mb)
    if poison:
        poison_unused(kc, vc, tables, lens)
    return PagedCase(q, kc, vc, tables, torch.tensor(lens, dtype=torch.int32),
                     scale if scale is not None else 1.0 / math.sqrt(d), dtype)


def varlen_case(seed: int, q_lens: List[int], kv_lens: List[int], hq: int, hkv: int, d: int, bs: int,
                dtype: str = "f16", sigma: float = 1.0) -> PagedCase:
    c = decode_case(seed, kv_lens, hq, hkv, d, bs, dtype, sigma)
    g = W.generator(seed + 7)
    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + n)
    q = W.normal(g, (cu[-1], hq, d), sigma, dtype)
    return dataclasses.replace(c, q=q, cu_q=torch.tensor(cu, dtype=torch.int32))


def assert_close(got: torch.Tensor, want: np.ndarray, tol: float = TOL, what: str = "") -> float:
    """max-abs check; 16-bit outputs get half an ulp of the rounded oracle on top."""
    g = got.detach().float().cpu().double().numpy()
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    bound = np.full_like(w, tol)
    if got.dtype in (torch.float16, torch.bfloat16):
        rounded = torch.from_numpy(w).to(got.dtype).double().numpy()
        if got.dtype == torch.float16:
            ulp = np.spacing(np.abs(rounded).astype(np.float16)).astype(np.float64)
        else:  # bfloat16: 8 significant bits
            mag = np.maximum(np.abs(rounded), 2.0 ** -126)
            ulp = np.exp2(np.floor(np.log2(mag)) - 7)
        bound = bound + 0.5 * ulp
        w = rounded
    err = np.abs(g - w)
    worst = float(err.max()) if err.size else 0.0
    assert (err <= bound).all(), f"{what}: max abs err {worst:.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Subset:
    """Host copy of the blocks a set of sequences use, with ids renumbered; the
    oracle replays writes and copies on it and attends over it."""

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

    def attend(self, q_rows, table_rows, lens, scale, dtype, cu_q=None, window=0):
        """Binary64 attention over the host copy: one row per sequence, or
        packed causal rows when cu_q is given; window > 0 keeps each row's most
        recent ``window`` keys."""
        mb = max(len(t) for t in table_rows)
        tab = np.full((len(table_rows), mb), -1, dtype=np.int32)
        for i, t in enumerate(table_rows):
            tab[i, :len(t)] = t
        return oracle.paged_attention(q_rows, self.k, self.v, dtype, tab, np.array(lens, dtype=np.int32), scale,
                                      cu_q=cu_q, causal=cu_q is not None, window=window)
