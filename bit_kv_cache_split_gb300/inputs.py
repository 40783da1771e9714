"""Seeded synthetic inputs for decode attention over a 2-/4-bit KV cache.

This module only draws random numbers in the documented layout; it holds none
of the method's arithmetic. The CUDA path, the tests and the benchmark all take
their inputs from here, so both sides of every parity check see identical
tensors.

Workload shapes follow the pages' setup (32 query heads, 8 KV heads,
head_dim 128, token-wise groups of 128; explainer "FOSCAR speeds up 2-bit KV
decode", measured-payoff paragraph) and the value distributions stated for
each workload below. Draw order within one seed: K codes, K scales, K offsets,
V codes, V scales, V offsets, Q, then the window's K and V.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Union

import numpy as np
import torch

TOKENWISE = 0
CHANNELWISE = 1
TOKEN_TILE = 128  # token capacity is rounded up to a multiple of this


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclasses.dataclass
class Workload:
    """One decode-attention problem: shapes, format and value distributions."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    seq_lens: Union[int, Sequence[int]]
    bits: int = 2
    k_layout: int = TOKENWISE
    v_layout: int = TOKENWISE
    group: int = 128
    head_dim: int = 128
    s_range: tuple = (0.01, 0.1)
    z_range: tuple = (-0.2, 0.2)
    q_std: float = 1.0
    window: int = 0  # bf16 tokens after the quantized ones (0: none)
    win_range: tuple = (-0.2, 0.5)
    sm_scale: float = 0.0  # 0 selects 1/sqrt(head_dim)
    seed: int = 0

    @property
    def lens(self) -> List[int]:
        if isinstance(self.seq_lens, int):
            return [self.seq_lens] * self.batch
        return [int(x) for x in self.seq_lens]

    @property
    def t_cap(self) -> int:
        return max(TOKEN_TILE, round_up(max(self.lens) if self.batch else 0, TOKEN_TILE))

    @property
    def hq_per_kv(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def sz_shape(self, layout: int):
        B, H, T, D, g = self.batch, self.num_kv_heads, self.t_cap, self.head_dim, self.group
        return (B, H, T, D // g) if layout == TOKENWISE else (B, H, T // g, D)

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["seq_lens"] = self.lens if len(set(self.lens)) > 1 else self.lens[0] if self.lens else 0
        d["t_cap"] = self.t_cap
        return d


def _uniform(shape, lo, hi, g, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def generate(wl: Workload, device: Union[str, torch.device] = "cpu") -> dict:
    """Draw every input tensor of `wl` on `device` with a generator seeded by wl.seed."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(wl.seed))
    B, Hq, Hkv, D, T = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.t_cap
    row = D * wl.bits // 8
    out = {}
    for side, layout in (("k", wl.k_layout), ("v", wl.v_layout)):
        out[f"{side}_codes"] = torch.randint(0, 256, (B, Hkv, T, row), generator=g, device=device, dtype=torch.uint8)
        out[f"{side}_scale"] = _uniform(wl.sz_shape(layout), *wl.s_range, g, device).to(torch.float16)
        out[f"{side}_off"] = _uniform(wl.sz_shape(layout), *wl.z_range, g, device).to(torch.float16)
    out["q"] = (torch.randn((B, Hq, D), generator=g, device=device, dtype=torch.float32) * wl.q_std).to(torch.bfloat16)
    out["seq_lens"] = torch.tensor(wl.lens, dtype=torch.int32, device=device)
    if wl.window:
        for side in ("k", "v"):
            out[f"{side}_win"] = _uniform((B, Hkv, wl.window, D), *wl.win_range, g, device).to(torch.bfloat16)
        out["win_lens"] = torch.full((B,), wl.window, dtype=torch.int32, device=device)
    return out


def generate_pack_source(batch: int, num_kv_heads: int, seq_lens, head_dim: int = 128, seed: int = 2,
                         device="cpu") -> tuple:
    """bf16 K or V ~ N(0, 1) in [B][Hkv][T_cap][D], the quantizer's input. Returns (x, seq_lens)."""
    device = torch.device(device)
    lens = [seq_lens] * batch if isinstance(seq_lens, int) else list(seq_lens)
    T = max(TOKEN_TILE, round_up(max(lens), TOKEN_TILE))
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((batch, num_kv_heads, T, head_dim), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16), torch.tensor(lens, dtype=torch.int32, device=device)


# ---------------------------------------------------------------- workloads

CONTEXTS = (4096, 16384, 32768, 65536, 131072)  # "4K ... 128K", K = 1024 tokens
BATCHES = (1, 8, 32, 64)


def tiny_int2(seed: int = 0) -> Workload:
    """Batch 1, 1 KV head, 4 query heads, 512 tokens, INT2 token-wise g=128."""
    return Workload("tiny-int2", 1, 4, 1, 512, bits=2, group=128, s_range=(0.01, 0.1), seed=seed)


def decode_int2(batch: int, ctx: int, seed: int = 1) -> Workload:
    """32q/8kv heads, head_dim 128, INT2 token-wise K/V with group 128."""
    return Workload(f"int2-tokenwise-b{batch}-ctx{ctx}", batch, 32, 8, ctx, bits=2, group=128,
                    s_range=(0.01, 0.1), seed=seed)


def decode_int4(batch: int, ctx: int, seed: int = 2) -> Workload:
    """Same shape at INT4: codes in 0..15, s ~ U[0.002, 0.02]."""
    return Workload(f"int4-tokenwise-b{batch}-ctx{ctx}", batch, 32, 8, ctx, bits=4, group=128,
                    s_range=(0.002, 0.02), seed=seed)


def ragged_lens(batch: int = 16, lo: int = 1024, hi: int = 65536, seed: int = 3) -> List[int]:
    """Lengths uniform in [lo, hi], redrawn while a multiple of 128."""
    rng = np.random.default_rng(seed)
    lens = []
    while len(lens) < batch:
        x = int(rng.integers(lo, hi + 1))
        if x % TOKEN_TILE:
            lens.append(x)
    return lens


def mixed_layout(bits: int, k_layout: int, v_layout: int, batch: int = 16, seed: int = 3,
                 lens: Optional[Sequence[int]] = None) -> Workload:
    """32q/8kv, ragged lengths, the given K/V layout pair (channel-wise over 128-token groups)."""
    lens = list(lens) if lens is not None else ragged_lens(batch, seed=seed)
    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    tag = f"{'cw' if k_layout else 'tw'}K-{'cw' if v_layout else 'tw'}V"
    return Workload(f"mixed-int{bits}-{tag}", len(lens), 32, 8, lens, bits=bits, k_layout=k_layout,
                    v_layout=v_layout, group=128, s_range=s, seed=seed)


def long_context(batch: int, group: int = 128, hq_per_kv: int = 4, seed: int = 4) -> Workload:
    """100,000-token context = 99,872 INT2 tokens + a 128-token bf16 window; 32 query heads."""
    return Workload(f"longctx-b{batch}-g{group}-gqa{hq_per_kv}", batch, 32, 32 // hq_per_kv, 99872, bits=2,
                    group=group, s_range=(0.01, 0.1), window=128, seed=seed)


# ---------------------------------------------------------------- paged cache

def page_table(lens: Sequence[int], page_tokens: int, max_pages: int, spare_pages: int = 3, seed: int = 5):
    """A page table int32 [B][max_pages] over a shuffled pool: the pages that hold a
    sequence's first lens[b] tokens take distinct pool pages in random order, the other
    entries are -1. The pool has `spare_pages` unused pages besides. Returns (table,
    num_pages)."""
    need = [(int(L) + page_tokens - 1) // page_tokens for L in lens]
    if any(n > max_pages for n in need):
        raise ValueError("a sequence needs more pages than a table row holds")
    num_pages = sum(need) + spare_pages
    perm = np.random.default_rng(seed).permutation(num_pages)
    table = np.full((len(lens), max_pages), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    return torch.from_numpy(table), num_pages


def to_pages(x: torch.Tensor, table: torch.Tensor, num_pages: int, page_tokens: int, tokens_per_row: int = 1):
    """Scatter a contiguous cache tensor [B][Hkv][R][...] (one row per `tokens_per_row`
    tokens: 1 for codes and token-wise scales, the group for channel-wise scales) into a
    pool [num_pages][Hkv][page_tokens / tokens_per_row][...] through the page table.
    Pool pages that no entry names are zero."""
    B, H, R = x.shape[:3]
    rp = page_tokens // tokens_per_row
    max_pages = table.shape[1]
    if R < max_pages * rp:
        pad = torch.zeros((B, H, max_pages * rp - R) + tuple(x.shape[3:]), dtype=x.dtype, device=x.device)
        x = torch.cat([x, pad], dim=2)
    xs = x[:, :, :max_pages * rp].reshape((B, H, max_pages, rp) + tuple(x.shape[3:])).transpose(1, 2)
    pool = torch.zeros((num_pages, H, rp) + tuple(x.shape[3:]), dtype=x.dtype, device=x.device)
    t = table.to(x.device).long()
    bs, js = torch.nonzero(t >= 0, as_tuple=True)
    pool[t[bs, js]] = xs[bs, js]
    return pool


def from_pages(pool: torch.Tensor, table: torch.Tensor, rows: int, tokens_per_row: int = 1):
    """The inverse of to_pages: a contiguous [B][Hkv][rows][...] tensor gathered from the
    pool (rows of -1 entries are zero)."""
    NP, H, rp = pool.shape[:3]
    B, max_pages = table.shape
    out = torch.zeros((B, max_pages, H, rp) + tuple(pool.shape[3:]), dtype=pool.dtype, device=pool.device)
    t = table.to(pool.device).long()
    bs, js = torch.nonzero(t >= 0, as_tuple=True)
    out[bs, js] = pool[t[bs, js]]
    out = out.transpose(1, 2).reshape((B, H, max_pages * rp) + tuple(pool.shape[3:]))
    return out[:, :, :rows].contiguous()
