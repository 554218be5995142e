"""Seeded synthetic inputs for the decode-step tail.

This module only draws inputs: logits with the shapes and value distributions
of the five workloads, per-request sampling parameters, uniforms, write-back
targets and paged-KV lengths / free lists.  It holds none of the method's
arithmetic, so both the CUDA path's tests and the CPU oracle's tests can use
it.  Every tensor is a CPU tensor; callers move what they need to the device.

Workloads (B rows, V vocabulary):
  * ``pr1``     -- B=4, V=32000 fp32 N(0, 3^2); rows 0-1 greedy, row 2
                   T=0.7 top_p=0.9, row 3 T=1.0 top_k=50 top_p=0.95; pages of 4.
  * ``greedy``  -- B=64, V=128256 bf16 N(0, 2^2) with a planted +16 maximum per
                   row (two or three tied maxima in every 4th row); all greedy;
                   write-back into an int32 token pool [64, 8192].
  * ``mixed``   -- B=256, V=151936 bf16 N(0, 3^2); every 3rd row greedy, the rest
                   T~U[0.5,1.5], top_k in {off, 20, 50}, top_p in {1, 0.9, 0.95};
                   pages of 16.
  * ``nucleus`` -- B=256, V=151936 fp32 Zipf-shaped rows
                   (logit = -1.1 ln(rank) + N(0, 0.5^2), ranks permuted per row),
                   T=0.8 top_p=0.9; one-token decode step with pages of 1.
  * ``large``   -- B=1024, V=256000 bf16 N(0, 4^2); T~U[0.3,1.2], top_k=1024 then
                   top_p=0.95; pages of 64 from 200000 free pages.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

NAMES = ("pr1", "greedy", "mixed", "nucleus", "large")
SEEDS = {name: 1000 + i for i, name in enumerate(NAMES)}


@dataclass
class Workload:
    name: str
    logits: torch.Tensor                    # [B, V] fp32 or bf16
    temperature: Optional[torch.Tensor]     # [B] fp32; None = all greedy
    top_k: Optional[torch.Tensor]           # [B] int32; None = off
    top_p: Optional[torch.Tensor]           # [B] fp32; None = off
    uniform: Optional[torch.Tensor]         # [B] fp32 in [0, 1)
    pool_shape: tuple                       # token pool [rows, cols] int32
    wb_rows: torch.Tensor                   # [B] int32 (table_idx)
    wb_cols: torch.Tensor                   # [B] int64 (device_len, or -1)
    page_size: int = 1
    cached_len: Optional[torch.Tensor] = None   # [B] int32
    device_len: Optional[torch.Tensor] = None   # [B] int32
    table_idx: Optional[torch.Tensor] = None    # [B] int32
    free_slots: Optional[torch.Tensor] = None   # [F] int32 page-start token locations
    pt_shape: tuple = (0, 0)                # page table [rows, cols] int32
    notes: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def V(self) -> int:
        return self.logits.shape[1]

    @property
    def elt(self) -> int:
        return self.logits.element_size()


def _align_up_32(x: int) -> int:
    return (x + 31) // 32 * 32


def _gen(name: str, seed: Optional[int]) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(SEEDS[name] if seed is None else seed)
    return g


def pr1(seed: Optional[int] = None) -> Workload:
    g = _gen("pr1", seed)
    B, V = 4, 32000
    logits = torch.randn(B, V, generator=g) * 3.0
    temperature = torch.tensor([0.0, 0.0, 0.7, 1.0], dtype=torch.float32)
    top_k = torch.tensor([-1, -1, -1, 50], dtype=torch.int32)
    top_p = torch.tensor([1.0, 1.0, 0.9, 0.95], dtype=torch.float32)
    uniform = torch.rand(B, generator=g)
    cached = torch.tensor([0, 6, 3, 10], dtype=torch.int32)
    device = torch.tensor([5, 9, 4, 13], dtype=torch.int32)
    table_idx = torch.arange(B, dtype=torch.int32)
    return Workload(
        name="pr1", logits=logits, temperature=temperature, top_k=top_k,
        top_p=top_p, uniform=uniform, pool_shape=(B + 1, 32),
        wb_rows=table_idx.clone(), wb_cols=device.to(torch.int64), page_size=4,
        cached_len=cached, device_len=device, table_idx=table_idx,
        free_slots=torch.arange(64, dtype=torch.int32) * 4, pt_shape=(B + 1, 32))


def greedy(seed: Optional[int] = None) -> Workload:
    g = _gen("greedy", seed)
    B, V = 64, 128256
    base = torch.randn(B, V, generator=g) * 2.0
    planted = torch.randint(0, V, (B,), generator=g)
    base[torch.arange(B), planted] = 16.0
    for r in range(0, B, 4):  # exact ties at the maximum in every 4th row
        extra = int(torch.randint(1, 3, (1,), generator=g))
        idx = torch.randint(0, V, (extra,), generator=g)
        base[r, idx] = 16.0
    logits = base.to(torch.bfloat16)
    rows = torch.randperm(B, generator=g).to(torch.int32)
    cols = torch.randint(0, 8192, (B,), generator=g).to(torch.int64)
    return Workload(
        name="greedy", logits=logits, temperature=None, top_k=None, top_p=None,
        uniform=None, pool_shape=(B, 8192), wb_rows=rows, wb_cols=cols)


def mixed(seed: Optional[int] = None, B: int = 256, V: int = 151936) -> Workload:
    g = _gen("mixed", seed)
    logits = (torch.randn(B, V, generator=g) * 3.0).to(torch.bfloat16)
    temperature = torch.rand(B, generator=g) + 0.5
    greedy_rows = torch.arange(B) % 3 == 0
    temperature[greedy_rows] = 0.0
    k_choice = torch.tensor([-1, 20, 50], dtype=torch.int32)
    p_choice = torch.tensor([1.0, 0.9, 0.95], dtype=torch.float32)
    top_k = k_choice[torch.randint(0, 3, (B,), generator=g)]
    top_p = p_choice[torch.randint(0, 3, (B,), generator=g)]
    uniform = torch.rand(B, generator=g)
    ps = 16
    cached = torch.randint(0, 2000, (B,), generator=g).to(torch.int32)
    device = cached + torch.randint(1, 513, (B,), generator=g).to(torch.int32)
    table_idx = torch.randperm(B + 1, generator=g)[:B].to(torch.int32)
    free_slots = (torch.randperm(65536, generator=g) * ps).to(torch.int32)
    width = _align_up_32(2000 + 512)
    return Workload(
        name="mixed", logits=logits, temperature=temperature, top_k=top_k,
        top_p=top_p, uniform=uniform, pool_shape=(B + 1, width),
        wb_rows=table_idx.clone(), wb_cols=device.to(torch.int64), page_size=ps,
        cached_len=cached, device_len=device, table_idx=table_idx,
        free_slots=free_slots, pt_shape=(B + 1, width))


def nucleus(seed: Optional[int] = None, B: int = 256, V: int = 151936) -> Workload:
    g = _gen("nucleus", seed)
    ranks = torch.arange(1, V + 1, dtype=torch.float64)
    shape = (-1.1 * torch.log(ranks)).to(torch.float32)
    logits = torch.empty(B, V, dtype=torch.float32)
    for b in range(B):
        perm = torch.randperm(V, generator=g)
        logits[b, perm] = shape + torch.randn(V, generator=g) * 0.5
    temperature = torch.full((B,), 0.8, dtype=torch.float32)
    top_p = torch.full((B,), 0.9, dtype=torch.float32)
    uniform = torch.rand(B, generator=g)
    cached = torch.randint(0, 2000, (B,), generator=g).to(torch.int32)
    device = cached + 1
    table_idx = torch.randperm(B + 1, generator=g)[:B].to(torch.int32)
    free_slots = torch.randperm(65536, generator=g).to(torch.int32)
    width = _align_up_32(2000 + 1)
    return Workload(
        name="nucleus", logits=logits, temperature=temperature, top_k=None,
        top_p=top_p, uniform=uniform, pool_shape=(B + 1, width),
        wb_rows=table_idx.clone(), wb_cols=device.to(torch.int64), page_size=1,
        cached_len=cached, device_len=device, table_idx=table_idx,
        free_slots=free_slots, pt_shape=(B + 1, width))


def large(seed: Optional[int] = None, B: int = 1024, V: int = 256000) -> Workload:
    g = _gen("large", seed)
    logits = (torch.randn(B, V, generator=g) * 4.0).to(torch.bfloat16)
    temperature = torch.rand(B, generator=g) * 0.9 + 0.3
    top_k = torch.full((B,), 1024, dtype=torch.int32)
    top_p = torch.full((B,), 0.95, dtype=torch.float32)
    uniform = torch.rand(B, generator=g)
    ps = 64
    cached = torch.randint(0, 32768, (B,), generator=g).to(torch.int32)
    device = cached + torch.randint(1, 4097, (B,), generator=g).to(torch.int32)
    table_idx = torch.randperm(B + 1, generator=g)[:B].to(torch.int32)
    free_slots = (torch.randperm(200000, generator=g) * ps).to(torch.int32)
    width = _align_up_32(32767 + 4096)
    return Workload(
        name="large", logits=logits, temperature=temperature, top_k=top_k,
        top_p=top_p, uniform=uniform, pool_shape=(B + 1, width),
        wb_rows=table_idx.clone(), wb_cols=device.to(torch.int64), page_size=ps,
        cached_len=cached, device_len=device, table_idx=table_idx,
        free_slots=free_slots, pt_shape=(B + 1, width))


BUILDERS = {"pr1": pr1, "greedy": greedy, "mixed": mixed, "nucleus": nucleus,
            "large": large}


def make(name: str, seed: Optional[int] = None, **kw) -> Workload:
    return BUILDERS[name](seed=seed, **kw)


def random_rows(B: int, V: int, dtype: torch.dtype, seed: int, scale: float = 3.0,
                discrete: bool = False) -> torch.Tensor:
    """Generic seeded logits; ``discrete`` draws small integers to force ties."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if discrete:
        x = torch.randint(-4, 5, (B, V), generator=g).to(torch.float32)
    else:
        x = torch.randn(B, V, generator=g) * scale
    return x.to(dtype)


def random_params(B: int, seed: int, greedy_frac: float = 0.3,
                  k_values=(-1, 1, 2, 5, 20, 50), p_values=(1.0, 0.5, 0.9, 0.95, 1e-6),
                  t_range=(0.3, 1.5)):
    """Seeded per-request temperature / top_k / top_p / uniform vectors."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    t = torch.rand(B, generator=g) * (t_range[1] - t_range[0]) + t_range[0]
    t[torch.rand(B, generator=g) < greedy_frac] = 0.0
    kv = torch.tensor(k_values, dtype=torch.int32)
    pv = torch.tensor(p_values, dtype=torch.float32)
    k = kv[torch.randint(0, len(k_values), (B,), generator=g)]
    p = pv[torch.randint(0, len(p_values), (B,), generator=g)]
    u = torch.rand(B, generator=g)
    return t, k, p, u


def release_batch(B: int, page_size: int, num_pages: int, seed: int, max_len: int = 2512,
                  ragged: bool = True):
    """Seeded inputs of a batched release of finished requests.

    Every request first owns ``device_len`` tokens from position 0 (allocated
    from ``free_slots``, a permutation of the pool's page starts); then the
    slice ``[begin, end)`` of its table row is freed.  ``ragged`` mixes whole
    rows (begin 0), unaligned begins, empty and reversed ranges; otherwise
    every request frees [0, device_len).  Returns a dict of CPU tensors and
    the page-table shape.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    device_len = torch.randint(1, max_len + 1, (B,), generator=g).to(torch.int32)
    table_idx = torch.randperm(B + 1, generator=g)[:B].to(torch.int32)
    free_slots = (torch.randperm(num_pages, generator=g) * page_size).to(torch.int32)
    if ragged:
        begin = torch.randint(0, 2 * page_size + 1, (B,), generator=g).to(torch.int32)
        end = (device_len - torch.randint(0, 3, (B,), generator=g).to(torch.int32))
        begin[torch.rand(B, generator=g) < 0.5] = 0
        end[torch.rand(B, generator=g) < 0.1] = 0  # empty or reversed
    else:
        begin = torch.zeros(B, dtype=torch.int32)
        end = device_len.clone()
    width = _align_up_32(max_len)
    return {"device_len": device_len, "table_idx": table_idx, "free_slots": free_slots,
            "begin": begin, "end": end.to(torch.int32), "pt_shape": (B + 1, width)}
