"""Seeded synthetic inputs shaped like the serving workloads on the pages.

This module draws random numbers and builds index structures (page pools,
page tables, length mixes); it holds none of the kernels' arithmetic.  Both the
CUDA path and the fp64 oracle are fed from here, and from nowhere else.

Every generator takes an integer seed and a torch device; the same seed on the
same device gives the same tensors.  Values are drawn in fp32 and rounded once
to bf16.  Index tensors are int32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, std: float = 1.0, mean: float = 0.0,
                device="cpu") -> torch.Tensor:
    """N(mean, std^2) drawn in fp32, rounded to bf16."""
    g = _gen(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def uniform_int(n: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive), CPU int64."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


def loguniform_int(n: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """n integers log-uniform in [lo, hi]: round(exp(u * ln(hi/lo)) * lo),
    u ~ U(0,1), clamped to the range.  CPU int64."""
    g = _gen(seed, "cpu")
    u = torch.rand(n, generator=g, dtype=torch.float64)
    v = torch.exp(u * math.log(hi / lo)) * lo
    return v.round().clamp(lo, hi).to(torch.int64)


@dataclass
class PagedKV:
    """A paged K/V cache: k_cache, v_cache [num_pages, Hkv, page, D] bf16;
    block_table [B, max_blocks] int32 (unused slots hold 0); kv_lens [B] int32.
    Pages of all sequences are drawn from one shuffled pool, so neighbouring
    logical blocks live in unrelated physical pages."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    kv_lens: torch.Tensor
    page_size: int

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def num_pages(self) -> int:
        return self.k_cache.shape[0]


def paged_kv(kv_lens, Hkv: int, D: int, page_size: int, seed: int,
             reserve_tokens: int = 0, max_blocks: int | None = None,
             device="cpu", std: float = 1.0) -> PagedKV:
    """Build a shuffled page pool holding, for every sequence b, room for
    kv_lens[b] + reserve_tokens tokens, fill it with N(0, std^2) bf16 values
    and return the cache with its page table.  ``reserve_tokens`` leaves
    pages for tokens appended later (decode growth)."""
    lens = [int(v) for v in kv_lens]
    B = len(lens)
    need = [-(-(L + reserve_tokens) // page_size) for L in lens]
    mb = max(need + [1]) if max_blocks is None else int(max_blocks)
    if any(n > mb for n in need):
        raise ValueError("max_blocks too small for the requested lengths")
    total = max(sum(need), 1)
    g = _gen(seed, "cpu")
    perm = torch.randperm(total, generator=g)
    bt = torch.zeros(B, mb, dtype=torch.int32)
    pos = 0
    for b in range(B):
        bt[b, : need[b]] = perm[pos: pos + need[b]].to(torch.int32)
        pos += need[b]
    k = normal_bf16((total, Hkv, page_size, D), seed + 1, std=std, device=device)
    v = normal_bf16((total, Hkv, page_size, D), seed + 2, std=std, device=device)
    return PagedKV(k, v, bt.to(device), torch.tensor(lens, dtype=torch.int32,
                                                      device=device), page_size)


# ---------------------------------------------------------------------------
# the workloads (seeded; sizes as the serving scenarios on the pages)
# ---------------------------------------------------------------------------
TINY = dict(H=256, N=512, Hq=4, Hkv=2, D=64, B=8, max_len=512, page=16, split=64,
            eps=1e-6)
"""Tiny layer: RMSNorm over 256, GEMM 256->512, decode with 4/2 heads, D=64,
8 requests of KV length uniform in 1..512, page 16, split size 64."""

LLAMA_PROJ = dict(H=4096, N_qkv=6144, N_up=14336, eps=1e-6,
                  M_list=(1, 3, 16, 64, 256, 1024, 8192))
"""Llama-3-8B-shaped projection: RMSNorm over 4096, QKV GEMM 4096->6144,
MLP up-GEMM 4096->14336, M swept over the token counts listed."""

GQA_DECODE = dict(Hq=32, Hkv=8, D=128, page=16, B=64, max_len=32768, split=256,
                  steps=512)
"""GQA decode: 32/8 heads, D=128, page 16, 64 requests with KV length
log-uniform in 1..32768 (less the growth steps), split size 256."""

CHUNKED_PREFILL = dict(Hq=32, Hkv=8, D=128, page=16, T=8192, chunks=(512, 2048, 8192),
                       split=256)
"""Chunked prefill: one 8192-token prompt, 32/8 heads, D=128, chunks of 512,
2048 and 8192 tokens, split size 256."""


def seed_for(workload: int, stream: int) -> int:
    """Seeds are 1000 * workload number + stream id."""
    return 1000 * workload + stream
