"""Seeded synthetic inputs for the sparse decode step.

This module only draws random numbers and fixes shapes. It computes nothing of
the method itself (no paging arithmetic, no scores, no selection, no
attention), so that both the CUDA path and the CPU oracle can take their inputs
from it without sharing any of the method's arithmetic.

The five named workloads follow the shapes of the long-context,
high-concurrency decode workloads that the sources describe ("Sparse Attention
on GLM5.3 and HBM", HiSparse section; "Paged KV cache", worked example):

* ``paging_example``  - the five requests of the paged-KV worked example
  (403/96/241/30/176 tokens, 16-token pages), small enough for the oracle.
* ``b32_4k``          - 32 x 4096 tokens, 64-token pages, pool pages permuted.
* ``b64_ragged_prefix`` - 64 ragged requests (1k-32k tokens), groups of 8
  sharing a 2000-token prefix, 16-token pages.
* ``b16_128k``        - 16 x 131072 tokens, 4-head indexer, top-2048.
* ``b256_8k_lru``     - 256 x 8192 tokens, HBM slot table holding half of the
  pages (LRU), compacted miss list per step.

Three more follow the DeepSeek Sparse Attention paragraphs of the same page,
whose sparse MLA runs in MQA mode (latent d = 512 plus RoPE r = 64 per token,
one row shared by all query heads; H = 128 for DeepSeek V3.2, 64 for GLM-5).
Their ``Hq`` is the MLA head count H, ``D`` the key width d + r, ``Hkv`` 1:

* ``mla_paging_example`` - the worked example's five requests, H = 128, top-64.
* ``mla_b16_128k``       - 16 x 131072 tokens, H = 128, top-2048.
* ``mla_b64_32k_h64``    - 64 x 32768 tokens, H = 64, top-2048.

``hs_b16_32k`` (below) is the HBM-residency workload of the miss fetch
(HiSparse paragraph): a top-k that leaves about a third of the pages
unselected, and a slot table for three quarters of the pages.

Value distributions: K/V and attention queries are N(0, 1) rounded to bf16
(round to nearest even); indexer queries and keys are integers uniform in
[-127, 127]; indexer head weights are all one ("summed").
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    """Shape of one decode-step workload.

    ``seq_lens`` fixes the request lengths outright; otherwise they are drawn
    uniformly from ``[len_lo, len_hi]``.  ``group_size > 0`` puts consecutive
    blocks of ``group_size`` requests into prefix groups sharing the first
    ``prefix_len`` tokens.  ``num_pages`` is the size of the physical page pool
    (an upper bound on what the requests need), ``max_pages`` the width of a
    block-table row.  ``capacity > 0`` enables the HBM residency table with that
    many slots, initially holding ``initial_resident`` randomly chosen pages.
    """

    name: str
    B: int
    page_size: int
    Hq: int
    Hkv: int
    D: int
    Hi: int
    Di: int
    k: int
    num_pages: int
    max_pages: int
    seed: int
    seq_lens: Optional[tuple] = None
    len_lo: int = 0
    len_hi: int = 0
    prefix_len: int = 0
    group_size: int = 0
    permute_pool: bool = False
    capacity: int = 0
    initial_resident: int = 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def max_len(self) -> int:
        return self.max_pages * self.page_size


WORKLOADS = {
    "paging_example": Workload(
        name="paging_example", B=5, seq_lens=(403, 96, 241, 30, 176), page_size=16,
        Hq=8, Hkv=2, D=64, Hi=1, Di=64, k=64, num_pages=64, max_pages=32, seed=0),
    "b32_4k": Workload(
        name="b32_4k", B=32, seq_lens=(4096,) * 32, page_size=64, Hq=32, Hkv=8, D=128,
        Hi=1, Di=128, k=512, num_pages=2048, max_pages=64, seed=1, permute_pool=True),
    "b64_ragged_prefix": Workload(
        name="b64_ragged_prefix", B=64, len_lo=1024, len_hi=32768, page_size=16,
        Hq=32, Hkv=8, D=128, Hi=1, Di=128, k=2048, num_pages=64 * 2048, max_pages=2048,
        seed=2, prefix_len=2000, group_size=8),
    "b16_128k": Workload(
        name="b16_128k", B=16, seq_lens=(131072,) * 16, page_size=64, Hq=64, Hkv=8,
        D=128, Hi=4, Di=128, k=2048, num_pages=16 * 2048, max_pages=2048, seed=3),
    "b256_8k_lru": Workload(
        name="b256_8k_lru", B=256, seq_lens=(8192,) * 256, page_size=64, Hq=32, Hkv=8,
        D=128, Hi=1, Di=128, k=1024, num_pages=256 * 128, max_pages=128, seed=4,
        capacity=16384, initial_resident=16384),
}

#: the workloads in the order they are listed above
WORKLOAD_ORDER = ["paging_example", "b32_4k", "b64_ragged_prefix", "b16_128k", "b256_8k_lru"]

MLA_LATENT = 512  # d; the key width D of an MLA workload is d + r = 576

MLA_WORKLOADS = {
    "mla_paging_example": Workload(
        name="mla_paging_example", B=5, seq_lens=(403, 96, 241, 30, 176), page_size=16,
        Hq=128, Hkv=1, D=576, Hi=1, Di=64, k=64, num_pages=64, max_pages=32, seed=10),
    "mla_b16_128k": Workload(
        name="mla_b16_128k", B=16, seq_lens=(131072,) * 16, page_size=64, Hq=128, Hkv=1,
        D=576, Hi=4, Di=128, k=2048, num_pages=32768, max_pages=2048, seed=13),
    "mla_b64_32k_h64": Workload(
        name="mla_b64_32k_h64", B=64, seq_lens=(32768,) * 64, page_size=64, Hq=64, Hkv=1,
        D=576, Hi=1, Di=128, k=2048, num_pages=32768, max_pages=512, seed=14,
        permute_pool=True),
}


#: HBM-residency workloads whose top-k leaves pages unselected, so that a
#: slot table larger than one step's pages admits the misses of the next:
#: 16 x 32768 tokens in 16-token pages, top-2048 (about 64% of a request's
#: pages touched per step), 75% of the pages fit in HBM.
HISPARSE_WORKLOADS = {
    "hs_b16_32k": Workload(
        name="hs_b16_32k", B=16, seq_lens=(32768,) * 16, page_size=16, Hq=64, Hkv=8, D=128,
        Hi=4, Di=128, k=2048, num_pages=16 * 2048, max_pages=2048, seed=5,
        capacity=24576, initial_resident=24576),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_host(wl: Workload) -> dict:
    """Small host-side draws (CPU generator, independent of where tensors live).

    Returns int32 CPU tensors: ``seq_lens`` [B]; ``prefix_group`` [B] (-1 = no
    group) or None; ``free_order`` [num_pages] (a permutation of the pool) or
    None for the ascending pool; ``initial_resident`` (sorted page ids) or None.
    """
    g = _gen("cpu", wl.seed)
    if wl.seq_lens is not None:
        assert len(wl.seq_lens) == wl.B
        seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32)
    else:
        seq_lens = torch.randint(wl.len_lo, wl.len_hi + 1, (wl.B,), generator=g,
                                 dtype=torch.int64).to(torch.int32)
    prefix_group = None
    if wl.group_size > 0:
        prefix_group = (torch.arange(wl.B, dtype=torch.int32) // wl.group_size).to(torch.int32)
    free_order = None
    if wl.permute_pool:
        free_order = torch.randperm(wl.num_pages, generator=g, dtype=torch.int64).to(torch.int32)
    initial_resident = None
    if wl.capacity > 0:
        pick = torch.randperm(wl.num_pages, generator=g, dtype=torch.int64)[: wl.initial_resident]
        initial_resident = torch.sort(pick).values.to(torch.int32)
    return dict(seq_lens=seq_lens, prefix_group=prefix_group, free_order=free_order,
                initial_resident=initial_resident)


def draw_tensors(wl: Workload, device="cpu", seed_offset: int = 0) -> dict:
    """Large draws on ``device``: query tensors and the physical page pools.

    ``seed_offset`` gives a fresh query set over the same shapes (used to vary
    the selection between steps).  Returns: ``q`` bf16 [B, Hq, D]; ``q_idx``
    int8 [B, Hi, Di]; ``w_idx`` int32 [Hi] (ones); ``kv_k`` / ``kv_v`` bf16
    [num_pages, page_size, Hkv, D]; ``idx_k`` int8 [num_pages, page_size, Di].
    """
    g = _gen(device, wl.seed * 1000003 + 7919 * seed_offset + 17)
    P = wl.page_size
    pool = (wl.num_pages, P, wl.Hkv, wl.D)
    kv_k = torch.randn(pool, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    kv_v = torch.randn(pool, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    idx_k = torch.randint(-127, 128, (wl.num_pages, P, wl.Di), generator=g, device=device,
                          dtype=torch.int8)
    q, q_idx = draw_queries(wl, device, seed_offset)
    w_idx = torch.ones(wl.Hi, dtype=torch.int32, device=device)
    return dict(q=q, q_idx=q_idx, w_idx=w_idx, kv_k=kv_k, kv_v=kv_v, idx_k=idx_k)


def draw_queries(wl: Workload, device="cpu", seed_offset: int = 0):
    """Per-step query draws: ``q`` bf16 [B, Hq, D] and ``q_idx`` int8 [B, Hi, Di]."""
    g = _gen(device, wl.seed * 7777 + 104729 * (seed_offset + 1) + 3)
    q = torch.randn((wl.B, wl.Hq, wl.D), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    q_idx = torch.randint(-127, 128, (wl.B, wl.Hi, wl.Di), generator=g, device=device,
                          dtype=torch.int8)
    return q, q_idx


def draw_mla_tensors(wl: Workload, device="cpu", seed_offset: int = 0) -> dict:
    """Large draws of an MLA workload on ``device``: ``q`` bf16 [B, H, d + r];
    ``kv`` bf16 [num_pages, page_size, d + r] (one latent row per token);
    ``q_idx`` int8 [B, Hi, Di]; ``w_idx`` int32 [Hi] (ones); ``idx_k`` int8
    [num_pages, page_size, Di]."""
    g = _gen(device, wl.seed * 1000003 + 7919 * seed_offset + 29)
    P = wl.page_size
    kv = torch.randn((wl.num_pages, P, wl.D), generator=g, device=device,
                     dtype=torch.float32).to(torch.bfloat16)
    idx_k = torch.randint(-127, 128, (wl.num_pages, P, wl.Di), generator=g, device=device,
                          dtype=torch.int8)
    q, q_idx = draw_queries(wl, device, seed_offset)
    w_idx = torch.ones(wl.Hi, dtype=torch.int32, device=device)
    return dict(q=q, q_idx=q_idx, w_idx=w_idx, kv=kv, idx_k=idx_k)


def draw_float_weights(wl: Workload, device="cpu", seed_offset: int = 0, signed: bool = False):
    """Real-valued indexer head weights, float32 [B, Hi]: uniform in [0.25, 2)
    (or [-2, 2) when ``signed``), one row per request."""
    g = _gen("cpu", wl.seed * 4099 + 31 * seed_offset + 5)
    u = torch.rand((wl.B, wl.Hi), generator=g, dtype=torch.float32)
    w = u * 4.0 - 2.0 if signed else 0.25 + u * 1.75
    return w.to(device)


def draw_fp8_indexer(wl: Workload, device="cpu", seed_offset: int = 0):
    """FP8 e4m3 indexer queries [B, Hi, Di] and keys [num_pages, page_size, Di]:
    N(0, 4^2) rounded to e4m3 (finite codes only), returned as int8 tensors
    holding the bit patterns."""
    g = _gen(device, wl.seed * 6007 + 13 * seed_offset + 11)
    q = (torch.randn((wl.B, wl.Hi, wl.Di), generator=g, device=device) * 4.0)
    k = (torch.randn((wl.num_pages, wl.page_size, wl.Di), generator=g, device=device) * 4.0)
    f8 = torch.float8_e4m3fn
    return q.clamp(-448, 448).to(f8).view(torch.int8), k.clamp(-448, 448).to(f8).view(torch.int8)
