"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random tensors and names the workload shapes. It holds
none of the attention arithmetic, so both the CUDA path and the fp64 oracle can
take their inputs from it without sharing any computation.

Workload shapes follow the pages' examples:

* ``mha_l256_d64``: a small non-causal multi-head case (two heads, 256 tokens,
  head_dim 64), the size at which the oracle checks every element.
* ``single_head_l8192_d128_causal``: the L=8192, d=128 BF16 single-head case of
  the FlashAttention accounting table ("把平方级的中间矩阵变成统计量", §3 table
  of the clxhxhhr.top S23-J17 page).
* ``mha_b2_h16_l2048_d64_fp16_causal``: B=2, H=16, N=2048, D=64 in FP16 with
  ``is_causal=True``, the SDPA backend experiment of the ans20xx.com day14 page
  (实验 2), generated directly in (B, L, H, d) layout.
* ``gqa_b2_hq32_hkv8_l4096_d128_causal``: the GQA module of the lei6393.com
  training-integration page (§2.3: num_heads=32, num_heads_kv=8, embed 4096,
  causal), at L=4096 and B=2.
* ``varlen_b16_h12_d64``: the BERT-style 768/12 module with a key padding mask
  (same page, §2.1 and §2.5), as 16 sequences whose lengths are uniform in
  [64, 512], packed back to back (padding at the end of each row is dropped).

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
as float32 N(0, 1) and then rounded once to the storage dtype; the rounded
tensors are what both sides consume.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Workload:
    """Shape of one attention forward problem."""

    name: str
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    d: int
    dtype: str = "bf16"
    causal: bool = False
    seed: int = 0
    # varlen: per-sequence lengths are drawn from U[len_lo, len_hi]
    varlen: bool = False
    len_lo: int = 0
    len_hi: int = 0
    scale: Optional[float] = None

    @property
    def softmax_scale(self) -> float:
        # default 1/sqrt(head_dim) (lei6393.com training page, §8.5)
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "mha_l256_d64": Workload("mha_l256_d64", B=1, Hq=2, Hkv=2, Lq=256, Lk=256, d=64,
                             dtype="bf16", causal=False, seed=0),
    "single_head_l8192_d128_causal": Workload(
        "single_head_l8192_d128_causal", B=1, Hq=1, Hkv=1, Lq=8192, Lk=8192, d=128,
        dtype="bf16", causal=True, seed=1),
    "mha_b2_h16_l2048_d64_fp16_causal": Workload(
        "mha_b2_h16_l2048_d64_fp16_causal", B=2, Hq=16, Hkv=16, Lq=2048, Lk=2048, d=64,
        dtype="fp16", causal=True, seed=2),
    "gqa_b2_hq32_hkv8_l4096_d128_causal": Workload(
        "gqa_b2_hq32_hkv8_l4096_d128_causal", B=2, Hq=32, Hkv=8, Lq=4096, Lk=4096, d=128,
        dtype="bf16", causal=True, seed=3),
    "varlen_b16_h12_d64": Workload(
        "varlen_b16_h12_d64", B=16, Hq=12, Hkv=12, Lq=512, Lk=512, d=64,
        dtype="bf16", causal=False, seed=4, varlen=True, len_lo=64, len_hi=512),
}

# The configuration the headline metric is quoted on.
HEADLINE = "single_head_l8192_d128_causal"


@dataclass
class Inputs:
    """One drawn problem.

    Dense: q is (B, Lq, Hq, d), k and v are (B, Lk, Hkv, d).
    Varlen: q, k, v are packed (total, H, d); ``lengths`` holds the B sequence
    lengths and ``cu_seqlens`` their B+1 running offsets (int32, cu[0] = 0).
    """

    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    lengths: Optional[List[int]] = None
    cu_seqlens: Optional[torch.Tensor] = None
    max_len: int = 0
    extra: dict = field(default_factory=dict)


def _randn(g: torch.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def draw_lengths(wl: Workload, g: torch.Generator) -> List[int]:
    return [int(x) for x in torch.randint(wl.len_lo, wl.len_hi + 1, (wl.B,), generator=g)]


def generate(wl: Workload, seed: Optional[int] = None, lengths: Optional[List[int]] = None) -> Inputs:
    """Draw q, k, v (and lengths for varlen) for ``wl`` on the CPU."""
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    dt = wl.torch_dtype
    if wl.varlen:
        if lengths is None:
            lengths = draw_lengths(wl, g)
        assert len(lengths) == wl.B
        total = int(sum(lengths))
        q = _randn(g, (total, wl.Hq, wl.d), dt)
        k = _randn(g, (total, wl.Hkv, wl.d), dt)
        v = _randn(g, (total, wl.Hkv, wl.d), dt)
        cu = [0]
        for n in lengths:
            cu.append(cu[-1] + int(n))
        cu_t = torch.tensor(cu, dtype=torch.int32)
        return Inputs(wl, q, k, v, lengths=list(lengths), cu_seqlens=cu_t,
                      max_len=max(lengths) if lengths else 0)
    q = _randn(g, (wl.B, wl.Lq, wl.Hq, wl.d), dt)
    k = _randn(g, (wl.B, wl.Lk, wl.Hkv, wl.d), dt)
    v = _randn(g, (wl.B, wl.Lk, wl.Hkv, wl.d), dt)
    return Inputs(wl, q, k, v)


def sample_rows(wl: Workload, n: int, seed: int = 1234, lengths: Optional[List[int]] = None):
    """Pick ``n`` (b, h, i) query rows spread over the problem, always
    including the first and last row of every batch and both extreme heads."""
    g = torch.Generator().manual_seed(seed)
    rows = set()
    Bs = range(wl.B)
    for b in Bs:
        L = lengths[b] if lengths is not None else wl.Lq
        for h in {0, wl.Hq - 1}:
            for i in {0, 1, L // 2, L - 2, L - 1}:
                if 0 <= i < L:
                    rows.add((b, h, i))
    while len(rows) < n:
        b = int(torch.randint(0, wl.B, (1,), generator=g))
        L = lengths[b] if lengths is not None else wl.Lq
        h = int(torch.randint(0, wl.Hq, (1,), generator=g))
        i = int(torch.randint(0, L, (1,), generator=g))
        rows.add((b, h, i))
    return sorted(rows)
