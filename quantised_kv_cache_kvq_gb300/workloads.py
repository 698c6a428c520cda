"""Seeded synthetic workloads for the quantised KV cache.

This module only draws random numbers.  It holds none of the method's arithmetic;
the CUDA path and the oracle both consume what it produces.  Inputs are shaped like
the Llama 3 8B attention layer the cache pages discuss ("Quantizing the KV cache",
"In an LLM": 32 query heads, 8 KV heads, head size 128), with the structure the
pages describe for real caches:
  * keys have a few outlier channels that are large in every token
    ("Keys and values are shaped differently");
  * a few value tokens have a larger magnitude in all their channels (same section).

Recipe (all normal draws N(0, 1), scaling in fp32, then one round-to-nearest-even
conversion to bf16 when the workload is bf16):
  * K[token, head, c] = N(0,1) * mult[head, c], where each (layer, kv head) has
    `k_outliers` distinct channels drawn without replacement, each with a fixed
    multiplier drawn from U[mult_lo, mult_hi] (or exactly `mult_lo` when the two
    are equal); all other channels have multiplier 1.
  * V[token, head, c] = N(0,1) * (v_outlier_mult if token is a value outlier else 1),
    each (sequence, token) being an outlier with probability `v_outlier_prob`,
    shared by all KV heads of that token.
  * q ~ N(0,1) * q_mult.
"""
from dataclasses import dataclass, field
import math
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    scheme: int                 # 0 KIVI, 1 INT8 per-token symmetric, 2 FP8 E4M3
    layers: int
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    context: Tuple[int, int]    # (lo, hi) tokens per sequence; lo == hi for a fixed context
    bits: int = 8
    group_k: int = 32
    group_v: int = 32
    residual: int = 0
    in_dtype: str = "bf16"      # "bf16" or "f32"
    k_outliers: int = 4
    mult_lo: float = 8.0
    mult_hi: float = 16.0
    v_outlier_prob: float = 0.01
    v_outlier_mult: float = 8.0
    q_mult: float = 1.0
    softmax_scale: Optional[float] = None   # None: 1/sqrt(head_dim)
    seed: int = 0
    steps: int = 1              # decode steps in the workload
    page_groups: int = 0        # KIVI paged layout: group records per page (0: contiguous)
    rope_base: float = 0.0      # KIVI keys cached before the rotary embedding (its base)
    outliers: int = 0           # KIVI dense-and-sparse: elements per quantisation vector kept in bf16

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def gqa(self) -> int:
        return self.q_heads // self.kv_heads


# The five workloads: a tiny INT8 case, the KIVI 2-bit Llama-3-8B layer, the 32-layer FP8
# cache, the 128k-token KIVI 4-bit context and the ragged serving mix.
WORKLOADS = {
    "int8_tiny": Workload(
        "int8_tiny", scheme=1, layers=1, batch=1, q_heads=4, kv_heads=4, head_dim=32,
        context=(256, 256), in_dtype="f32", k_outliers=2, mult_lo=10.0, mult_hi=10.0,
        v_outlier_prob=0.0, q_mult=1.0 / math.sqrt(32.0), softmax_scale=1.0, seed=0),
    "kivi2_llama3_8b": Workload(
        "kivi2_llama3_8b", scheme=0, layers=1, batch=8, q_heads=32, kv_heads=8, head_dim=128,
        context=(4096, 4096), bits=2, group_k=32, group_v=32, residual=128, seed=1),
    "fp8_32layer": Workload(
        "fp8_32layer", scheme=2, layers=32, batch=64, q_heads=32, kv_heads=8, head_dim=128,
        context=(8192, 8192), seed=2),
    "kivi4_128k": Workload(
        "kivi4_128k", scheme=0, layers=1, batch=1, q_heads=32, kv_heads=8, head_dim=128,
        context=(131072, 131072), bits=4, group_k=128, group_v=128, residual=128, seed=3),
    "serve_mix": Workload(
        "serve_mix", scheme=0, layers=1, batch=256, q_heads=32, kv_heads=8, head_dim=128,
        context=(1024, 32768), bits=2, group_k=32, group_v=32, residual=128, seed=4, steps=64),
    # the serving mix with its group records in a page pool (16 groups = 512 tokens a page),
    # pages handed out in a shuffled order
    "serve_mix_paged": Workload(
        "serve_mix_paged", scheme=0, layers=1, batch=256, q_heads=32, kv_heads=8, head_dim=128,
        context=(1024, 32768), bits=2, group_k=32, group_v=32, residual=128, seed=4, steps=64,
        page_groups=16),
    # the KIVI 2-bit Llama-3-8B layer with its keys cached before the rotary embedding
    # (Llama 3's base 500000), the decode turning every key by its position
    "kivi2_llama3_8b_rope": Workload(
        "kivi2_llama3_8b_rope", scheme=0, layers=1, batch=8, q_heads=32, kv_heads=8, head_dim=128,
        context=(4096, 4096), bits=2, group_k=32, group_v=32, residual=128, seed=1, rope_base=500000.0),
    # the 4-bit 128k-token context with one outlier per quantisation vector kept in bf16
    # (1 of 128 elements, 0.8%: the dense-and-sparse split at about 1%)
    "kivi4_128k_sparse": Workload(
        "kivi4_128k_sparse", scheme=0, layers=1, batch=1, q_heads=32, kv_heads=8, head_dim=128,
        context=(131072, 131072), bits=4, group_k=128, group_v=128, residual=128, seed=3, outliers=1),
}


def block_table(w: Workload, max_tokens: int, device="cpu"):
    """Paged workloads: (num_pages, int32 [batch][max_pages] block table) for caches of
    `max_tokens` tokens per sequence -- every page of every sequence, in a shuffled order
    over a pool with 1% spare pages."""
    ng = (max_tokens - w.residual) // w.group_k if max_tokens > w.residual else 0
    mp = (ng + w.page_groups - 1) // w.page_groups
    pool = w.batch * mp + max(1, w.batch * mp // 100)
    g = _gen((w.seed, "pages"), "cpu")
    perm = torch.randperm(pool, generator=g)[: w.batch * mp].to(torch.int32)
    return pool, perm.view(w.batch, mp).to(device)


def _gen(seed_parts, device) -> torch.Generator:
    # a stable 63-bit seed from the tuple, independent of Python's hash randomisation
    h = 1469598103934665603
    for p in seed_parts:
        for byte in str(p).encode():
            h = ((h ^ byte) * 1099511628211) & ((1 << 63) - 1)
    g = torch.Generator(device=device)
    g.manual_seed(h)
    return g


def key_multipliers(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    """[kv_heads, head_dim] fp32 per-channel key multipliers of one layer."""
    g = _gen((w.seed, "kmult", layer), "cpu")
    mult = torch.ones(w.kv_heads, w.head_dim, dtype=torch.float32)
    for h in range(w.kv_heads):
        idx = torch.randperm(w.head_dim, generator=g)[: w.k_outliers]
        if w.mult_hi > w.mult_lo:
            vals = w.mult_lo + (w.mult_hi - w.mult_lo) * torch.rand(w.k_outliers, generator=g)
        else:
            vals = torch.full((w.k_outliers,), w.mult_lo)
        mult[h, idx] = vals
    return mult.to(device)


def context_lengths(w: Workload) -> torch.Tensor:
    """[batch] int64 context length of every sequence."""
    lo, hi = w.context
    if lo == hi:
        return torch.full((w.batch,), lo, dtype=torch.int64)
    g = _gen((w.seed, "ctx"), "cpu")
    return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64)


def _dtype(w: Workload):
    return torch.bfloat16 if w.in_dtype == "bf16" else torch.float32


def kv_tokens(w: Workload, layer: int, seq0: int, nseq: int, tok0: int, ntok: int,
              device="cpu", tag="ctx") -> Tuple[torch.Tensor, torch.Tensor]:
    """K, V for sequences [seq0, seq0+nseq) and token positions [tok0, tok0+ntok), laid out
    [nseq][ntok][kv_heads][head_dim] in the workload's input dtype.  Deterministic in
    (seed, layer, seq0, nseq, tok0, ntok, tag, device type)."""
    g = _gen((w.seed, tag, layer, seq0, nseq, tok0, ntok), device)
    shape = (nseq, ntok, w.kv_heads, w.head_dim)
    mult = key_multipliers(w, layer, device)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    k.mul_(mult.view(1, 1, w.kv_heads, w.head_dim))
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if w.v_outlier_prob > 0:
        hit = torch.rand((nseq, ntok), generator=g, device=device) < w.v_outlier_prob
        v.mul_(torch.where(hit, w.v_outlier_mult, 1.0).view(nseq, ntok, 1, 1))
    return k.to(_dtype(w)), v.to(_dtype(w))


def queries(w: Workload, layer: int, step: int = 0, device="cpu") -> torch.Tensor:
    """[batch][q_heads][head_dim] query of one decode step."""
    g = _gen((w.seed, "q", layer, step), device)
    q = torch.randn((w.batch, w.q_heads, w.head_dim), generator=g, device=device,
                    dtype=torch.float32) * w.q_mult
    return q.to(_dtype(w))


def fp8_scales(w: Workload, k: torch.Tensor, v: torch.Tensor) -> torch.Tensor:
    """[kv_heads][2] per-(kv head) amax/448 scales (K, V) over a layer's fill, the static
    per-head scale the FP8 cache uses."""
    ka = k.float().abs().amax(dim=(0, 1, 3))
    va = v.float().abs().amax(dim=(0, 1, 3))
    s = torch.stack([ka, va], dim=1) / 448.0
    return torch.where(s > 0, s, torch.ones_like(s)).to(torch.float32).contiguous()
