"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module is shared by the tests, ``bench.py`` and the oracle-side checks.  It
holds the workload shapes and the random draws only: no attention arithmetic.
The encoding steps here are the FP8 cache formats of the inputs:
* 656 bytes (FlashMLA "Hopper FP8 sparse decode" note, section "The FP8
  KVCache Format"): per token 512 float8_e4m3 latent values quantised in
  1x128 tiles, 4 float32 scales, then 64 bfloat16 RoPE values; scales are
  ``absmax / 448`` in fp32;
* 528 bytes (FlashMLA README, "FP8 / FP4 KV Cache Format", DeepSeek V4.1,
  head_dim 512): 512 float8_e4m3 values covering all dimensions, then 16
  float8_e8m0 scales, one per 32 values; an e8m0 scale is a power of two, here
  the smallest one at or above ``absmax / 448`` (so no code saturates).
The e4m3 rounding itself is ``torch.float8_e4m3fn``'s cast (round to nearest
even).

Shapes follow the DeepSeek-V3 MLA decode setting described on the pages
(128 query heads, one shared 576-wide latent+RoPE key row, V = the first 512
columns of that row, page blocks of 64 tokens).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

D_QK = 576          # 512 latent + 64 RoPE
D_V = 512
D_ROPE = 64
PAGE = 64           # page block size (tokens)
FP8_TOKEN_BYTES = 656   # 512 e4m3 + 4 x fp32 scale + 64 x bf16
FP8_TILE = 128      # channels per fp32 scale
FP8_V41_TOKEN_BYTES = 528   # 512 e4m3 + 16 e8m0 scales
V41_HEAD_DIM = 512  # V4.1: key = value = 512 dims (RoPE dims included)
V41_TILE = 32       # values per e8m0 scale
E4M3_MAX = 448.0
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)
TAIL_MAGNITUDE = 1.0e4  # finite junk placed in page slots past the sequence end


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload."""
    name: str
    kind: str                 # "dense" | "sparse" | "fp8" (656 B) | "fp8_v41" (528 B)
    b: int
    s_q: int
    h: int
    seqlens: Optional[tuple] = None     # fixed per-request cache lengths
    seqlen_range: Optional[tuple] = None  # (lo, hi) uniform integer draw
    causal: bool = True
    extra_pages: int = 0      # unused pool pages (dense / fp8)
    s_kv: int = 0             # sparse pool rows
    topk: int = 0
    invalid_per_row: int = 0  # sparse: indices set to -1 per row
    seed: int = 0
    prefill: bool = False     # sparse: run through the prefill entry point (b tokens, s_q = 1)


# The five graded shapes.  Seeds 1..5 follow the configuration order.
WORKLOADS = {
    "tiny": Workload("tiny", "dense", b=2, s_q=1, h=16, seqlens=(200, 333),
                     extra_pages=6, seed=1),
    "dense_v3": Workload("dense_v3", "dense", b=64, s_q=1, h=128,
                         seqlens=(4096,) * 64, seed=2),
    "spec": Workload("spec", "dense", b=128, s_q=2, h=128,
                     seqlen_range=(1024, 16384), seed=3),
    "dsa": Workload("dsa", "sparse", b=64, s_q=1, h=128, s_kv=32768,
                    topk=2048, invalid_per_row=102, seed=4),
    "fp8": Workload("fp8", "fp8", b=64, s_q=1, h=128, seqlens=(8192,) * 64,
                    seed=5),
}
# Sparse prefill (FlashMLA README, "DeepSeek Sparse Attention (DSA) Prefill";
# no shape is given there): a chunk of 2048 query tokens over a 32768-row pool,
# 2048 index slots per token with the DSA recipe above.  Held as 2048
# "requests" of one query token each, the layout the prefill call maps to.
WORKLOADS["sparse_prefill"] = Workload("sparse_prefill", "sparse", b=2048, s_q=1, h=128, s_kv=32768,
                                       topk=2048, invalid_per_row=102, seed=6, prefill=True)


def scaled(w: Workload, **kw) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **kw)


def _draw_seqlens(w: Workload, g: torch.Generator) -> torch.Tensor:
    if w.seqlens is not None:
        assert len(w.seqlens) == w.b
        return torch.tensor(w.seqlens, dtype=torch.int32)
    lo, hi = w.seqlen_range
    return torch.randint(lo, hi + 1, (w.b,), generator=g, dtype=torch.int64).to(torch.int32)


def _bf16_normal(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _page_layout(seqlens: torch.Tensor, extra_pages: int, g: torch.Generator):
    """Random physical placement of each request's pages.

    Returns (block_table [b, max_pages] int32 with -1 past each request's last
    page, n_pool_pages).
    """
    n_pages = [(int(L) + PAGE - 1) // PAGE for L in seqlens.tolist()]
    total = sum(n_pages) + extra_pages
    perm = torch.randperm(total, generator=g).to(torch.int32)
    max_pages = max(1, max(n_pages))
    bt = torch.full((len(n_pages), max_pages), -1, dtype=torch.int32)
    pos = 0
    for i, n in enumerate(n_pages):
        bt[i, :n] = perm[pos:pos + n]
        pos += n
    return bt, total


def _tail_junk(shape, g: torch.Generator) -> torch.Tensor:
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.int64) * 2 - 1
    return (sign.to(torch.float32) * TAIL_MAGNITUDE)


def _fill_tails(rows: torch.Tensor, seqlens, block_table, g) -> None:
    """Overwrite page slots past each request's length with +-1e4 (in place).

    ``rows`` is the float32 pool [n_pages, PAGE, D].  These slots are never
    part of any attention row; large finite values prove the masking.
    """
    for i, L in enumerate(seqlens.tolist()):
        if L % PAGE == 0 or L == 0:
            continue
        last = int(block_table[i, (L - 1) // PAGE])
        off = L % PAGE
        rows[last, off:] = _tail_junk(rows[last, off:].shape, g)


def dense_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """bf16 paged-cache inputs (also the base of the fp8 inputs)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    seqlens = _draw_seqlens(w, g)
    bt, n_pool = _page_layout(seqlens, w.extra_pages, g)
    kv = torch.randn((n_pool, PAGE, D_QK), generator=g, dtype=torch.float32)
    _fill_tails(kv, seqlens, bt, g)
    q = _bf16_normal((w.b, w.s_q, w.h, D_QK), g)
    return dict(q=q, kv_cache=kv.to(torch.bfloat16), block_table=bt,
                cache_seqlens=seqlens, softmax_scale=SOFTMAX_SCALE,
                causal=w.causal)


def quantize_fp8_tokens(x: torch.Tensor) -> torch.Tensor:
    """Encode float32 token rows [..., 576] into the 656-byte FP8 layout.

    Bytes [0, 512): e4m3 codes of x[:512] / scale[c // 128]; bytes [512, 528):
    four little-endian fp32 scales (absmax of each 128-channel tile / 448, or
    1.0 for an all-zero tile); bytes [528, 656): the 64 RoPE values as bf16.
    """
    lead = x.shape[:-1]
    lat = x[..., :D_V].reshape(*lead, D_V // FP8_TILE, FP8_TILE)
    amax = lat.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    codes = (lat / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    codes = codes.reshape(*lead, D_V)
    scale_b = scale.contiguous().view(torch.uint8).reshape(*lead, 16)
    rope_b = x[..., D_V:].to(torch.bfloat16).contiguous().view(torch.uint8).reshape(*lead, 2 * D_ROPE)
    return torch.cat([codes, scale_b, rope_b], dim=-1).contiguous()


def fp8_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """FP8 (656 B/token) paged-cache inputs with bf16 queries."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    seqlens = _draw_seqlens(w, g)
    bt, n_pool = _page_layout(seqlens, w.extra_pages, g)
    kv = torch.randn((n_pool, PAGE, D_QK), generator=g, dtype=torch.float32)
    _fill_tails(kv, seqlens, bt, g)
    q = _bf16_normal((w.b, w.s_q, w.h, D_QK), g)
    return dict(q=q, kv_cache=quantize_fp8_tokens(kv), block_table=bt,
                cache_seqlens=seqlens, softmax_scale=SOFTMAX_SCALE,
                causal=w.causal)


def quantize_fp8_v41_tokens(x: torch.Tensor) -> torch.Tensor:
    """Encode float32 token rows [..., 512] into the 528-byte V4.1 layout.

    Bytes [0, 512): e4m3 codes of x / scale[c // 32]; bytes [512, 528): the 16
    e8m0 scale codes (biased exponents: scale = 2^(code - 127)), each the
    smallest power of two at or above absmax / 448 of its 32 values (code 127,
    scale 1, for an all-zero block).
    """
    lead = x.shape[:-1]
    blocks = x.reshape(*lead, V41_HEAD_DIM // V41_TILE, V41_TILE)
    ratio = blocks.abs().amax(dim=-1) / E4M3_MAX
    mant, expo = torch.frexp(ratio)              # ratio = mant * 2^expo, 0.5 <= mant < 1
    up = torch.where(mant == 0.5, expo - 1, expo)  # ceil(log2(ratio))
    up = torch.where(ratio > 0, up, torch.zeros_like(up)).clamp(-127, 127)
    scale = torch.pow(2.0, up.to(torch.float32))
    codes = (blocks / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    codes = codes.reshape(*lead, V41_HEAD_DIM)
    sc = (up + 127).to(torch.uint8)
    return torch.cat([codes, sc], dim=-1).contiguous()


def fp8_v41_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """V4.1 FP8 (528 B/token) paged-cache inputs with bf16 queries of 512."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    seqlens = _draw_seqlens(w, g)
    bt, n_pool = _page_layout(seqlens, w.extra_pages, g)
    kv = torch.randn((n_pool, PAGE, V41_HEAD_DIM), generator=g, dtype=torch.float32)
    _fill_tails(kv, seqlens, bt, g)
    q = _bf16_normal((w.b, w.s_q, w.h, V41_HEAD_DIM), g)
    return dict(q=q, kv_cache=quantize_fp8_v41_tokens(kv), block_table=bt,
                cache_seqlens=seqlens, softmax_scale=SOFTMAX_SCALE,
                causal=w.causal)


def sparse_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """DSA top-k inputs: a flat pool of latent rows and per-query indices.

    Per (b, s) query row: ``topk`` distinct pool rows drawn without
    replacement; ``invalid_per_row`` slots among 1..topk-1 set to -1; slot 0
    is a valid "selected" row i*.  Heads h = 0 (mod 4) get q = 0.25 * kv[i*]
    (peaked rows dominated by one key); the other heads are N(0,1).
    """
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    pool = _bf16_normal((w.s_kv, D_QK), g)
    idx = torch.empty((w.b, w.s_q, w.topk), dtype=torch.int32)
    for bi in range(w.b):
        for si in range(w.s_q):
            idx[bi, si] = torch.randperm(w.s_kv, generator=g)[:w.topk].to(torch.int32)
            if w.invalid_per_row:
                slots = torch.randperm(w.topk - 1, generator=g)[:w.invalid_per_row] + 1
                idx[bi, si, slots] = -1
    q = torch.randn((w.b, w.s_q, w.h, D_QK), generator=g, dtype=torch.float32)
    for bi in range(w.b):
        for si in range(w.s_q):
            star = int(idx[bi, si, 0])
            q[bi, si, 0::4] = 0.25 * pool[star].to(torch.float32)
    return dict(q=q.to(torch.bfloat16), kv=pool, indices=idx,
                softmax_scale=SOFTMAX_SCALE)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    if w.kind == "dense":
        return dense_inputs(w, seed)
    if w.kind == "fp8":
        return fp8_inputs(w, seed)
    if w.kind == "fp8_v41":
        return fp8_v41_inputs(w, seed)
    if w.kind == "sparse":
        return sparse_inputs(w, seed)
    raise ValueError(w.kind)
