"""Algorithmic FLOP and byte counts for one MLA decode call.

FLOPs: each visible (row, token) pair costs one 576-long dot product and one
512-long accumulation, 2 * (576 + 512) = 2176 FLOP (mla-analysis cost model,
FlashMLA: 2bhst(2k + p); FlashMLA deep dive: 2 h_q s_q s_k (d_k + d_v)).

Bytes: every KV token a request needs is read once (1152 B bf16, 656 B FP8),
every query row reads its q (1152 B) and writes its output (1024 B) and LSE
(4 B); the page table and lengths are read once (mla-analysis byte model
w(bhs(2k + p) + bt(k + p)) plus the LSE, page table and length words).
"""
from __future__ import annotations

D_QK, D_V = 576, 512
FLOP_PER_PAIR = 2 * (D_QK + D_V)
BF16_TOKEN_BYTES = 2 * D_QK
FP8_TOKEN_BYTES = 656


def visible_lengths(seqlens, s_q: int, causal: bool):
    """Per (request, query token) visible key count, causal aligned to the end."""
    out = []
    for L in seqlens:
        for j in range(s_q):
            out.append(max(0, int(L) - s_q + 1 + j) if causal else int(L))
    return out


def dense_counts(seqlens, s_q: int, h: int, causal: bool = True, fp8: bool = False,
                 page: int = 64):
    """(flops, bytes, kv_bytes) for a paged dense decode call."""
    vis = visible_lengths(seqlens, s_q, causal)
    flops = FLOP_PER_PAIR * h * sum(vis)
    tok_bytes = FP8_TOKEN_BYTES if fp8 else BF16_TOKEN_BYTES
    kv_bytes = tok_bytes * sum(int(L) for L in seqlens)
    rows = len(seqlens) * s_q * h
    pages = sum((int(L) + page - 1) // page for L in seqlens)
    bytes_ = kv_bytes + rows * (2 * D_QK + 2 * D_V + 4) + 4 * pages + 4 * len(seqlens)
    return flops, bytes_, kv_bytes


def sparse_counts(valid_per_query, h: int, topk: int):
    """(flops_valid, flops_nominal, bytes, kv_bytes) for a top-k sparse call.

    ``valid_per_query`` lists the valid index count of each (request, query
    token); the nominal figure counts all ``topk`` slots (how sparse TFLOPS
    are usually quoted).
    """
    n_q = len(valid_per_query)
    flops = FLOP_PER_PAIR * h * sum(valid_per_query)
    flops_nom = FLOP_PER_PAIR * h * topk * n_q
    kv_bytes = BF16_TOKEN_BYTES * sum(valid_per_query)
    rows = n_q * h
    bytes_ = kv_bytes + rows * (2 * D_QK + 2 * D_V + 4) + 4 * topk * n_q
    return flops, flops_nom, bytes_, kv_bytes


def mla_analysis_bytes(b, h, s, t, k=512, p=64, w=2):
    """The mla-analysis page's FlashMLA byte model w(bhs(2k+p) + bt(k+p))."""
    return w * (b * h * s * (2 * k + p) + b * t * (k + p))


def mla_analysis_flops(b, h, s, t, k=512, p=64):
    """The mla-analysis page's FlashMLA FLOP model 2bhst(2k+p)."""
    return 2 * b * h * s * t * (2 * k + p)
