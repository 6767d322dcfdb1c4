"""Plain fp64 CPU oracle for absorbed MLA decode over a paged latent KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never calls it, and it shares no code with the CUDA library.

What it computes (one "row" = one query token of one head):

* Absorbed decode is MQA with one shared key head of width 576 = 512 latent
  + 64 RoPE, and V is the first 512 columns of that same cached row
  (FlashMLA deep dive, "Theoretical Analysis"; DeepGEMM & FlashMLA article,
  section 6 "MLA", absorption identity; mla-analysis "absorption trick").
* Scores are ``softmax_scale * <q, k>`` over all 576 columns; the output is
  ``softmax(scores) @ V`` and ``lse`` is the natural log-sum-exp of the scaled
  scores (FlashMLA README, "Return Values": out [b, s_q, h_q, d_v],
  lse [b, h_q, s_q]).  The plain definition is written out directly: split-KV,
  online softmax and the split combine are exact rewrites of it
  (DeepGEMM & FlashMLA article, section 5 flash decode and section 7
  "split-KV" merge formula), so they appear here only as separate helpers
  (``attend_online``, ``combine``) that the tests use as pins.
* Paged cache: token ``t`` of request ``b`` is row ``t % 64`` of physical page
  ``block_table[b, t // 64]`` (FlashMLA README usage; the 64-token page block).
* Sparse (DSA) decode: the key set of query (b, s) is the multiset
  ``{indices[b, s, k] : index valid}``; each index is a flat pool row
  (page * page_size + offset), -1 marks an invalid slot (FlashMLA README,
  "indices Tensor").
* Sparse (DSA) prefill (FlashMLA README, "DeepSeek Sparse Attention (DSA)
  Prefill"): q [s_q, h_q, 576], kv [s_kv, 1, 576], indices [s_q, 1, topk];
  token i attends to the rows its own index list names, i.e. the sparse decode
  definition for one request of s_q query tokens (``sparse_prefill``).
* FP8 cache: 656 bytes per token = 512 e4m3 codes, 4 fp32 scales (one per 128
  channels), 64 bf16 RoPE values (FlashMLA "Hopper FP8 sparse decode" note,
  "The FP8 KVCache Format").
* V4.1 FP8 cache (FlashMLA README, "FP8 / FP4 KV Cache Format"): head_dim 512,
  528 bytes per token = 512 e4m3 codes covering all 512 dimensions (the RoPE
  dimensions are quantised too) followed by 16 e8m0 scales, one per 32
  consecutive codes.  A key is 512 wide and, with no separate latent part,
  the value is the whole key row (d_qk = d_v = 512).  e8m0 holds a power of
  two only, so e4m3 * scale has at most 4 significant bits: it is exactly a
  bf16 value, and the dequantised key is that exact product.  The kernel dequantises the codes into bf16
  before its bf16 MMAs (same note: convert e4m3 to bf16, multiply by the fp32
  scale; "we first dequantize ... into 512 bfloat16s"), so a key's latent value
  is bf16(e4m3(code) * scale): the exact product rounded once to bf16.

Readings where the pages are silent (each is listed in the design notes):

* Causal decode with s_q > 1: the last s_q cached positions are the new
  tokens, so query j of request b sees positions 0 .. L_b - s_q + j.
* An empty key set gives out = 0 and lse = -inf.
* An index outside [0, s_kv) other than -1 is treated as invalid.
* The FP8 dequantised value is the exact product e4m3 * scale rounded once to
  the nearest bf16 (ties to even).

Every array here is numpy float64 unless stated.  bf16 inputs may be passed
as uint16 bit patterns and are widened exactly (``widen``).
"""
from __future__ import annotations

import numpy as np

PAGE = 64
D_QK = 576
D_V = 512
FP8_TOKEN_BYTES = 656
FP8_V41_TOKEN_BYTES = 528
V41_HEAD_DIM = 512


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly.

    A bfloat16 is the upper half of an IEEE binary32 word.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """float8 e4m3 (fn variant) codes -> float64, from the bit definition.

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
    encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities,
    so the largest finite magnitude is 1.75 * 2^8 = 448 (the DeepGEMM & FlashMLA
    article's e4m3 description: 4 exponent + 3 mantissa bits, max 448).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    mag = np.where(e == 0, sub, normal)
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


def fp8_tokens_to_f64(raw: np.ndarray) -> np.ndarray:
    """656-byte FP8 cache tokens [..., 656] uint8 -> [..., 576] float64.

    latent[c] = e4m3(raw[c]) * scale[c // 128] for c < 512, where the four
    fp32 scales sit at bytes 512..527 (little-endian); the 64 RoPE values are
    bf16 at bytes 528..655.
    """
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == FP8_TOKEN_BYTES
    lead = raw.shape[:-1]
    codes = raw[..., :512]
    scales = raw[..., 512:528].copy().view("<f4").astype(np.float64)  # [..., 4]
    rope_bits = raw[..., 528:656].copy().view("<u2")                  # [..., 64]
    lat = e4m3_to_f64(codes).reshape(*lead, 4, 128) * scales[..., :, None]
    return np.concatenate([lat.reshape(*lead, 512), bf16_bits_to_f64(rope_bits)], axis=-1)


def e8m0_to_f64(codes: np.ndarray) -> np.ndarray:
    """float8 e8m0 scale codes -> float64: an 8-bit biased exponent and no
    sign or mantissa, value 2^(code - 127); code 255 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    return np.where(c == 255, np.nan, np.exp2(c - 127.0))


def fp8_v41_tokens_to_f64(raw: np.ndarray) -> np.ndarray:
    """528-byte V4.1 cache tokens [..., 528] uint8 -> [..., 512] float64:
    value[c] = e4m3(raw[c]) * e8m0(raw[512 + c // 32]) for c < 512."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == FP8_V41_TOKEN_BYTES
    lead = raw.shape[:-1]
    codes = e4m3_to_f64(raw[..., :512]).reshape(*lead, 16, 32)
    scales = e8m0_to_f64(raw[..., 512:528])
    return (codes * scales[..., :, None]).reshape(*lead, 512)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 value (8 significant bits, ties to even), as float64.

    x = m * 2^e with 0.5 <= |m| < 1; keep 8 bits of m by rounding m * 2^8 to
    the nearest integer (numpy's rint rounds halves to even).  Values in the
    bf16 normal range only (enough for dequantised cache values).
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def fp8_tokens_to_keys(raw: np.ndarray) -> np.ndarray:
    """656-byte FP8 tokens -> the bf16 keys the method attends over, as float64:
    latent = bf16(e4m3 * scale), RoPE = the stored bf16 values."""
    x = fp8_tokens_to_f64(raw)
    x[..., :512] = round_to_bf16(x[..., :512])
    return x


# ---------------------------------------------------------------------------
# The attention row definition
# ---------------------------------------------------------------------------

def attend(q_rows: np.ndarray, keys: np.ndarray, softmax_scale: float):
    """softmax(scale * q K^T) V for query rows sharing one key set.

    q_rows [R, d], keys [T, d] with V = keys[:, :512] (d = 576: 512 latent +
    64 RoPE; d = 512: the V4.1 head, where V is the whole key).
    Returns out [R, 512], lse [R] (natural log of sum exp of scaled scores).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    R = q_rows.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((R, D_V)), np.full(R, -np.inf)
    s = softmax_scale * (q_rows @ keys.T)                 # [R, T]
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)
    out = (e @ keys[:, :D_V]) / z[:, None]
    return out, m + np.log(z)


def attend_online(q_row: np.ndarray, keys: np.ndarray, softmax_scale: float):
    """One query row by the streaming (flash-decode) recurrence.

    Keeps a running max m, running sum l and accumulator acc; each key
    rescales the old state by exp(m_old - m_new) (DeepGEMM & FlashMLA
    article, section 5).  Used only as a pin for ``attend``.
    """
    q_row = np.asarray(q_row, dtype=np.float64)
    m, l = -np.inf, 0.0
    acc = np.zeros(D_V)
    for k in np.asarray(keys, dtype=np.float64):
        s = softmax_scale * float(q_row @ k)
        m_new = max(m, s)
        alpha = np.exp(m - m_new) if m != -np.inf else 0.0
        p = np.exp(s - m_new)
        l = l * alpha + p
        acc = acc * alpha + p * k[:D_V]
        m = m_new
    if l == 0.0:
        return np.zeros(D_V), -np.inf
    return acc / l, m + np.log(l)


def combine(parts):
    """Merge per-split (out_i, lse_i) into the result over the union of keys.

    The article's split-KV merge: m = max m_i, l = sum l_i e^{m_i - m},
    o = sum o_i l_i e^{m_i - m} / l, written with lse_i = m_i + ln l_i, so the
    weight of split i is exp(lse_i - lse).  Splits with lse = -inf (empty)
    contribute nothing.
    """
    outs = np.stack([np.asarray(o, dtype=np.float64) for o, _ in parts])      # [S, R, 512]
    lses = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])      # [S, R]
    mx = lses.max(axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    w = np.exp(lses - safe[None, :])
    tot = w.sum(axis=0)
    lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    out = np.einsum("sr,srd->rd", w, outs) / np.where(tot > 0, tot, 1.0)[:, None]
    return out, lse


# ---------------------------------------------------------------------------
# Key sets
# ---------------------------------------------------------------------------

def visible_length(seqlen: int, s_q: int, j: int, causal: bool) -> int:
    """Keys visible to query token j of a request with ``seqlen`` cached tokens."""
    if not causal:
        return int(seqlen)
    return max(0, int(seqlen) - s_q + 1 + j)


def widen(x: np.ndarray) -> np.ndarray:
    """float64 view of an input array: uint16 arrays are bf16 bit patterns,
    uint8 arrays with a last dimension of 656 are FP8 cache tokens (decoded
    to their bf16 keys), of 528 V4.1 FP8 tokens (decoded exactly), anything
    else is converted with ``astype``."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    if x.dtype == np.uint8 and x.shape[-1] == FP8_TOKEN_BYTES:
        return fp8_tokens_to_keys(x)
    if x.dtype == np.uint8 and x.shape[-1] == FP8_V41_TOKEN_BYTES:
        return fp8_v41_tokens_to_f64(x)
    return x.astype(np.float64)


def paged_keys(kv_cache: np.ndarray, block_table_row: np.ndarray, n: int) -> np.ndarray:
    """The first ``n`` tokens of one request, read through its page table,
    widened to float64 [n, 576]."""
    t = np.arange(n)
    pages = np.asarray(block_table_row)[t // PAGE].astype(np.int64)
    return widen(kv_cache[pages, t % PAGE])


def sparse_keys(kv_pool: np.ndarray, index_row: np.ndarray) -> np.ndarray:
    """Pool rows named by one query's index list; -1 and out-of-range skipped."""
    idx = np.asarray(index_row).astype(np.int64)
    valid = (idx >= 0) & (idx < kv_pool.shape[0])
    return widen(kv_pool[idx[valid]])


# ---------------------------------------------------------------------------
# Whole-call references
# ---------------------------------------------------------------------------

def dense_decode(q, kv_cache, block_table, cache_seqlens, softmax_scale,
                 causal=True, rows=None):
    """Paged dense decode.

    q [b, s_q, h, 576] and kv_cache [n_pages, 64, 576] (float64, or uint16
    bf16 bit patterns; kv_cache may also be [n_pages, 64, 656] uint8 FP8
    tokens), block_table [b, max_pages] int, cache_seqlens [b] int.
    Returns out [b, s_q, h, 512], lse [b, h, s_q].  With ``rows`` (a list of
    (b, j) pairs) only those query tokens are computed and the rest of the
    output is NaN.
    """
    q = widen(q)
    b, s_q, h, _ = q.shape
    out = np.full((b, s_q, h, D_V), np.nan)
    lse = np.full((b, h, s_q), np.nan)
    todo = rows if rows is not None else [(bi, j) for bi in range(b) for j in range(s_q)]
    for bi, j in todo:
        n = visible_length(int(cache_seqlens[bi]), s_q, j, causal)
        keys = paged_keys(kv_cache, block_table[bi], n)
        o, l = attend(q[bi, j], keys, softmax_scale)
        out[bi, j] = o
        lse[bi, :, j] = l
    return out, lse


def fp8_v41_dense_decode(q, kv_raw, block_table, cache_seqlens, softmax_scale,
                         causal=True, rows=None):
    """Paged decode over the 528-byte V4.1 FP8 cache: q [b, s_q, h, 512],
    kv_raw [n_pages, 64, 528] uint8; each gathered token decodes exactly to
    its 512-wide key, which is also its value row."""
    kv_raw = np.asarray(kv_raw, dtype=np.uint8)
    assert kv_raw.shape[-1] == FP8_V41_TOKEN_BYTES
    return dense_decode(q, kv_raw, block_table, cache_seqlens, softmax_scale, causal, rows)


def fp8_dense_decode(q, kv_raw, block_table, cache_seqlens, softmax_scale,
                     causal=True, rows=None):
    """Paged decode over the 656-byte FP8 cache; each gathered token is decoded
    to its bf16 key by ``fp8_tokens_to_keys`` before the dense definition applies."""
    kv_raw = np.asarray(kv_raw, dtype=np.uint8)
    assert kv_raw.shape[-1] == FP8_TOKEN_BYTES
    return dense_decode(q, kv_raw, block_table, cache_seqlens, softmax_scale, causal, rows)


def sink_factor(lse: np.ndarray, attn_sink: np.ndarray) -> np.ndarray:
    """exp(lse) / (exp(lse) + exp(attn_sink)) per head, the factor the
    FlashMLA sparse interface ("attn_sink") multiplies each output row by; 0
    when the key set is empty (lse = -inf)."""
    lse = np.asarray(lse, dtype=np.float64)
    sink = np.asarray(attn_sink, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        f = 1.0 / (1.0 + np.exp(sink - lse))
    return np.where(np.isneginf(lse), 0.0, f)


def sparse_decode(q, kv_pool, indices, softmax_scale, rows=None, attn_sink=None, topk_length=None):
    """DSA top-k decode: q [b, s_q, h, 576], kv_pool [s_kv, 576],
    indices [b, s_q, topk] int (-1 = invalid).

    attn_sink [h] (optional): each head's output row is scaled by
    sink_factor(lse, attn_sink[h]); lse is unchanged.  topk_length [b, s_q]
    (optional): query token (b, j) uses only its first topk_length[b, j]
    index slots, clamped to [0, topk] (FlashMLA sparse interface,
    "attn_sink" and "topk_length")."""
    q = widen(q)
    b, s_q, h, _ = q.shape
    topk = indices.shape[-1]
    out = np.full((b, s_q, h, D_V), np.nan)
    lse = np.full((b, h, s_q), np.nan)
    todo = rows if rows is not None else [(bi, j) for bi in range(b) for j in range(s_q)]
    lengths = None if topk_length is None else np.asarray(topk_length).reshape(b, s_q)
    for bi, j in todo:
        n = topk if lengths is None else min(max(int(lengths[bi, j]), 0), topk)
        keys = sparse_keys(kv_pool, indices[bi, j][:n])
        o, l = attend(q[bi, j], keys, softmax_scale)
        if attn_sink is not None:
            o = o * sink_factor(l, attn_sink)[:, None]
        out[bi, j] = o
        lse[bi, :, j] = l
    return out, lse


def sparse_prefill(q, kv_pool, indices, softmax_scale, tokens=None, attn_sink=None, topk_length=None):
    """DSA sparse prefill (FlashMLA README, "DeepSeek Sparse Attention (DSA)
    Prefill", flash_mla_sparse_fwd): q [s_q, h, 576], kv_pool [s_kv, 576] or
    [s_kv, 1, 576], indices [s_q, topk] or [s_q, 1, topk] (-1 = invalid),
    optional attn_sink [h] and topk_length [s_q] as for sparse_decode.

    Each query token attends to the rows its own index list names: the sparse
    decode definition with each token a request of one query token.  Returns
    out [s_q, h, 512] and lse [s_q, h] (the decode call's lse [b, h, s_q] with
    b = s_q tokens of one query each).  ``tokens`` limits the work to those
    query tokens (others stay NaN)."""
    q = np.asarray(q)
    s_q = q.shape[0]
    pool = np.asarray(kv_pool).reshape(np.asarray(kv_pool).shape[0], -1)
    idx = np.asarray(indices).reshape(s_q, 1, -1)
    rows = None if tokens is None else [(int(j), 0) for j in tokens]
    tl = None if topk_length is None else np.asarray(topk_length).reshape(s_q, 1)
    out, lse = sparse_decode(q[:, None], pool, idx, softmax_scale, rows=rows, attn_sink=attn_sink,
                             topk_length=tl)
    return out[:, 0], lse[:, :, 0]
