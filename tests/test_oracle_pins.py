"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against a closed form, an invariant of the
mathematics, a brute-force computation written independently here, a library
routine (torch's float8 / bfloat16 conversions), or a number printed on the
pages (tests/golden/page_numbers.json).  Chosen so that a dropped term (RoPE
columns), a wrong operand (V columns, transposes), a wrong index (page/offset,
causal end, scale block) or a wrong sign fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_gb300 import roofline, workloads
from tests._util import bf16_np

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
SCALE = 1.0 / math.sqrt(192.0)


def rng(seed=0):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- formats

def test_bf16_widening_matches_torch():
    bits = rng(1).integers(0, 1 << 16, size=20000, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_bits_to_f64(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e4m3_closed_values():
    v = oracle.e4m3_to_f64(np.array([0x7E, 0x01, 0x08, 0x38, 0xB8, 0x00, 0x80], dtype=np.uint8))
    assert v[0] == GOLDEN["e4m3_max"]["value"] == 448.0
    assert v[1] == 2.0 ** -9          # smallest subnormal
    assert v[2] == 2.0 ** -6          # smallest normal
    assert v[3] == 1.0 and v[4] == -1.0
    assert v[5] == 0.0 and v[6] == 0.0
    assert np.isnan(oracle.e4m3_to_f64(np.array([0x7F], dtype=np.uint8)))[0]


def test_fp8_token_layout_offsets():
    """Byte offsets 0 / 512 / 528 and the c // 128 scale block, built by hand."""
    tok = np.zeros(656, dtype=np.uint8)
    tok[0:512] = 0x38                                     # every code = 1.0
    scales = np.array([2.0, 3.0, 5.0, 7.0], dtype="<f4")
    tok[512:528] = scales.view(np.uint8)
    rope = torch.arange(64, dtype=torch.float32).to(torch.bfloat16)
    tok[528:656] = rope.view(torch.int16).numpy().view(np.uint8)
    x = oracle.fp8_tokens_to_f64(tok[None])[0]
    assert x.shape == (576,)
    for blk in range(4):
        assert np.all(x[blk * 128:(blk + 1) * 128] == scales[blk])
    assert np.array_equal(x[512:], np.arange(64, dtype=np.float64))
    parts = GOLDEN["fp8_token_bytes"]["parts"]
    assert sum(parts) == GOLDEN["fp8_token_bytes"]["value"] == oracle.FP8_TOKEN_BYTES == 656


def test_fp8_quantise_decode_error_bound():
    """Input encoder + oracle decoder: e4m3 round-to-nearest bound per element.

    |x - decode(encode(x))| <= 2^-4 |x| (half an ulp of a 3-bit mantissa) for
    normal codes, <= 2^-10 * scale for subnormal ones; RoPE round-trips bf16.
    """
    g = torch.Generator().manual_seed(7)
    x = torch.randn(32, 576, generator=g)
    x[:, 128:256] *= 50.0
    x[:, 256:384] *= 0.001
    raw = workloads.quantize_fp8_tokens(x).numpy()
    assert raw.shape == (32, 656)
    dec = oracle.fp8_tokens_to_f64(raw)
    xs = x.to(torch.float64).numpy()
    scales = raw[:, 512:528].copy().view("<f4").astype(np.float64)
    for blk in range(4):
        sl = slice(blk * 128, (blk + 1) * 128)
        amax = np.abs(xs[:, sl]).max(axis=1)
        assert np.allclose(scales[:, blk], (amax.astype(np.float32) / np.float32(448.0)), rtol=0, atol=0)
        err = np.abs(dec[:, sl] - xs[:, sl])
        bound = np.maximum(2.0 ** -4 * np.abs(xs[:, sl]), 2.0 ** -10 * scales[:, blk:blk + 1]) * (1 + 1e-6)
        assert np.all(err <= bound + 1e-12)
    rope_ref = x[:, 512:].to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(dec[:, 512:], rope_ref)


def test_e8m0_all_codes_match_torch():
    """All 256 e8m0 scale codes decode like torch's float8_e8m0fnu (2^(c-127),
    255 = NaN)."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e8m0_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).float().double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert ours[127] == 1.0 and ours[0] == 2.0 ** -127 and ours[254] == 2.0 ** 127


def test_fp8_v41_token_layout_offsets():
    """A 528-byte token built by hand: codes at bytes 0..511, one e8m0 scale
    per 32 codes at bytes 512..527 (the page's 512 + 16 = 528)."""
    g = GOLDEN["fp8_v41_token_bytes"]
    assert g["value"] == sum(g["parts"]) == oracle.FP8_V41_TOKEN_BYTES
    assert g["parts"][0] // g["values_per_scale"] == g["parts"][1]
    raw = np.zeros((1, 528), dtype=np.uint8)
    raw[0, 0] = 0x38        # e4m3 1.0
    raw[0, 31] = 0x40       # 2.0, same 32-block as byte 0
    raw[0, 32] = 0x38       # 1.0, the next block
    raw[0, 480] = 0x3C      # 1.5, block 15
    raw[0, 511] = 0xB8      # -1.0, block 15
    raw[0, 512] = 127 + 3   # block 0 scale 8
    raw[0, 513] = 127 - 2   # block 1 scale 0.25
    raw[0, 527] = 127       # block 15 scale 1
    dec = oracle.fp8_v41_tokens_to_f64(raw)[0]
    want = np.zeros(512)
    want[0], want[31], want[32], want[480], want[511] = 8.0, 16.0, 0.25, 1.5, -1.0
    assert np.array_equal(dec, want)


def test_fp8_v41_quantise_decode_error_bound():
    """Each 32-value block's scale is the power of two at or above
    absmax / 448 and below twice that; each value is within half an e4m3 step
    (2^-4 relative, or 2^-10 * scale below the e4m3 normal range)."""
    from mla_decode_attention_gb300 import workloads
    x = torch.randn((7, 512), generator=torch.Generator().manual_seed(5)) * 3
    x[2, :32] = 0.0                                       # an all-zero block
    raw = workloads.quantize_fp8_v41_tokens(x).numpy()
    dec = oracle.fp8_v41_tokens_to_f64(raw)
    scale = oracle.e8m0_to_f64(raw[:, 512:]).repeat(32, axis=1)
    amax = np.abs(x.double().numpy()).reshape(7, 16, 32).max(axis=2).repeat(32, axis=1)
    nz = amax > 0
    assert np.all(scale[nz] >= amax[nz] / 448) and np.all(scale[nz] < 2 * amax[nz] / 448)
    assert np.all(scale[~nz] == 1.0) and np.all(dec[2, :32] == 0.0)
    err = np.abs(dec - x.double().numpy())
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(x.double().numpy()), 2.0 ** -10 * scale))


def test_fp8_v41_keys_are_exact_bf16_values():
    """e4m3 * 2^k has at most 4 significant bits, so the dequantised key is a
    bf16 value exactly: no rounding between the format and the bf16 MMA."""
    from mla_decode_attention_gb300 import workloads
    x = torch.randn((64, 512), generator=torch.Generator().manual_seed(6))
    dec = oracle.fp8_v41_tokens_to_f64(workloads.quantize_fp8_v41_tokens(x).numpy())
    assert np.array_equal(oracle.round_to_bf16(dec), dec)


def test_fp8_v41_single_key_returns_the_whole_key_row():
    """V4.1 keys are 512 wide and the value is the whole key (RoPE dims
    included): one key gives out = that key row."""
    r = rng(33)
    keys = oracle.fp8_v41_tokens_to_f64(
        __import__("mla_decode_attention_gb300.workloads", fromlist=["x"]).quantize_fp8_v41_tokens(
            torch.from_numpy(r.standard_normal((1, 512))).float()).numpy())
    out, lse = oracle.attend(r.standard_normal((4, 512)), keys, SCALE)
    assert np.array_equal(out, np.repeat(keys, 4, axis=0))


def test_round_to_bf16_matches_torch_on_fp32_values():
    x = rng(40).standard_normal(50000).astype(np.float32) * np.exp2(rng(41).integers(-20, 20, 50000))
    x = x.astype(np.float32)
    x[:6] = [0.0, 1.0, 1.00390625, 1.01171875, -3.0078125, 2.0 ** -100]  # ties and exact values
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_to_bf16(x.astype(np.float64)), ref)


def test_fp8_keys_are_bf16_rounded_dequantised_values():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(16, 576, generator=g)
    raw = workloads.quantize_fp8_tokens(x).numpy()
    exact = oracle.fp8_tokens_to_f64(raw)
    keys = oracle.fp8_tokens_to_keys(raw)
    assert np.array_equal(keys[:, 512:], exact[:, 512:])
    assert np.array_equal(keys[:, :512], oracle.round_to_bf16(exact[:, :512]))
    assert np.all(np.abs(keys[:, :512] - exact[:, :512]) <= 2.0 ** -8 * np.abs(exact[:, :512]))


def test_fp8_representable_roundtrip_exact():
    """Values already on the e4m3 grid times a power-of-two scale survive."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    x = np.zeros((1, 576))
    x[0, :512] = np.resize(vals, 512)
    for blk in range(4):          # block absmax = 448 -> scale exactly 1
        x[0, blk * 128] = 448.0
    raw = workloads.quantize_fp8_tokens(torch.from_numpy(x).to(torch.float32)).numpy()
    dec = oracle.fp8_tokens_to_f64(raw)
    assert np.array_equal(dec[0, :512], x[0, :512])


# ----------------------------------------------------------- attention core

def test_single_key_returns_its_value_row():
    q = rng(2).standard_normal((5, 576))
    k = rng(3).standard_normal((1, 576))
    out, lse = oracle.attend(q, k, SCALE)
    assert np.array_equal(out, np.repeat(k[:, :512], 5, axis=0))
    assert np.allclose(lse, SCALE * (q @ k[0]), rtol=0, atol=1e-14)


def test_equal_scores_give_mean_of_values():
    keys = rng(4).standard_normal((37, 576))
    out, lse = oracle.attend(np.zeros((3, 576)), keys, SCALE)
    assert np.allclose(out, keys[:, :512].mean(axis=0)[None], rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(37), rtol=0, atol=1e-13)


def test_two_keys_closed_form():
    """Scores chosen through one coordinate; weights from math.exp by hand."""
    q = np.zeros((1, 576)); q[0, 3] = 1.0
    keys = np.zeros((2, 576))
    keys[0, 3], keys[1, 3] = 2.0, -1.5
    keys[0, :3] = [1.0, 2.0, 3.0]
    keys[1, :3] = [-4.0, 0.5, 8.0]
    a, b = SCALE * 2.0, SCALE * -1.5
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    wb = 1.0 - wa
    out, lse = oracle.attend(q, keys, SCALE)
    expect = wa * keys[0, :512] + wb * keys[1, :512]
    assert np.allclose(out[0], expect, rtol=0, atol=1e-14)
    assert abs(lse[0] - math.log(math.exp(a) + math.exp(b))) < 1e-14


def test_rope_columns_score_but_are_not_values():
    """Columns 512..575 enter the score only; the output has 512 columns."""
    q = np.zeros((1, 576)); q[0, 512:] = 1.0
    keys = np.zeros((2, 576))
    keys[0, 512:] = 0.2            # rope dot = 12.8
    keys[1, 512:] = -0.2
    keys[0, :512] = 1.0
    keys[1, :512] = -1.0
    out, lse = oracle.attend(q, keys, 1.0)
    w0 = 1.0 / (1.0 + math.exp(-25.6))
    assert out.shape == (1, 512)
    assert np.allclose(out[0], w0 * 1.0 + (1 - w0) * -1.0, atol=1e-14)
    assert abs(lse[0] - math.log(math.exp(12.8) + math.exp(-12.8))) < 1e-12


def _naive_rows(q_rows, keys, scale):
    """Three-pass softmax attention with plain Python loops (no BLAS)."""
    outs, lses = [], []
    for q in q_rows.tolist():
        s = [scale * sum(a * b for a, b in zip(q, k)) for k in keys.tolist()]
        m = max(s)
        e = [math.exp(v - m) for v in s]
        z = sum(e)
        o = [0.0] * 512
        for w, k in zip(e, keys.tolist()):
            for d in range(512):
                o[d] += w * k[d]
        outs.append([v / z for v in o])
        lses.append(m + math.log(z))
    return np.array(outs), np.array(lses)


def test_brute_force_tiny():
    q = rng(5).standard_normal((3, 576)) * 2
    keys = rng(6).standard_normal((7, 576))
    out, lse = oracle.attend(q, keys, SCALE)
    ref_o, ref_l = _naive_rows(q, keys, SCALE)
    assert np.allclose(out, ref_o, rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_online_recurrence_equals_definition():
    q = rng(7).standard_normal((1, 576)) * 3
    keys = rng(8).standard_normal((300, 576))
    o1, l1 = oracle.attend(q, keys, SCALE)
    o2, l2 = oracle.attend_online(q[0], keys, SCALE)
    assert np.allclose(o1[0], o2, rtol=0, atol=1e-12)
    assert abs(l1[0] - l2) < 1e-12


def test_combine_of_splits_equals_unsplit():
    q = rng(9).standard_normal((4, 576))
    keys = rng(10).standard_normal((250, 576))
    cuts = [0, 0, 17, 130, 250]            # includes an empty split
    parts = [oracle.attend(q, keys[a:b], SCALE) for a, b in zip(cuts[:-1], cuts[1:])]
    o, l = oracle.combine(parts)
    o_ref, l_ref = oracle.attend(q, keys, SCALE)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
    assert np.allclose(l, l_ref, rtol=0, atol=1e-12)


def test_absorption_identity():
    """Per-head attention with expanded K/V equals absorbed MQA on the latent.

    score_h(t) = q_C,h . (W_UK,h c_t) + q_R,h . k_R,t
               = (W_UK,h^T q_C,h) . c_t + q_R,h . k_R,t
    o_h = sum_t p_h(t) W_UV,h c_t = W_UV,h (sum_t p_h(t) c_t)
    """
    r = rng(11)
    H, dh, T = 3, 16, 9
    W_UK = r.standard_normal((H, dh, 512)) / 20
    W_UV = r.standard_normal((H, dh, 512)) / 20
    c = r.standard_normal((T, 512))
    k_R = r.standard_normal((T, 64))
    q_C = r.standard_normal((H, dh))
    q_R = r.standard_normal((H, 64))
    for h in range(H):
        k_full = np.concatenate([c @ W_UK[h].T, k_R], axis=1)          # [T, dh+64]
        v_full = c @ W_UV[h].T                                          # [T, dh]
        s = SCALE * (k_full @ np.concatenate([q_C[h], q_R[h]]))
        p = np.exp(s - s.max()); p /= p.sum()
        o_expanded = p @ v_full
        q_abs = np.concatenate([W_UK[h].T @ q_C[h], q_R[h]])[None]      # [1, 576]
        keys = np.concatenate([c, k_R], axis=1)                         # [T, 576]
        lat, lse = oracle.attend(q_abs, keys, SCALE)
        o_absorbed = W_UV[h] @ lat[0]
        assert np.allclose(o_absorbed, o_expanded, rtol=1e-12, atol=1e-13)
        assert abs(lse[0] - (s.max() + math.log(np.exp(s - s.max()).sum()))) < 1e-12


# ------------------------------------------------------------------ gathers

def _id_cache(n_pages):
    """Cache whose column 0 holds the flat physical row id (page*64 + slot)."""
    kv = np.zeros((n_pages, 64, 576))
    kv[:, :, 0] = np.arange(n_pages * 64).reshape(n_pages, 64)
    return kv


def test_paged_gather_follows_block_table():
    perm = rng(12).permutation(16)
    bt = perm[:10].reshape(2, 5)
    kv = _id_cache(16)
    keys = oracle.paged_keys(kv, bt[1], 300)
    t = np.arange(300)
    assert np.array_equal(keys[:, 0], bt[1][t // 64] * 64 + t % 64)


def test_dense_single_token_rows_copy_their_page_row():
    """seqlen 1: out is the V row of block_table[b, 0] slot 0, bit for bit."""
    kv = rng(13).standard_normal((8, 64, 576))
    bt = np.array([[5, 1], [2, 7], [0, 3]])
    q = rng(14).standard_normal((3, 1, 4, 576))
    out, lse = oracle.dense_decode(q, kv, bt, np.array([1, 1, 1]), SCALE)
    for b in range(3):
        assert np.array_equal(out[b, 0], np.repeat(kv[bt[b, 0], 0, :512][None], 4, axis=0))


def test_causal_end_alignment():
    """s_q = 2 causal: token j sees L - 2 + j + 1 keys (bottom-right)."""
    kv = rng(15).standard_normal((12, 64, 576))
    bt = rng(16).permutation(12).reshape(2, 6)
    L = np.array([300, 129])
    q = rng(17).standard_normal((2, 2, 3, 576))
    out, lse = oracle.dense_decode(q, kv, bt, L, SCALE, causal=True)
    for b in range(2):
        for j in range(2):
            o1, l1 = oracle.dense_decode(q[b:b + 1, j:j + 1], kv, bt[b:b + 1],
                                         np.array([L[b] - 1 + j]), SCALE)
            assert np.array_equal(out[b, j], o1[0, 0])
            assert np.array_equal(lse[b, :, j], l1[0, :, 0])
    # and the two tokens really differ by the last key
    assert not np.allclose(out[0, 0], out[0, 1])


def test_sparse_index_order_invariance():
    pool = rng(18).standard_normal((500, 576))
    idx = rng(19).permutation(500)[:64].reshape(1, 1, 64)
    idx[0, 0, [5, 40]] = -1
    q = rng(20).standard_normal((1, 1, 8, 576))
    o1, l1 = oracle.sparse_decode(q, pool, idx, SCALE)
    for s in range(3):
        perm = rng(21 + s).permutation(64)
        o2, l2 = oracle.sparse_decode(q, pool, idx[:, :, perm], SCALE)
        assert np.allclose(o1, o2, rtol=0, atol=1e-12)
        assert np.allclose(l1, l2, rtol=0, atol=1e-12)


def test_sparse_invalid_and_out_of_range_are_skipped():
    pool = rng(22).standard_normal((100, 576))
    q = rng(23).standard_normal((1, 1, 2, 576))
    good = np.array([3, 50, 99, 0, 17])
    idx = np.array([3, -1, 50, 100, 99, 0, -7, 17, 1 << 30]).reshape(1, 1, -1)
    o1, l1 = oracle.sparse_decode(q, pool, idx, SCALE)
    o2, l2 = oracle.sparse_decode(q, pool, good.reshape(1, 1, -1), SCALE)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_prefill_brute_force_and_layout():
    """Sparse prefill on a tiny case against a brute-force softmax written
    here: token i's output is the softmax over the rows its list names (each
    named slot counted once, -1 skipped), out is [s_q, h, 512] and lse
    [s_q, h]."""
    pool = rng(60).standard_normal((7, 576))
    idx = np.array([[0, 3, -1], [6, 6, 2], [5, -1, -1], [-1, -1, -1]])
    q = rng(61).standard_normal((4, 3, 576))
    out, lse = oracle.sparse_prefill(q, pool.reshape(7, 1, 576), idx.reshape(4, 1, 3), SCALE)
    assert out.shape == (4, 3, 512) and lse.shape == (4, 3)
    for i in range(4):
        rows = [int(r) for r in idx[i] if r >= 0]
        for hh in range(3):
            if not rows:
                assert np.all(out[i, hh] == 0.0) and np.isneginf(lse[i, hh])
                continue
            sc = np.array([SCALE * float(np.dot(q[i, hh], pool[r])) for r in rows])
            w = np.exp(sc - sc.max())
            ref_out = sum(w[k] * pool[rows[k], :512] for k in range(len(rows))) / w.sum()
            ref_lse = sc.max() + math.log(w.sum())
            assert np.allclose(out[i, hh], ref_out, rtol=1e-12, atol=1e-12)
            assert abs(lse[i, hh] - ref_lse) < 1e-12
    # a token naming exactly one row returns that row's V part exactly
    assert np.array_equal(out[2, 1], pool[5, :512])


def test_sparse_prefill_topk_length_and_sink_follow_decode_rules():
    pool = rng(62).standard_normal((40, 576))
    idx = rng(63).permutation(40)[:30].reshape(3, 10)
    q = rng(64).standard_normal((3, 2, 576))
    tl = np.array([10, 4, 0])
    sink = np.array([0.5, -1.0])
    out, lse = oracle.sparse_prefill(q, pool, idx, SCALE, attn_sink=sink, topk_length=tl)
    for i in range(3):
        cut = idx[i].copy()
        cut[tl[i]:] = -1
        o1, l1 = oracle.sparse_prefill(q[i:i + 1], pool, cut.reshape(1, 10), SCALE)
        f = oracle.sink_factor(l1[0], sink)
        assert np.allclose(out[i], o1[0] * f[:, None], rtol=0, atol=1e-12)
        assert np.allclose(lse[i], l1[0], rtol=0, atol=1e-12, equal_nan=True)


def test_dense_equals_sparse_over_all_rows_of_the_request():
    kv = rng(24).standard_normal((10, 64, 576))
    bt = rng(25).permutation(10).reshape(2, 5)
    L = np.array([260, 70])
    q = rng(26).standard_normal((2, 1, 4, 576))
    od, ld = oracle.dense_decode(q, kv, bt, L, SCALE)
    pool = kv.reshape(-1, 576)
    for b in range(2):
        t = np.arange(L[b])
        idx = (bt[b][t // 64] * 64 + t % 64).reshape(1, 1, -1)
        os_, ls_ = oracle.sparse_decode(q[b:b + 1], pool, idx, SCALE)
        assert np.allclose(os_[0], od[b], rtol=0, atol=1e-12)
        assert np.allclose(ls_[0], ld[b], rtol=0, atol=1e-12)


def test_empty_key_sets():
    q = rng(27).standard_normal((2, 2, 3, 576))
    kv = rng(28).standard_normal((4, 64, 576))
    bt = np.array([[0, 1], [2, 3]])
    out, lse = oracle.dense_decode(q, kv, bt, np.array([0, 1]), SCALE)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(out[1, 0] == 0) and np.all(np.isneginf(lse[1, :, 0]))   # L - s_q + 1 + 0 = 0
    assert np.array_equal(out[1, 1], np.repeat(kv[2, 0, :512][None], 3, axis=0))
    idx = -np.ones((1, 1, 8), dtype=np.int64)
    o, l = oracle.sparse_decode(q[:1, :1], kv.reshape(-1, 576), idx, SCALE)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_bf16_bits_input_equals_float_input():
    g = torch.Generator().manual_seed(3)
    qt = torch.randn(1, 1, 4, 576, generator=g).to(torch.bfloat16)
    kt = torch.randn(3, 64, 576, generator=g).to(torch.bfloat16)
    bt = np.array([[2, 0, 1]])
    a = oracle.dense_decode(bf16_np(qt), bf16_np(kt), bt, np.array([150]), SCALE)
    b = oracle.dense_decode(qt.double().numpy(), kt.double().numpy(), bt, np.array([150]), SCALE)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------ numbers on the pages

def test_page_numbers_dimensions_and_token_bytes():
    assert GOLDEN["d_qk"]["value"] == oracle.D_QK == workloads.D_QK == 512 + 64
    assert GOLDEN["d_v"]["value"] == oracle.D_V == workloads.D_V
    assert GOLDEN["bf16_token_bytes"]["value"] == roofline.BF16_TOKEN_BYTES
    t = GOLDEN["kv_bytes_128k_request"]["terms"]
    n = t["d"] * t["bytes"] * t["layers"] * t["tokens"]
    assert n == GOLDEN["kv_bytes_128k_request"]["value"]
    assert round(n / 2 ** 30, 2) == GOLDEN["kv_bytes_128k_request"]["gib"]


def test_page_numbers_cost_model():
    c = GOLDEN["ai_dsv3_decode"]["config"]
    fl = roofline.mla_analysis_flops(c["b"], c["h"], c["s"], c["t"], c["k"], c["p"])
    by = roofline.mla_analysis_bytes(c["b"], c["h"], c["s"], c["t"], c["k"], c["p"], c["w"])
    assert round(fl / by) == GOLDEN["ai_dsv3_decode"]["value"]
    # our accounting adds LSE, page-table and length words: still ~228
    f2, b2, kv = roofline.dense_counts([c["t"]] * c["b"], 1, c["h"])
    assert f2 == fl
    assert round(f2 / b2) == GOLDEN["ai_dsv3_decode"]["value"]
    assert roofline.FLOP_PER_PAIR == GOLDEN["flops_per_token_per_row"]["value"]
    g = GOLDEN["mma_cycles_per_token_64_heads_h800"]
    assert round(64 * (576 + 512) * 2 / g["flop_per_clk_per_sm"]) == g["value"]


# ------------------------------------------------------- the parity checker

def test_parity_checker_accepts_the_bf16_floor_and_rejects_real_errors():
    """The ideal bf16 output passes; a 1% gain error or a dropped key fails."""
    from tests._util import assert_parity
    r = rng(30)
    q = r.standard_normal((16, 576))
    keys = r.standard_normal((40, 576))
    o, l = oracle.attend(q, keys, SCALE)
    o[3, 7] = 1.9                      # an element far above the RMS
    ideal = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
    assert_parity(ideal, o, l, l, "ideal bf16")
    with pytest.raises(AssertionError):
        assert_parity(ideal * 1.01, o, l, l, "gain")
    o2, l2 = oracle.attend(q, keys[1:], SCALE)
    with pytest.raises(AssertionError):
        assert_parity(torch.from_numpy(o2).to(torch.bfloat16).double().numpy(), o, l2, l, "drop")
    with pytest.raises(AssertionError):
        assert_parity(ideal, o, l + 2e-3, l, "lse")


def test_per_token_parity_checker_scales_with_each_token():
    """Two tokens of very different output size (4 keys vs 4000 keys): the
    ideal bf16 output passes per token; a 1% gain on the small-valued token
    alone, or a dropped key of the short token, fails."""
    from tests._util import assert_parity_per_token
    r = rng(31)
    outs, lses = [], []
    for n in (4, 4000):
        q = r.standard_normal((8, 576))
        keys = r.standard_normal((n, 576))
        o, l = oracle.attend(q, keys, SCALE)
        outs.append(o)
        lses.append(l)
    o = np.stack(outs)[:, None]                 # [2, 1, 8, 512]
    l = np.stack(lses)[:, :, None]              # [2, 8, 1]
    ideal = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
    assert_parity_per_token(ideal, o, l, l, "ideal bf16")
    bad = ideal.copy()
    bad[1] *= 1.01
    with pytest.raises(AssertionError):
        assert_parity_per_token(bad, o, l, l, "gain on the long token")
    q = r.standard_normal((8, 576))
    keys = r.standard_normal((4, 576))
    o0, l0 = oracle.attend(q, keys, SCALE)
    o1, l1 = oracle.attend(q, keys[1:], SCALE)
    o[0, 0], l[0, :, 0] = o0, l0
    drop = o.copy()
    drop[0, 0] = o1
    with pytest.raises(AssertionError):
        assert_parity_per_token(torch.from_numpy(drop).to(torch.bfloat16).double().numpy(), o, l, l, "drop")


# ------------------------------------------- attention sink and topk length

def test_attention_sink_is_a_zero_valued_key_with_the_sink_as_its_score():
    """exp(lse) / (exp(lse) + exp(sink)) scaling equals attending over the
    keys plus one extra key whose score is the sink and whose value is 0
    (brute force through the plain definition, one head at a time)."""
    r = rng(41)
    pool = r.standard_normal((50, 576))
    idx = r.permutation(50)[:12].reshape(1, 1, 12).astype(np.int64)
    q = r.standard_normal((1, 1, 3, 576))
    sink = np.array([-1.5, 0.4, 3.0])
    out, lse = oracle.sparse_decode(q, pool, idx, SCALE, attn_sink=sink)
    base, base_lse = oracle.sparse_decode(q, pool, idx, SCALE)
    assert np.array_equal(lse, base_lse)                    # lse is not changed by the sink
    for h in range(3):
        k_sink = np.zeros(576)
        c = 512 + int(np.argmax(np.abs(q[0, 0, h, 512:])))  # a RoPE column with q != 0
        k_sink[c] = sink[h] / (SCALE * q[0, 0, h, c])       # score = sink, value = 0
        keys = np.vstack([pool[idx[0, 0]], k_sink])
        o, _ = oracle.attend(q[0, 0, h:h + 1], keys, SCALE)
        np.testing.assert_allclose(out[0, 0, h], o[0], rtol=1e-12, atol=1e-14)
    # special cases: sink = -inf changes nothing, sink = lse halves the output
    o1, _ = oracle.sparse_decode(q, pool, idx, SCALE, attn_sink=np.full(3, -np.inf))
    assert np.array_equal(o1, base)
    o2, _ = oracle.sparse_decode(q, pool, idx, SCALE, attn_sink=base_lse[0, :, 0])
    np.testing.assert_allclose(o2, 0.5 * base, rtol=1e-12, atol=0)


def test_topk_length_equals_masking_the_later_slots():
    """Using the first n index slots is the same as marking the rest -1;
    n = 0 gives an empty key set, n > topk is clamped to topk."""
    r = rng(42)
    pool = r.standard_normal((80, 576))
    idx = r.permutation(80)[:40].reshape(2, 2, 10).astype(np.int64)
    q = r.standard_normal((2, 2, 4, 576))
    lengths = np.array([[0, 3], [10, 25]])
    out, lse = oracle.sparse_decode(q, pool, idx, SCALE, topk_length=lengths)
    masked = idx.copy()
    for b in range(2):
        for j in range(2):
            masked[b, j, min(lengths[b, j], 10):] = -1
    ref, ref_l = oracle.sparse_decode(q, pool, masked, SCALE)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_l)
    assert np.all(out[0, 0] == 0) and np.all(np.isneginf(lse[0, :, 0]))
