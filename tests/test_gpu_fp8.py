"""GPU parity of decode over the 656-byte FP8 latent cache against the fp64 oracle.

The oracle's key is what the pages' FP8 kernel multiplies: each latent value
dequantised to bf16, bf16(e4m3 * fp32 scale) (the exact product rounded once
to nearest-even), and the stored bf16 RoPE values.  The kernel converts in
shared memory the same way before its bf16 MMAs, so the bf16 tolerances of
the dense tests apply.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_gb300 import binding, workloads
from tests._util import assert_parity, assert_parity_per_token, bf16_half_ulp, bf16_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def library():
    from mla_decode_attention_gb300 import build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def run_fp8(inp, num_sm_parts=None, causal=True):
    q = inp["q"].to(DEV)
    kv = inp["kv_cache"].to(DEV)
    bt = inp["block_table"].to(DEV)
    sl = inp["cache_seqlens"].to(DEV)
    b, s_q, h, _ = q.shape
    buf = binding.DecodeBuffers(b, s_q, h, DEV, num_sm_parts)
    binding.mla_get_metadata(sl, b, s_q, causal, 0, buf.num_sm_parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_FP8_656, bt, sl, inp["softmax_scale"], causal,
                       buf.metadata, buf.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    return buf.out.float().cpu().numpy(), buf.lse.cpu().numpy(), int(buf.err.item())


def oracle_fp8(inp, causal=True, rows=None):
    return oracle.fp8_dense_decode(bf16_np(inp["q"]), inp["kv_cache"].numpy(),
                                   inp["block_table"].numpy(), inp["cache_seqlens"].numpy(),
                                   inp["softmax_scale"], causal, rows)


def fp8_case(seed, b, s_q, h, seqlens, extra_pages=0):
    w = workloads.Workload("f8", "fp8", b=b, s_q=s_q, h=h, seqlens=tuple(seqlens),
                           extra_pages=extra_pages, seed=seed)
    return workloads.make_inputs(w)


def test_fp8_small_parity():
    inp = fp8_case(51, 2, 1, 16, (200, 333), extra_pages=6)
    out, lse, err = run_fp8(inp)
    ref_o, ref_l = oracle_fp8(inp)
    assert_parity(out, ref_o, lse, ref_l, "fp8 small")
    assert err == 0


@pytest.mark.parametrize("parts", [None, 5])
def test_fp8_h128_spec_ragged(parts):
    inp = fp8_case(52, 4, 2, 128, (2, 129, 1000, 2500))
    out, lse, err = run_fp8(inp, parts)
    ref_o, ref_l = oracle_fp8(inp)
    assert_parity(out, ref_o, lse, ref_l, f"fp8 spec parts={parts}")


@pytest.mark.parametrize("h", [64, 128])
def test_fp8_single_key_rows_are_the_dequantised_row(h):
    # one visible key: the output row is that key's dequantised latent part
    # (h = 128: the two head-block CTAs of a cluster each convert half of the
    # latent chunks and copy them to the other)
    inp = fp8_case(53, 4, 1, h, (1, 1, 1, 1), extra_pages=8)
    out, lse, err = run_fp8(inp)
    dec = oracle.fp8_tokens_to_f64(inp["kv_cache"].numpy())
    bt = inp["block_table"].numpy()
    for b in range(4):
        row = dec[bt[b, 0], 0, :512]
        # one rounding of e4m3*scale to bf16 (the f32 product may round once before)
        assert np.all(np.abs(out[b, 0] - row[None]) <= bf16_half_ulp(row)[None] * 1.01 + 1e-30)


def test_full_size_fp8_all_rows():
    """b=64, h=128, t=8192 over the 656-byte cache: every request and head."""
    w = workloads.WORKLOADS["fp8"]
    inp = workloads.make_inputs(w)
    out, lse, err = run_fp8(inp)
    ref_o, ref_l = oracle_fp8(inp)
    st = assert_parity_per_token(out, ref_o, lse, ref_l, "fp8")
    print("fp8 parity:", st)
    assert err == 0


def test_combine_after_decodes_of_two_kernels_on_one_metadata():
    """One metadata buffer shared by a bf16 decode (two-SM kernel, which
    walks the whole-sequence schedule here) and an FP8 decode (one-SM kernel,
    which keeps the balanced split here), each with its own workspace; the
    split entry points run back to back, then each workspace is combined.
    The combine follows the schedule recorded in its own workspace, so both
    results match their oracle (the metadata is never written)."""
    b, h, parts = 4, 128, 76
    w = workloads.Workload("share", "dense", b=b, s_q=1, h=h, seqlens=(1000,) * b, seed=27)
    dense = workloads.make_inputs(w)
    fp8 = fp8_case(28, b, 1, h, (1000,) * b)
    sl = dense["cache_seqlens"].to(DEV)
    meta = binding.DecodeBuffers(b, 1, h, DEV, parts).metadata
    binding.mla_get_metadata(sl, b, 1, True, 0, parts, meta)
    before = meta.clone()
    bufs = [binding.DecodeBuffers(b, 1, h, DEV, parts) for _ in range(2)]
    binding.mla_decode_splitkv(dense["q"].to(DEV), dense["kv_cache"].to(DEV), binding.MLA_KV_BF16,
                               dense["block_table"].to(DEV), sl, dense["softmax_scale"], True, meta, parts,
                               bufs[0].workspace, bufs[0].out, bufs[0].lse, bufs[0].err)
    binding.mla_decode_splitkv(fp8["q"].to(DEV), fp8["kv_cache"].to(DEV), binding.MLA_KV_FP8_656,
                               fp8["block_table"].to(DEV), fp8["cache_seqlens"].to(DEV), fp8["softmax_scale"],
                               True, meta, parts, bufs[1].workspace, bufs[1].out, bufs[1].lse, bufs[1].err)
    for bf in bufs:
        binding.mla_combine(meta, b, 1, h, parts, bf.workspace, bf.out, bf.lse)
    torch.cuda.synchronize()
    assert torch.equal(meta, before)
    rows = (b * 1 + parts) * h
    walked = [int(bf.workspace[rows * 513:].view(torch.int32)[0].item()) for bf in bufs]
    assert walked == [1, 0]
    ref = [oracle.dense_decode(bf16_np(dense["q"]), bf16_np(dense["kv_cache"]), dense["block_table"].numpy(),
                               dense["cache_seqlens"].numpy(), dense["softmax_scale"]),
           oracle_fp8(fp8)]
    for bf, (ro, rl), name in zip(bufs, ref, ("bf16", "fp8")):
        assert int(bf.err.item()) == 0
        assert_parity(bf.out.float().cpu().numpy(), ro, bf.lse.cpu().numpy(), rl, name)


# ------------------------------------------------ V4.1 cache (528 bytes per token)

def v41_case(seed, b, s_q, h, seqlens, extra_pages=0):
    w = workloads.Workload("v41", "fp8_v41", b=b, s_q=s_q, h=h, seqlens=tuple(seqlens),
                           extra_pages=extra_pages, seed=seed)
    return workloads.make_inputs(w)


def run_v41(inp, num_sm_parts=None, causal=True):
    q = inp["q"].to(DEV)
    kv = inp["kv_cache"].to(DEV)
    bt = inp["block_table"].to(DEV)
    sl = inp["cache_seqlens"].to(DEV)
    b, s_q, h, _ = q.shape
    buf = binding.DecodeBuffers(b, s_q, h, DEV, num_sm_parts)
    binding.mla_get_metadata(sl, b, s_q, causal, 0, buf.num_sm_parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_FP8_528, bt, sl, inp["softmax_scale"], causal,
                       buf.metadata, buf.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    return buf.out.float().cpu().numpy(), buf.lse.cpu().numpy(), int(buf.err.item())


def oracle_v41(inp, causal=True, rows=None):
    return oracle.fp8_v41_dense_decode(bf16_np(inp["q"]), inp["kv_cache"].numpy(),
                                       inp["block_table"].numpy(), inp["cache_seqlens"].numpy(),
                                       inp["softmax_scale"], causal, rows)


def test_v41_small_parity():
    inp = v41_case(61, 2, 1, 16, (200, 333), extra_pages=6)
    out, lse, err = run_v41(inp)
    ref_o, ref_l = oracle_v41(inp)
    assert_parity(out, ref_o, lse, ref_l, "v41 small")
    assert err == 0


@pytest.mark.parametrize("h,parts", [(64, None), (128, None), (128, 5), (32, 3)])
def test_v41_spec_ragged(h, parts):
    inp = v41_case(62 + h, 4, 2, h, (2, 129, 1000, 2500))
    out, lse, err = run_v41(inp, parts)
    ref_o, ref_l = oracle_v41(inp)
    assert_parity(out, ref_o, lse, ref_l, f"v41 h={h} parts={parts}")
    assert err == 0


@pytest.mark.parametrize("h", [64, 128])
def test_v41_single_key_rows_are_the_exact_key_row(h):
    """One visible key: the output row is that key's whole 512-wide dequantised
    row (RoPE dimensions included), bit for bit: e4m3 times a power of two is
    a bf16 value, so nothing rounds."""
    inp = v41_case(63, 4, 1, h, (1, 1, 1, 1), extra_pages=8)
    out, lse, err = run_v41(inp)
    dec = oracle.fp8_v41_tokens_to_f64(inp["kv_cache"].numpy())
    bt = inp["block_table"].numpy()
    for b in range(4):
        row = dec[bt[b, 0], 0]
        assert np.array_equal(out[b, 0], np.repeat(row[None], h, axis=0))
    assert err == 0


def test_v41_full_size_all_rows():
    """b=64, h=128, every request 8192 tokens of the 528-byte cache: every
    request and head compared with the oracle."""
    w = workloads.Workload("v41_full", "fp8_v41", b=64, s_q=1, h=128, seqlens=(8192,) * 64, seed=64)
    inp = workloads.make_inputs(w)
    out, lse, err = run_v41(inp)
    ref_o, ref_l = oracle_v41(inp)
    st = assert_parity_per_token(out, ref_o, lse, ref_l, "v41")
    print("v41 parity:", st)
    assert err == 0
