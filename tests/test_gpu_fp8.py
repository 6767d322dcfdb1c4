"""GPU parity of decode over the 656-byte FP8 latent cache against the fp64 oracle.

The oracle decodes each token exactly (e4m3 * fp32 scale, bf16 RoPE); the
kernel dequantises to bf16 in shared memory (one rounding) before the bf16
MMAs, so the same bf16 tolerances apply.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_gb300 import binding, workloads
from tests._util import assert_parity, bf16_half_ulp, bf16_np

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


def test_full_size_fp8_sampled_rows():
    w = workloads.WORKLOADS["fp8"]
    inp = workloads.make_inputs(w)
    out, lse, err = run_fp8(inp)
    rows = [(0, 0), (21, 0), (42, 0), (63, 0)]
    ref_o, ref_l = oracle_fp8(inp, rows=rows)
    for b, j in rows:
        assert_parity(out[b, j], ref_o[b, j], lse[b, :, j], ref_l[b, :, j], f"fp8 row {b}")
    assert err == 0 and np.all(np.isfinite(out))
