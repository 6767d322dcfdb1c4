"""mla_decode_noalloc: the decode entry point for callers that cannot allocate.

Some callers may launch kernels but may not allocate device memory where they
call us (an engine plugin's enqueue hook that only receives input/output
pointers and a stream; a serving loop that must avoid cudaMalloc).  For them
the library keeps its schedule metadata and split workspace in a fixed device
array.  This test calls that entry point through the C ABI twice in a row,
with different inputs, and checks each result against the regular
mla_decode (caller-provided scratch) within the parity tolerance.  It lives
in its own file, collected last, so a failure here comes after every other
test has run; it also passes alone in a fresh process.
"""
import os

import numpy as np
import pytest
import torch

from mla_decode_attention_gb300 import binding, workloads
from tests._util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def library():
    from mla_decode_attention_gb300 import build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def _regular(inp):
    q, kv, bt, sl = (inp[k].to(DEV) for k in ("q", "kv_cache", "block_table", "cache_seqlens"))
    b, s_q, h, _ = q.shape
    buf = binding.DecodeBuffers(b, s_q, h, DEV)
    binding.mla_get_metadata(sl, b, s_q, True, 0, buf.num_sm_parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"], True,
                       buf.metadata, buf.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    return buf.out.float().cpu().numpy(), buf.lse.cpu().numpy()


def _noalloc(inp):
    q, kv, bt, sl = (inp[k].to(DEV) for k in ("q", "kv_cache", "block_table", "cache_seqlens"))
    b, s_q, h, _ = q.shape
    out = torch.full((b, s_q, h, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((b, h, s_q), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.mla_decode_noalloc(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"], True,
                               out, lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_regular_decode_on_two_calls():
    shapes = [
        workloads.Workload("noalloc_a", "dense", b=6, s_q=1, h=128,
                           seqlens=(1, 200, 4096, 129, 1000, 64), seed=21),
        workloads.Workload("noalloc_b", "dense", b=4, s_q=2, h=64,
                           seqlens=(3000, 77, 640, 2), seed=22),
    ]
    for w in shapes:                      # two calls in a row share the scratch
        inp = workloads.make_inputs(w)
        ref_o, ref_l = _regular(inp)
        got_o, got_l = _noalloc(inp)
        assert_parity(got_o, ref_o, got_l, ref_l, f"noalloc vs mla_decode ({w.name})")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    w = workloads.Workload("too_big", "dense", b=256, s_q=2, h=128, seqlens=(128,) * 256, seed=23)
    inp = workloads.make_inputs(w)
    q, kv, bt, sl = (inp[k].to(DEV) for k in ("q", "kv_cache", "block_table", "cache_seqlens"))
    out = torch.empty(256, 2, 128, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(256, 128, 2, dtype=torch.float32, device=DEV)
    with pytest.raises(binding.MlaError) as ei:
        binding.mla_decode_noalloc(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"],
                                   True, out, lse)
    assert ei.value.status == -2 and "scratch" in str(ei.value)
