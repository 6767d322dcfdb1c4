"""GPU parity of the dense paged decode against the fp64 oracle (through the C ABI).

Tolerances: bf16 out rel-L2 <= 3e-3 and max-abs <= 2e-2 * RMS(out_ref),
LSE abs error <= 1e-3; gathers (single-key rows) bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_gb300 import binding, workloads
from tests._util import assert_parity, bf16_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def library():
    from mla_decode_attention_gb300 import build
    import os
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def run_dense(inp, num_sm_parts=None, causal=True, out_pad=0):
    q = inp["q"].to(DEV)
    kv = inp["kv_cache"].to(DEV)
    bt = inp["block_table"].to(DEV)
    sl = inp["cache_seqlens"].to(DEV)
    b, s_q, h, _ = q.shape
    buf = binding.DecodeBuffers(b, s_q, h, DEV, num_sm_parts)
    out = buf.out
    if out_pad:
        big = torch.full((b * s_q * h * 512 + out_pad,), 7.0, dtype=torch.bfloat16, device=DEV)
        out = big[:b * s_q * h * 512].view(b, s_q, h, 512)
    binding.mla_get_metadata(sl, b, s_q, causal, 0, buf.num_sm_parts, buf.metadata)
    fmt = binding.MLA_KV_BF16 if kv.dtype == torch.bfloat16 else binding.MLA_KV_FP8_656
    binding.mla_decode(q, kv, fmt, bt, sl, inp["softmax_scale"], causal, buf.metadata,
                       buf.num_sm_parts, buf.workspace, out, buf.lse, buf.err)
    torch.cuda.synchronize()
    res = dict(out=out.float().cpu().numpy(), lse=buf.lse.cpu().numpy(),
               err=int(buf.err.item()), meta=buf.metadata.cpu().numpy())
    if out_pad:
        res["pad"] = big[b * s_q * h * 512:].float().cpu().numpy()
    return res


def oracle_dense(inp, causal=True, rows=None):
    kv = inp["kv_cache"]
    kv_np = bf16_np(kv) if kv.dtype == torch.bfloat16 else kv.numpy()
    return oracle.dense_decode(bf16_np(inp["q"]), kv_np, inp["block_table"].numpy(),
                               inp["cache_seqlens"].numpy(), inp["softmax_scale"], causal, rows)


def test_tiny_config_parity():
    inp = workloads.make_inputs(workloads.WORKLOADS["tiny"])
    res = run_dense(inp, out_pad=4096)
    ref_o, ref_l = oracle_dense(inp)
    assert_parity(res["out"], ref_o, res["lse"], ref_l, "tiny")
    assert res["err"] == 0
    assert np.all(res["pad"] == 7.0), "write past the end of out"


@pytest.mark.parametrize("parts", [1, 7, 152])
def test_schedule_invariance(parts):
    inp = workloads.make_inputs(workloads.WORKLOADS["tiny"])
    res = run_dense(inp, num_sm_parts=parts)
    ref_o, ref_l = oracle_dense(inp)
    assert_parity(res["out"], ref_o, res["lse"], ref_l, f"parts={parts}")


def test_ragged_lengths_h128():
    w = workloads.Workload("ragged", "dense", b=8, s_q=1, h=128,
                           seqlens=(1, 63, 64, 65, 127, 128, 129, 1000), extra_pages=3, seed=11)
    inp = workloads.make_inputs(w)
    for parts in (None, 3):
        res = run_dense(inp, num_sm_parts=parts)
        ref_o, ref_l = oracle_dense(inp)
        assert_parity(res["out"], ref_o, res["lse"], ref_l, f"ragged parts={parts}")


@pytest.mark.parametrize("h", [32, 48, 64])
def test_head_counts(h):
    w = workloads.Workload("heads", "dense", b=3, s_q=1, h=h, seqlens=(300, 5, 777), seed=12)
    inp = workloads.make_inputs(w)
    res = run_dense(inp)
    ref_o, ref_l = oracle_dense(inp)
    assert_parity(res["out"], ref_o, res["lse"], ref_l, f"h={h}")


def test_spec_decode_causal_s_q2():
    w = workloads.Workload("spec_small", "dense", b=4, s_q=2, h=128,
                           seqlens=(2, 130, 1025, 3000), seed=13)
    inp = workloads.make_inputs(w)
    res = run_dense(inp, causal=True)
    ref_o, ref_l = oracle_dense(inp, causal=True)
    assert_parity(res["out"], ref_o, res["lse"], ref_l, "spec causal")


def test_non_causal_s_q2():
    w = workloads.Workload("spec_nc", "dense", b=2, s_q=2, h=64, seqlens=(200, 129), seed=14,
                           causal=False)
    inp = workloads.make_inputs(w)
    res = run_dense(inp, causal=False)
    ref_o, ref_l = oracle_dense(inp, causal=False)
    assert_parity(res["out"], ref_o, res["lse"], ref_l, "non-causal")


def test_single_key_rows_are_exact_copies():
    """seqlen 1: out must equal the bf16 V row of page block_table[b, 0], bit for bit."""
    w = workloads.Workload("one", "dense", b=5, s_q=1, h=128, seqlens=(1,) * 5, extra_pages=20,
                           seed=15)
    inp = workloads.make_inputs(w)
    res = run_dense(inp)
    kv = inp["kv_cache"].float().numpy()
    bt = inp["block_table"].numpy()
    for b in range(5):
        row = kv[bt[b, 0], 0, :512]
        assert np.array_equal(res["out"][b, 0], np.repeat(row[None], 128, axis=0))


def test_empty_sequences():
    w = workloads.Workload("empty", "dense", b=3, s_q=2, h=16, seqlens=(0, 1, 70), seed=16)
    inp = workloads.make_inputs(w)
    res = run_dense(inp)
    ref_o, ref_l = oracle_dense(inp)
    assert np.all(res["out"][0] == 0) and np.all(np.isneginf(res["lse"][0]))
    assert np.all(res["out"][1, 0] == 0) and np.all(np.isneginf(res["lse"][1, :, 0]))
    assert_parity(res["out"][2], ref_o[2], res["lse"][2], ref_l[2], "empty/nonempty")


def test_bad_page_ids_are_flagged_not_faulted():
    w = workloads.Workload("badpage", "dense", b=2, s_q=1, h=16, seqlens=(100, 200), seed=17)
    inp = workloads.make_inputs(w)
    inp["block_table"][1, 1] = 10 ** 6      # past the cache
    inp["block_table"][0, 0] = -5
    res = run_dense(inp)
    assert res["err"] & binding.MLA_DEVERR_BAD_PAGE
    assert np.all(np.isfinite(res["out"]))


def test_repeat_calls_are_deterministic():
    inp = workloads.make_inputs(workloads.scaled(workloads.WORKLOADS["dense_v3"], b=4,
                                                 seqlens=(4096, 100, 2000, 333)))
    a = run_dense(inp)
    b = run_dense(inp)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


@pytest.mark.parametrize("h,parts,walked", [(128, 76, 1), (128, 3, 0), (64, 76, 0), (64, 4, 1)])
def test_kernels_record_the_schedule_they_walk(h, parts, walked):
    """Four requests of 1000 keys (8 tiles, cost 10).  Schedule B (one whole
    sequence per part) exists when parts >= 4.  With 76 parts A's balanced
    cost is 1: the two-SM kernel (h = 128, split penalty 11) takes B, the
    one-SM kernel (penalty 4) keeps A; with 4 parts A costs 10 as well and
    the one-SM kernel takes B."""
    w = workloads.Workload("choice", "dense", b=4, s_q=1, h=h, seqlens=(1000,) * 4, seed=21)
    inp = workloads.make_inputs(w)
    q, kv = inp["q"].to(DEV), inp["kv_cache"].to(DEV)
    bt, sl = inp["block_table"].to(DEV), inp["cache_seqlens"].to(DEV)
    buf = binding.DecodeBuffers(4, 1, h, DEV, parts)
    binding.mla_get_metadata(sl, 4, 1, True, 0, parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"], True, buf.metadata,
                       parts, buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    assert int(buf.metadata[12].item()) == walked
    ref_o, ref_l = oracle_dense(inp)
    assert_parity(buf.out.float().cpu().numpy(), ref_o, buf.lse.cpu().numpy(), ref_l, f"h={h} parts={parts}")


@pytest.mark.parametrize("batch", [70, 2100])  # the 128- and the 1024-thread schedule kernel
def test_device_metadata_matches_host_mirror(batch):
    rng = np.random.default_rng(5)
    sl = rng.integers(0, 9000, size=batch).astype(np.int32)
    for s_q, causal, parts in ((1, True, 76), (2, True, 152), (3, False, 5), (1, True, 4096)):
        n = binding.mla_metadata_size(batch, s_q, parts) // 4
        meta = torch.zeros(n, dtype=torch.int32, device=DEV)
        binding.mla_get_metadata(torch.from_numpy(sl).to(DEV), batch, s_q, causal, 0, parts, meta)
        torch.cuda.synchronize()
        host = binding.mla_get_metadata_host(sl, batch, s_q, causal, 0, parts)
        assert np.array_equal(meta.cpu().numpy(), host)


def test_full_size_dense_v3_sampled_rows():
    """b=64, h=128, t=4096 in the bench's launch configuration; 6 requests checked."""
    w = workloads.WORKLOADS["dense_v3"]
    inp = workloads.make_inputs(w)
    res = run_dense(inp)
    rows = [(0, 0), (1, 0), (17, 0), (31, 0), (50, 0), (63, 0)]
    ref_o, ref_l = oracle_dense(inp, rows=rows)
    for b, j in rows:
        assert_parity(res["out"][b, j], ref_o[b, j], res["lse"][b, :, j], ref_l[b, :, j],
                      f"dense_v3 row {b}")
    assert res["err"] == 0
    assert np.all(np.isfinite(res["out"]))


def test_full_size_spec_decode_sampled_rows():
    """b=128, s_q=2 causal, lengths U[1024, 16384]: sampled query tokens of both positions."""
    w = workloads.WORKLOADS["spec"]
    inp = workloads.make_inputs(w)
    res = run_dense(inp, causal=True)
    rows = [(0, 0), (0, 1), (47, 1), (90, 0), (127, 1)]
    ref_o, ref_l = oracle_dense(inp, causal=True, rows=rows)
    for b, j in rows:
        assert_parity(res["out"][b, j], ref_o[b, j], res["lse"][b, :, j], ref_l[b, :, j],
                      f"spec row {b},{j}")
    assert res["err"] == 0 and np.all(np.isfinite(res["out"]))


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait on a barrier nothing completes gives up (MLA_DEVERR_TIMEOUT) and
    the kernel exits normally; a decode right after it is still correct."""
    import time
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    binding.mla_check_wait_timeout(err)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(err.item()) == binding.MLA_DEVERR_TIMEOUT
    assert 1.5 < dt < 30.0
    inp = workloads.make_inputs(workloads.WORKLOADS["tiny"])
    res = run_dense(inp)
    ref_o, ref_l = oracle_dense(inp)
    assert_parity(res["out"], ref_o, res["lse"], ref_l, "after timeout check")
    assert res["err"] == 0
