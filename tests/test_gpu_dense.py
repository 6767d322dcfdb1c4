"""GPU parity of the dense paged decode against the fp64 oracle (through the C ABI).

Tolerances: bf16 out rel-L2 <= 3e-3 and max-abs <= 2e-2 * RMS(out_ref),
LSE abs error <= 1e-3.  The block-table gather is checked bit-exactly: in the
probe tests each query row is built so that one cached token outweighs every
other by more than 2^-150 (all other weights are exactly 0 in fp32), so the
output row must be that token's V row, bit for bit; every token position of
every request (every block-table entry, every slot of a page, the partial
last page) is addressed by some row.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_gb300 import binding, workloads
from tests._util import assert_parity, assert_parity_per_token, bf16_np

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


@pytest.mark.parametrize("h", [16, 128])  # the split kernel; the two-SM kernel (schedule B, empty parts)
def test_empty_sequences(h):
    w = workloads.Workload("empty", "dense", b=3, s_q=2, h=h, seqlens=(0, 1, 70), seed=16)
    inp = workloads.make_inputs(w)
    res = run_dense(inp)
    ref_o, ref_l = oracle_dense(inp)
    assert np.all(res["out"][0] == 0) and np.all(np.isneginf(res["lse"][0]))
    assert np.all(res["out"][1, 0] == 0) and np.all(np.isneginf(res["lse"][1, :, 0]))
    assert_parity(res["out"][2], ref_o[2], res["lse"][2], ref_l[2], "empty/nonempty")


@pytest.mark.parametrize("h", [16, 128])
def test_bad_page_ids_are_flagged_not_faulted(h):
    """Bad page ids in two requests are flagged and read as nothing outside the
    cache; the third request, whose pages are all valid, is unaffected."""
    w = workloads.Workload("badpage", "dense", b=3, s_q=1, h=h, seqlens=(100, 200, 300), seed=17)
    inp = workloads.make_inputs(w)
    good = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in inp.items()}
    inp["block_table"][1, 1] = 10 ** 6      # past the cache
    inp["block_table"][0, 0] = -5
    res = run_dense(inp)
    assert res["err"] & binding.MLA_DEVERR_BAD_PAGE
    assert np.all(np.isfinite(res["out"]))
    ref_o, ref_l = oracle_dense(good, rows=[(2, 0)])
    assert_parity(res["out"][2], ref_o[2], res["lse"][2], ref_l[2], "request with valid pages")


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
    assert int(workspace_ctrl(buf)[0]) == walked
    ref_o, ref_l = oracle_dense(inp)
    assert_parity(buf.out.float().cpu().numpy(), ref_o, buf.lse.cpu().numpy(), ref_l, f"h={h} parts={parts}")


@pytest.mark.parametrize("batch", [70, 128, 2100])  # the 128- and the 1024-thread schedule kernel
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


def test_full_size_dense_v3_all_rows():
    """b=64, h=128, t=4096 in the bench's launch configuration; every request
    and head compared with the oracle, and each request on its own."""
    w = workloads.WORKLOADS["dense_v3"]
    inp = workloads.make_inputs(w)
    res = run_dense(inp)
    ref_o, ref_l = oracle_dense(inp)
    st = assert_parity_per_token(res["out"], ref_o, res["lse"], ref_l, "dense_v3")
    print("dense_v3 parity:", st)
    assert res["err"] == 0


def test_full_size_spec_decode_all_rows():
    """b=128, s_q=2 causal, lengths U[1024, 16384]: every query token of both
    positions and every head compared with the oracle."""
    w = workloads.WORKLOADS["spec"]
    inp = workloads.make_inputs(w)
    res = run_dense(inp, causal=True)
    ref_o, ref_l = oracle_dense(inp, causal=True)
    st = assert_parity_per_token(res["out"], ref_o, res["lse"], ref_l, "spec")
    print("spec parity:", st)
    assert res["err"] == 0


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


def workspace_ctrl(buf):
    """The workspace's control words (int32), after the partial O and LSE rows."""
    rows = (buf.batch * buf.s_q + buf.num_sm_parts) * buf.h_q
    return buf.workspace[rows * 513:].view(torch.int32).cpu().numpy()


# ---------------------------------------------------------------- gather probes

ROPE_GAIN = 256.0  # q's RoPE part = ROPE_GAIN * the target key's RoPE signs (exact in bf16)


def probe_cache(seqlens, extra_pages, seed):
    """A paged cache whose RoPE columns are random +-1 signs (latent columns
    N(0,1) bf16), with a shuffled block table.  Returns (kv [pages, 64, 576]
    bf16, block_table [b, max_pages] int32)."""
    g = torch.Generator().manual_seed(seed)
    n_pages = [(L + 63) // 64 for L in seqlens]
    total = sum(n_pages) + extra_pages
    perm = torch.randperm(total, generator=g).to(torch.int32)
    bt = torch.full((len(seqlens), max(n_pages)), -1, dtype=torch.int32)
    pos = 0
    for i, n in enumerate(n_pages):
        bt[i, :n] = perm[pos:pos + n]
        pos += n
    kv = torch.randn((total, 64, 576), generator=g).to(torch.bfloat16)
    signs = torch.randint(0, 2, (total, 64, 64), generator=g).to(torch.float32) * 2 - 1
    kv[:, :, 512:] = signs.to(torch.bfloat16)
    return kv, bt


def probe_queries(kv, bt, seqlens, h, rnd):
    """Query rows for round `rnd`: head hh of request b targets token
    t = rnd * h + hh (when t < seqlens[b], else a zero row).  Returns q
    [b, 1, h, 576] bf16 and the targets [b, h] (-1 = none)."""
    b = len(seqlens)
    q = torch.zeros((b, 1, h, 576), dtype=torch.bfloat16)
    tgt = torch.full((b, h), -1, dtype=torch.int64)
    for bi, L in enumerate(seqlens):
        if rnd * h >= L:
            continue
        t = torch.arange(rnd * h, min(L, (rnd + 1) * h))
        rows = kv[bt[bi, t // 64].long(), t % 64]                 # [n, 576]
        q[bi, 0, :len(t), 512:] = (rows[:, 512:].float() * ROPE_GAIN).to(torch.bfloat16)
        tgt[bi, :len(t)] = t
    return q, tgt


def assert_probe_preconditions(kv, bt, seqlens):
    """Every other visible token's RoPE signs differ from the target's in at
    least 3 of 64 places: its score is lower by >= 6 * 256 / sqrt(192) > 110,
    i.e. a weight below 2^-150, exactly 0 in fp32."""
    for bi, L in enumerate(seqlens):
        t = torch.arange(L)
        s = kv[bt[bi, t // 64].long(), t % 64][:, 512:].float()
        gram = s @ s.T
        gram.fill_diagonal_(-64)
        assert float(gram.max()) <= 64 - 6


def check_probe(out, lse, kv, bt, tgt, what):
    """Rows with a target equal that token's V row bit for bit; their lse is
    the target's score (every other weight is exactly 0)."""
    scale = workloads.SOFTMAX_SCALE
    bi, hh = torch.nonzero(tgt >= 0, as_tuple=True)
    t = tgt[bi, hh]
    want = kv[bt[bi, t // 64].long(), t % 64, :512]
    got = out[bi, 0, hh]
    same = torch.all(got.view(torch.int16) == want.view(torch.int16), dim=-1)
    if not bool(torch.all(same)):
        k = int(torch.nonzero(~same)[0])
        raise AssertionError(f"{what}: request {int(bi[k])} token {int(t[k])} (head {int(hh[k])}) "
                             f"is not an exact copy of its V row")
    err = torch.abs(lse[bi, hh, 0].double() - scale * ROPE_GAIN * 64)
    assert float(err.max()) < 1e-3, (what, float(err.max()))


def run_probe(kv, bt, seqlens, h, parts=None):
    dev_kv, dev_bt = kv.to(DEV), bt.to(DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    b = len(seqlens)
    buf = binding.DecodeBuffers(b, 1, h, DEV, parts)
    binding.mla_get_metadata(sl.to(DEV), b, 1, True, 0, buf.num_sm_parts, buf.metadata)
    for rnd in range((max(seqlens) + h - 1) // h):
        q, tgt = probe_queries(kv, bt, seqlens, h, rnd)
        buf.out.fill_(float("nan"))
        binding.mla_decode(q.to(DEV), dev_kv, binding.MLA_KV_BF16, dev_bt, sl.to(DEV),
                           workloads.SOFTMAX_SCALE, True, buf.metadata, buf.num_sm_parts,
                           buf.workspace, buf.out, buf.lse, buf.err)
        torch.cuda.synchronize()
        check_probe(buf.out.cpu(), buf.lse.cpu(), kv, bt, tgt, f"h={h} round {rnd}")
    assert int(buf.err.item()) == 0


@pytest.mark.parametrize("h,parts", [(16, None), (64, None), (128, None), (128, 5), (16, 3)])
def test_gather_bit_exact_every_token_small_cache(h, parts):
    """The small cache's shape (two requests of 200 and 333 tokens, 10 of 16
    pages used, shuffled): every token position of both requests is the
    target of one query row; its output must be the token's V row exactly."""
    seqlens = (200, 333)
    kv, bt = probe_cache(seqlens, 6, seed=71)
    assert_probe_preconditions(kv, bt, seqlens)
    run_probe(kv, bt, seqlens, h, parts)


def test_gather_bit_exact_every_token_full_size():
    """b=64, h=128, every request 4096 tokens, 4096 shuffled pages, in the
    bench's launch configuration: 32 calls, call k addressing tokens
    128k .. 128k+127 of every request (every block-table entry and slot)."""
    seqlens = (4096,) * 64
    kv, bt = probe_cache(seqlens, 0, seed=72)
    assert_probe_preconditions(kv, bt, seqlens[:4])
    run_probe(kv, bt, seqlens, 128)


# ---------------------------------------------------------------- metadata checks

@pytest.mark.parametrize("h", [64, 128])
def test_metadata_for_another_shape_is_rejected_on_the_device(h):
    """Metadata built for b=4 passed to a b=2 call (and metadata built for a
    sparse call, and for the other causal flag): the kernel sets
    MLA_DEVERR_METADATA and writes nothing."""
    w = workloads.Workload("meta", "dense", b=2, s_q=2, h=h, seqlens=(300, 500), seed=24)
    inp = workloads.make_inputs(w)
    q, kv = inp["q"].to(DEV), inp["kv_cache"].to(DEV)
    bt, sl = inp["block_table"].to(DEV), inp["cache_seqlens"].to(DEV)
    sl4 = torch.tensor([300, 500, 700, 900], dtype=torch.int32, device=DEV)
    big = binding.DecodeBuffers(4, 2, h, DEV)
    cases = [("batch", lambda m: binding.mla_get_metadata(sl4, 4, 2, True, 0, big.num_sm_parts, m)),
             ("topk", lambda m: binding.mla_get_metadata(None, 2, 2, False, 64, big.num_sm_parts, m)),
             ("causal", lambda m: binding.mla_get_metadata(sl, 2, 2, False, 0, big.num_sm_parts, m))]
    for name, build_meta in cases:
        build_meta(big.metadata)
        buf = binding.DecodeBuffers(2, 2, h, DEV, big.num_sm_parts)
        buf.out.fill_(7.0)
        buf.lse.fill_(7.0)
        binding.mla_decode(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"], True,
                           big.metadata, big.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
        torch.cuda.synchronize()
        assert int(buf.err.item()) & binding.MLA_DEVERR_METADATA, name
        assert torch.all(buf.out == 7.0) and torch.all(buf.lse == 7.0), name


@pytest.mark.parametrize("h", [64, 128])
def test_metadata_from_other_lengths_is_flagged(h):
    """The right shape but lengths that differ from cache_seqlens: flagged,
    no fault, and the result follows the metadata's key counts."""
    w = workloads.Workload("meta_len", "dense", b=2, s_q=1, h=h, seqlens=(300, 500), seed=25)
    inp = workloads.make_inputs(w)
    q, kv = inp["q"].to(DEV), inp["kv_cache"].to(DEV)
    bt, sl = inp["block_table"].to(DEV), inp["cache_seqlens"].to(DEV)
    buf = binding.DecodeBuffers(2, 1, h, DEV)
    binding.mla_get_metadata(torch.tensor([300, 260], dtype=torch.int32, device=DEV), 2, 1, True, 0,
                             buf.num_sm_parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"], True, buf.metadata,
                       buf.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    assert int(buf.err.item()) == binding.MLA_DEVERR_METADATA
    short = dict(inp)
    short["cache_seqlens"] = torch.tensor([300, 260], dtype=torch.int32)
    ref_o, ref_l = oracle_dense(short)
    assert_parity(buf.out.float().cpu().numpy(), ref_o, buf.lse.cpu().numpy(), ref_l, "metadata lengths")


@pytest.mark.parametrize("h", [64, 128])
def test_length_beyond_the_block_table_row_is_flagged(h):
    """A request whose length needs more page slots than block_table_stride:
    MLA_DEVERR_BAD_PAGE, nothing read past the row, the other request exact."""
    w = workloads.Workload("stride", "dense", b=2, s_q=1, h=h, seqlens=(300, 200), extra_pages=4, seed=26)
    inp = workloads.make_inputs(w)
    bt = inp["block_table"][:, :4].contiguous()          # room for 256 tokens per request
    lens = torch.tensor([300, 200], dtype=torch.int32)   # request 0 needs 5 slots
    q, kv = inp["q"].to(DEV), inp["kv_cache"].to(DEV)
    buf = binding.DecodeBuffers(2, 1, h, DEV)
    binding.mla_get_metadata(lens.to(DEV), 2, 1, True, 0, buf.num_sm_parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_BF16, bt.to(DEV), lens.to(DEV), inp["softmax_scale"], True,
                       buf.metadata, buf.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    assert int(buf.err.item()) & binding.MLA_DEVERR_BAD_PAGE
    out, lse = buf.out.float().cpu().numpy(), buf.lse.cpu().numpy()
    assert np.all(np.isfinite(out))
    ref_o, ref_l = oracle_dense(inp, rows=[(1, 0)])
    assert_parity(out[1], ref_o[1], lse[1], ref_l[1], "request within its row")
