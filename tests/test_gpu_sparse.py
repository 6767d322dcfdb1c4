"""GPU parity of DSA top-k sparse decode against the fp64 oracle (through the C ABI).

Order invariance follows the flash-attention sparse-MLA article's test design:
the same top-k set with the dominant key first and last; each order's
coherent row gain (<out - ref, ref> / <ref, ref> per row) must stay within 2x
that of the ideal bf16 output.  The index gather is checked bit-exactly: with
exactly one valid index per query token the output row is that pool row's V
part, bit for bit, and the probe walks every row of a 4096-row pool.
"""
import os

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
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def run_sparse(inp, num_sm_parts=None):
    q = inp["q"].to(DEV)
    kv = inp["kv"].to(DEV)
    idx = inp["indices"].to(DEV)
    b, s_q, h, _ = q.shape
    topk = idx.shape[-1]
    buf = binding.DecodeBuffers(b, s_q, h, DEV, num_sm_parts)
    binding.mla_get_metadata(None, b, s_q, False, topk, buf.num_sm_parts, buf.metadata)
    binding.mla_sparse_decode(q, kv, idx, inp["softmax_scale"], buf.metadata, buf.num_sm_parts,
                              buf.workspace, buf.out, buf.lse, buf.err)
    torch.cuda.synchronize()
    return buf.out.float().cpu().numpy(), buf.lse.cpu().numpy(), int(buf.err.item())


def oracle_sparse(inp, rows=None):
    return oracle.sparse_decode(bf16_np(inp["q"]), bf16_np(inp["kv"]), inp["indices"].numpy(),
                                inp["softmax_scale"], rows)


def small(seed, b=2, s_q=1, h=16, s_kv=1000, topk=300, invalid=17):
    w = workloads.Workload("sp", "sparse", b=b, s_q=s_q, h=h, s_kv=s_kv, topk=topk,
                           invalid_per_row=invalid, seed=seed)
    return workloads.make_inputs(w)


def test_small_sparse_parity():
    inp = small(31)
    out, lse, err = run_sparse(inp)
    ref_o, ref_l = oracle_sparse(inp)
    assert_parity(out, ref_o, lse, ref_l, "sparse small")
    assert err == 0


@pytest.mark.parametrize("topk,parts", [(1, None), (127, None), (129, 3), (640, 1)])
def test_sparse_ragged_topk(topk, parts):
    inp = small(32 + topk, b=3, h=64, s_kv=3000, topk=topk, invalid=min(5, topk - 1))
    out, lse, err = run_sparse(inp, parts)
    ref_o, ref_l = oracle_sparse(inp)
    assert_parity(out, ref_o, lse, ref_l, f"sparse topk={topk}")


def test_sparse_h128_peaked_rows_and_s_q2():
    inp = small(40, b=3, s_q=2, h=128, s_kv=9000, topk=1000, invalid=50)
    out, lse, err = run_sparse(inp)
    ref_o, ref_l = oracle_sparse(inp)
    assert_parity(out, ref_o, lse, ref_l, "sparse h128")


def _row_gain(out, ref):
    o = out.reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    return np.sum((o - r) * r, axis=1) / np.sum(r * r, axis=1)


def test_sparse_index_order_invariance_row_gain():
    inp = small(41, b=2, h=128, s_kv=20000, topk=2048, invalid=0)
    ref_o, ref_l = oracle_sparse(inp)
    ideal = torch.from_numpy(ref_o).to(torch.bfloat16).double().numpy()
    floor = np.sqrt(np.mean(_row_gain(ideal, ref_o) ** 2))
    first = inp
    last = dict(inp)
    idx = inp["indices"].clone()
    last["indices"] = torch.cat([idx[..., 1:], idx[..., :1]], dim=-1)  # dominant key last
    for name, case in (("dominant first", first), ("dominant last", last)):
        out, lse, err = run_sparse(case)
        assert_parity(out, ref_o, lse, ref_l, name)
        gain = np.sqrt(np.mean(_row_gain(out, ref_o) ** 2))
        assert gain <= 2.0 * floor + 1e-6, (name, gain, floor)


def test_sparse_bad_and_all_invalid_indices():
    inp = small(42, b=2, h=32, s_kv=500, topk=200, invalid=3)
    inp["indices"][0, 0, 5] = 500          # == s_kv: out of range
    inp["indices"][0, 0, 9] = -7
    inp["indices"][1, 0, :] = -1           # nothing valid
    out, lse, err = run_sparse(inp)
    assert err & binding.MLA_DEVERR_BAD_INDEX
    ref_o, ref_l = oracle_sparse(inp)
    assert_parity(out[0], ref_o[0], lse[0], ref_l[0], "bad indices skipped")
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_dense_equals_sparse_on_the_same_rows():
    w = workloads.Workload("ds", "dense", b=2, s_q=1, h=128, seqlens=(700, 129), extra_pages=4,
                           seed=43)
    inp = workloads.make_inputs(w)
    q = inp["q"].to(DEV)
    kv = inp["kv_cache"].to(DEV)
    bt, sl = inp["block_table"].to(DEV), inp["cache_seqlens"].to(DEV)
    buf = binding.DecodeBuffers(2, 1, 128, DEV)
    binding.mla_get_metadata(sl, 2, 1, True, 0, buf.num_sm_parts, buf.metadata)
    binding.mla_decode(q, kv, binding.MLA_KV_BF16, bt, sl, inp["softmax_scale"], True,
                       buf.metadata, buf.num_sm_parts, buf.workspace, buf.out, buf.lse)
    torch.cuda.synchronize()
    dense_o, dense_l = buf.out.float().cpu().numpy(), buf.lse.cpu().numpy()
    topk = 700
    idx = torch.full((2, 1, topk), -1, dtype=torch.int32)
    btn = inp["block_table"].numpy()
    for b, L in enumerate((700, 129)):
        t = np.arange(L)
        idx[b, 0, :L] = torch.from_numpy((btn[b][t // 64] * 64 + t % 64).astype(np.int32))
    sp = dict(q=inp["q"], kv=inp["kv_cache"].reshape(-1, 576), indices=idx,
              softmax_scale=inp["softmax_scale"])
    out, lse, err = run_sparse(sp)
    assert_parity(out, dense_o, lse, dense_l, "sparse vs dense (GPU)")


def test_full_size_dsa_all_rows():
    """b=64, h=128, topk=2048 over a 32768-row pool (5% invalid slots, peaked
    heads): every query token and head compared with the oracle."""
    w = workloads.WORKLOADS["dsa"]
    inp = workloads.make_inputs(w)
    out, lse, err = run_sparse(inp)
    ref_o, ref_l = oracle_sparse(inp)
    st = assert_parity_per_token(out, ref_o, lse, ref_l, "dsa")
    print("dsa parity:", st)
    assert err == 0


def test_split_entry_then_combine_equals_sparse_decode():
    """mla_sparse_decode_splitkv + mla_combine on the same metadata and
    workspace gives the bytes mla_sparse_decode gives (128 heads: the two-SM
    kernel; 64: the one-SM kernel), with splits forced by 76 parts."""
    for h in (128, 64):
        inp = small(31 + h, b=3, s_q=2, h=h, s_kv=5000, topk=700, invalid=40)
        ref_o, ref_l, ref_e = run_sparse(inp, 76)
        q, kv, idx = inp["q"].to(DEV), inp["kv"].to(DEV), inp["indices"].to(DEV)
        b, s_q, _, _ = q.shape
        buf = binding.DecodeBuffers(b, s_q, h, DEV, 76)
        binding.mla_get_metadata(None, b, s_q, False, idx.shape[-1], 76, buf.metadata)
        binding.mla_sparse_decode_splitkv(q, kv, idx, inp["softmax_scale"], buf.metadata, 76,
                                          buf.workspace, buf.out, buf.lse, buf.err)
        binding.mla_combine(buf.metadata, b, s_q, h, 76, buf.workspace, buf.out, buf.lse)
        torch.cuda.synchronize()
        assert int(buf.err.item()) == ref_e == 0
        assert np.array_equal(buf.out.float().cpu().numpy(), ref_o)
        assert np.array_equal(buf.lse.cpu().numpy(), ref_l)


@pytest.mark.parametrize("h,parts", [(128, None), (128, 3), (64, None), (64, 3)])
def test_sparse_attn_sink_and_topk_length(h, parts):
    """The sparse extensions: a per-head attention sink and a per-token topk
    length (through the schedule), on both kernels; with 3 parts the rows are
    split and the sink is applied by the combine, otherwise by the split
    kernel's epilogue.  Lengths include 0 (empty row), 1, a ragged tile and topk."""
    b, s_q, topk = 3, 2, 700
    inp = small(61 + h, b=b, s_q=s_q, h=h, s_kv=5000, topk=topk, invalid=40)
    q, kv, idx = inp["q"].to(DEV), inp["kv"].to(DEV), inp["indices"].to(DEV)
    lengths = torch.tensor([0, 1, 129, 700, 640, 255], dtype=torch.int32)
    g = torch.Generator().manual_seed(7)
    sink = (torch.randn(h, generator=g, dtype=torch.float64) * 3 + 6).to(torch.float32)
    buf = binding.DecodeBuffers(b, s_q, h, DEV, parts)
    binding.mla_get_metadata(lengths.to(DEV), b, s_q, False, topk, buf.num_sm_parts, buf.metadata)
    binding.mla_sparse_decode(q, kv, idx, inp["softmax_scale"], buf.metadata, buf.num_sm_parts,
                              buf.workspace, buf.out, buf.lse, buf.err, attn_sink=sink.to(DEV))
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.sparse_decode(bf16_np(inp["q"]), bf16_np(inp["kv"]), inp["indices"].numpy(),
                                        inp["softmax_scale"], attn_sink=sink.double().numpy(),
                                        topk_length=lengths.numpy().reshape(b, s_q))
    out, lse = buf.out.float().cpu().numpy(), buf.lse.cpu().numpy()
    assert_parity(out, ref_o, lse, ref_l, f"sink+length h={h} parts={parts}")
    assert int(buf.err.item()) == 0
    assert np.all(out[0, 0] == 0) and np.all(np.isneginf(lse[0, :, 0]))   # length 0


@pytest.mark.parametrize("h", [64, 128])
def test_index_gather_bit_exact_every_pool_row(h):
    """One valid index per query token (at a random slot of two 128-slot
    tiles, the rest -1): the output of every head is that pool row's first
    512 columns exactly.  Eight calls of 512 tokens address all 4096 rows."""
    s_kv, topk, n_tok = 4096, 256, 512
    g = torch.Generator().manual_seed(81 + h)
    pool = torch.randn((s_kv, 576), generator=g).to(torch.bfloat16)
    perm = torch.randperm(s_kv, generator=g)
    dev_pool = pool.to(DEV)
    for call in range(s_kv // n_tok):
        rows = perm[call * n_tok:(call + 1) * n_tok]
        idx = torch.full((n_tok, 1, topk), -1, dtype=torch.int32)
        slots = torch.randint(0, topk, (n_tok,), generator=g)
        idx[torch.arange(n_tok), 0, slots] = rows.to(torch.int32)
        q = torch.randn((n_tok, 1, h, 576), generator=g).to(torch.bfloat16)
        buf = binding.DecodeBuffers(n_tok, 1, h, DEV)
        binding.mla_get_metadata(None, n_tok, 1, False, topk, buf.num_sm_parts, buf.metadata)
        binding.mla_sparse_decode(q.to(DEV), dev_pool, idx.to(DEV), workloads.SOFTMAX_SCALE, buf.metadata,
                                  buf.num_sm_parts, buf.workspace, buf.out, buf.lse, buf.err)
        torch.cuda.synchronize()
        out = buf.out.cpu()
        want = pool[rows.long(), :512]
        assert torch.equal(out[:, 0], want[:, None, :].expand(n_tok, h, 512)), f"call {call}"
        s_ref = (q[:, 0].double() @ pool[rows.long()].double()[:, :, None])[:, :, 0] * workloads.SOFTMAX_SCALE
        assert torch.max(torch.abs(buf.lse.cpu()[:, :, 0].double() - s_ref)) < 1e-3
        assert int(buf.err.item()) == 0


@pytest.mark.parametrize("h,parts", [(128, None), (128, 3), (64, None), (64, 3)])
def test_unnamed_pool_rows_never_reach_the_output(h, parts):
    """Pool rows no token names hold NaN (row 0 included, the row invalid
    slots used to be read from).  Token 0 has 5% invalid slots, token 1 a
    first 256-slot stretch with no valid index, token 2 no valid index at
    all.  Outputs are finite and match the oracle; token 2 gets 0 / -inf."""
    b, topk, s_kv = 3, 640, 3000
    inp = small(91 + h, b=b, h=h, s_kv=s_kv, topk=topk, invalid=32)
    idx = inp["indices"]
    idx[1, 0, :256] = -1
    idx[2, 0, :] = -1
    named = torch.zeros(s_kv, dtype=torch.bool)
    named[idx[idx >= 0].long()] = True
    pool = inp["kv"].clone()
    pool[~named] = float("nan")
    case = dict(inp, kv=pool, indices=idx)
    out, lse, err = run_sparse(case, parts)
    assert err == 0
    assert np.all(np.isfinite(out))
    ref_o, ref_l = oracle_sparse(case)
    assert_parity(out[:2], ref_o[:2], lse[:2], ref_l[:2], "unnamed rows are NaN")
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


# ------------------------------------------------------------ sparse prefill

def run_prefill(q, kv, idx, scale, topk_length=None, attn_sink=None, num_sm_parts=None):
    """mla_sparse_prefill through the C ABI: q [s_q, h, 576], kv [s_kv, 1, 576],
    indices [s_q, 1, topk]; returns out [s_q, h, 512], lse [s_q, h], err."""
    q, kv, idx = q.to(DEV), kv.to(DEV), idx.to(DEV)
    s_q, h, _ = q.shape
    topk = idx.shape[-1]
    buf = binding.DecodeBuffers(s_q, 1, h, DEV, num_sm_parts)
    tl = None if topk_length is None else topk_length.to(DEV)
    sink = None if attn_sink is None else attn_sink.to(DEV)
    binding.mla_get_metadata(tl, s_q, 1, False, topk, buf.num_sm_parts, buf.metadata)
    out = torch.empty((s_q, h, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((s_q, h), dtype=torch.float32, device=DEV)
    binding.mla_sparse_prefill(q, kv, idx, scale, buf.metadata, buf.num_sm_parts, buf.workspace, out, lse,
                               buf.err, attn_sink=sink)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(buf.err.item())


def prefill_inputs(seed, s_q, h, s_kv, topk, invalid):
    inp = small(seed, b=s_q, s_q=1, h=h, s_kv=s_kv, topk=topk, invalid=invalid)
    return (inp["q"][:, 0], inp["kv"].reshape(s_kv, 1, 576), inp["indices"].reshape(s_q, 1, topk),
            inp["softmax_scale"])


@pytest.mark.parametrize("h,parts", [(128, None), (64, None), (128, 7)])
def test_sparse_prefill_parity(h, parts):
    """Many query tokens with their own index lists (ragged tiles, invalid
    slots, a per-token topk_length and an attention sink), every token
    compared with the oracle."""
    s_q, s_kv, topk = 96, 6000, 400
    q, kv, idx, scale = prefill_inputs(70 + h, s_q, h, s_kv, topk, 20)
    g = torch.Generator().manual_seed(71)
    tl = torch.randint(0, topk + 1, (s_q,), generator=g, dtype=torch.int64).to(torch.int32)
    tl[:4] = torch.tensor([topk, 1, 0, 129], dtype=torch.int32)
    sink = torch.randn((h,), generator=g, dtype=torch.float32)
    out, lse, err = run_prefill(q, kv, idx, scale, tl, sink, parts)
    ref_o, ref_l = oracle.sparse_prefill(bf16_np(q), bf16_np(kv), idx.numpy(), scale, attn_sink=sink.numpy(),
                                         topk_length=tl.numpy())
    # the decode helpers take [b, s_q, h, 512] / [b, h, s_q]
    assert_parity(out[:, None], ref_o[:, None], lse[:, :, None], ref_l[:, :, None], f"sparse prefill h={h}")
    assert err == 0


def test_sparse_prefill_single_index_rows_are_exact():
    """Each token names one row (the rest -1): its output is that row's V
    part bit for bit, so the per-token index gather is exact."""
    s_q, s_kv, h = 256, 5000, 128
    g = torch.Generator().manual_seed(72)
    kv = torch.randn((s_kv, 1, 576), generator=g).to(torch.bfloat16)
    q = torch.randn((s_q, h, 576), generator=g).to(torch.bfloat16)
    rows = torch.randperm(s_kv, generator=g)[:s_q].to(torch.int32)
    idx = torch.full((s_q, 1, 64), -1, dtype=torch.int32)
    slot = torch.randint(0, 64, (s_q,), generator=g)
    idx[torch.arange(s_q), 0, slot] = rows
    out, _, err = run_prefill(q, kv, idx, workloads.SOFTMAX_SCALE)
    want = kv[rows.long(), 0, :512].float().numpy()
    assert np.array_equal(out, np.broadcast_to(want[:, None, :], out.shape))
    assert err == 0
