"""Host-side tests of the C ABI (no GPU): exports, argument checks, schedule.

The schedule tests pin ``mla_get_metadata_host`` by invariants: every
(sequence, tile) pair is covered exactly once, pieces of a sequence are
numbered 0..n_splits-1 in order, split offsets are the exclusive prefix of
split counts, key counts follow the causal reading, and parts are balanced.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_decode_attention_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_are_exported():
    names = declared_functions()
    assert "mla_decode" in names and "mla_get_metadata" in names and len(names) >= 9
    lib = ctypes.CDLL(binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/mla_decode.h but not exported"


def test_binding_covers_every_declared_function():
    assert set(declared_functions()) <= set(binding._SIGS)


def test_status_strings():
    assert binding.status_string(0) == "ok"
    for s in (-1, -2, -3, -4, -5, -6):
        assert binding.status_string(s) not in ("ok", "unknown status")
    assert binding.status_string(12345) == "unknown status"


def test_sizes():
    # two schedules (A: balanced ranges, B: one whole sequence per part)
    assert binding.mla_metadata_size(64, 1, 76) == 2 * 4 * (16 + 8 * 76 + 8 * 64)
    # fp32 partial O and LSE rows, then 64 bytes of control words
    assert binding.mla_workspace_size(64, 1, 128, 76) == (64 + 76) * 128 * 513 * 4 + 64
    with pytest.raises(binding.MlaError):
        binding.mla_workspace_size(64, 1, 100, 76)      # unsupported head count
    with pytest.raises(binding.MlaError):
        binding.mla_metadata_size(0, 1, 76)
    with pytest.raises(binding.MlaError):
        binding.mla_metadata_size(4, 17, 76)             # s_q > 16


def _decode_args(**over):
    """Arguments of mla_decode with fake (never dereferenced) aligned pointers."""
    a = dict(q=0x10000, kv=0x20000, fmt=0, pages=16, bt=0x30000, bt_stride=8, sl=0x40000,
             batch=2, s_q=1, h=16, scale=0.07, causal=1, meta=0x50000, parts=4, ws=0x60000,
             out=0x70000, lse=0x80000, err=None, stream=None)
    a.update(over)
    return a


def _call_decode(a):
    return binding.lib().mla_decode(a["q"], a["kv"], a["fmt"], a["pages"], a["bt"],
                                    a["bt_stride"], a["sl"], a["batch"], a["s_q"], a["h"],
                                    a["scale"], a["causal"], a["meta"], a["parts"], a["ws"],
                                    a["out"], a["lse"], a["err"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(q=None), -1), (dict(kv=None), -1), (dict(out=None), -1), (dict(meta=None), -1),
    (dict(h=100), -2), (dict(h=256), -2), (dict(s_q=0), -2), (dict(s_q=17), -2),
    (dict(batch=0), -2), (dict(pages=0), -2), (dict(parts=0), -2), (dict(scale=0.0), -2),
    (dict(scale=float("nan")), -2), (dict(q=0x10008), -3), (dict(kv=0x20004), -3),
    (dict(out=0x70002), -3), (dict(fmt=7), -6),
])
def test_decode_rejects_bad_arguments_before_launch(over, code):
    assert _call_decode(_decode_args(**over)) == code


# ------------------------------------------------------------------ schedule

def parse_meta(m, n_seq, parts):
    hdr = m[:16]
    prt = m[16:16 + 8 * parts].reshape(parts, 8)
    seq = m[16 + 8 * parts:16 + 8 * parts + 8 * n_seq].reshape(n_seq, 8)
    return hdr, prt, seq


def walk_part(prt_row, seq):
    """Pieces (q, t0, t1, split) a part processes, as the kernels walk them
    (sequences q_begin, q_begin + q_step, ...)."""
    q, t, qe, te, split, step = [int(x) for x in prt_row[:6]]
    assert step >= 1
    pieces = []
    while q < qe or (q == qe and t < te):
        nt = int(seq[q, 0])
        stop = te if q == qe else nt
        if nt > 0 and t < stop:
            pieces.append((q, t, stop, split))
        q, t, split = q + step, 0, 0
    return pieces


# Cost of a sequence piece in tile units besides its tiles (the Q load and
# the epilogue), as include/mla_decode.h documents it.
FIXED_COST = 2


def check_schedule(seqlens, s_q, causal, topk, parts):
    b = len(seqlens)
    m = binding.mla_get_metadata_host(None if topk else seqlens, b, s_q, causal, topk, parts)
    hdr, prt, seq = parse_meta(m, b * s_q, parts)
    assert hdr[0] == 0x4D4C4131 and hdr[2] == b * s_q and hdr[3] == parts and hdr[4] == 128
    for q in range(b * s_q):
        bi, j = divmod(q, s_q)
        if topk:
            keys = topk
        else:
            keys = max(0, seqlens[bi] - s_q + 1 + j) if causal else max(0, seqlens[bi])
        assert seq[q, 3] == keys and seq[q, 0] == (keys + 127) // 128
    covered = {}
    per_part_cost = []
    for p in range(parts):
        cost = 0
        for (q, t0, t1, split) in walk_part(prt[p], seq):
            cost += (t1 - t0) + FIXED_COST
            for t in range(t0, t1):
                assert (q, t) not in covered
                covered[(q, t)] = (p, split)
        per_part_cost.append(cost)
    for q in range(b * s_q):
        nt = int(seq[q, 0])
        for t in range(nt):
            assert (q, t) in covered, (q, t)
        splits = [covered[(q, t)][1] for t in range(nt)]
        # piece numbers start at 0 and grow by one at each part change
        if nt:
            assert splits[0] == 0
            owners = [covered[(q, t)][0] for t in range(nt)]
            for t in range(1, nt):
                if owners[t] == owners[t - 1]:
                    assert splits[t] == splits[t - 1]
                else:
                    assert splits[t] == splits[t - 1] + 1
            assert seq[q, 2] == splits[-1] + 1
        else:
            assert seq[q, 2] == 0
    order = walk_order(hdr)
    offs = np.zeros(b * s_q, np.int64)
    offs[order] = np.concatenate([[0], np.cumsum(seq[order, 2])[:-1]])
    assert np.array_equal(seq[:, 1], offs)   # split offsets in the builders' walk order
    assert hdr[9] == seq[:, 2].sum() <= b * s_q + parts
    groups = int(hdr[13])
    assert groups == (s_q if s_q > 1 and parts % s_q == 0 else 1)
    assert max(per_part_cost) <= hdr[10] + FIXED_COST
    costs = [int(nt) + FIXED_COST if nt > 0 else 0 for nt in seq[:, 0]]
    assert hdr[11] == max(costs) and hdr[12] == (1 if b * s_q <= parts else 0)
    check_whole_sequence_schedule(m, b * s_q, parts, hdr, seq)
    return m


def walk_order(hdr):
    """Sequences in the builders' order: group-major (all first new tokens,
    then all second ones, ...) when schedule A has one group per token."""
    n_seq, groups = int(hdr[2]), int(hdr[13])
    n_g = n_seq // groups
    return np.array([(k % n_g) * groups + k // n_g for k in range(n_seq)], np.int64)


def check_whole_sequence_schedule(m, n_seq, parts, hdr_a, seq_a):
    """Schedule B: present iff n_seq <= parts; part p walks all of sequence p."""
    words = 16 + 8 * parts + 8 * n_seq
    assert len(m) == 2 * words
    hdr, prt, seq = parse_meta(m[words:], n_seq, parts)
    if n_seq > parts:
        assert not hdr.any()
        return
    assert np.array_equal(hdr[:9], hdr_a[:9]) and hdr[10] == hdr[11] == hdr_a[11]
    assert hdr[12] == 0  # no third schedule follows B
    assert np.array_equal(seq[:, [0, 3, 4]], seq_a[:, [0, 3, 4]])
    assert np.array_equal(seq[:, 2], (seq[:, 0] > 0).astype(np.int32))
    order = walk_order(hdr_a)
    offs = np.zeros(n_seq, np.int64)
    offs[order] = np.concatenate([[0], np.cumsum(seq[order, 2])[:-1]])
    assert np.array_equal(seq[:, 1], offs)
    assert hdr[9] == seq[:, 2].sum()
    for p in range(parts):
        pieces = walk_part(prt[p], seq)
        if p < n_seq and seq[p, 0] > 0:
            assert pieces == [(p, 0, int(seq[p, 0]), 0)]
        else:
            assert pieces == []


def walks_whole_sequences(m, penalty):
    """The kernels' choice: B when present and at most `penalty` tiles longer."""
    hdr = m[:16]
    words = 16 + 8 * int(hdr[3]) + 8 * int(hdr[2])
    has_b = m[words] == 0x4D4C4131
    assert hdr[12] == (1 if has_b else 0), "schedule A's header flags whether schedule B follows"
    return has_b and hdr[11] <= hdr[10] + penalty


@pytest.mark.parametrize("parts", [1, 2, 7, 76, 152, 400])
def test_schedule_dense_invariants(parts):
    rng = np.random.default_rng(parts)
    seqlens = rng.integers(0, 5000, size=37).astype(np.int32)
    seqlens[:4] = [0, 1, 128, 129]
    check_schedule(seqlens, 1, True, 0, parts)


@pytest.mark.parametrize("s_q,causal", [(2, True), (2, False), (3, True)])
def test_schedule_spec_invariants(s_q, causal):
    rng = np.random.default_rng(s_q)
    seqlens = rng.integers(0, 20000, size=19).astype(np.int32)
    seqlens[0] = 1   # causal: token 0 of this request sees nothing
    check_schedule(seqlens, s_q, causal, 0, 76)


def test_spec_schedule_walks_both_new_tokens_in_step():
    """s_q = 2 over 76 parts: group j = token j of every request, 38 parts
    each; part p and part p + 38 walk the same requests and tiles (token 0
    and token 1), so the second reader of a cache row finds it in L2."""
    rng = np.random.default_rng(9)
    seqlens = rng.integers(1024, 16385, size=128).astype(np.int32)
    m = check_schedule(seqlens, 2, False, 0, 76)   # non-causal: both tokens see L keys
    hdr, prt, seq = parse_meta(m, 256, 76)
    assert hdr[13] == 2
    for p in range(38):
        a = walk_part(prt[p], seq)
        b = walk_part(prt[p + 38], seq)
        assert [(q // 2, t0, t1) for q, t0, t1, _ in a] == [(q // 2, t0, t1) for q, t0, t1, _ in b]
        assert all(q % 2 == 0 for q, *_ in a) and all(q % 2 == 1 for q, *_ in b)


def test_schedule_sparse_invariants():
    check_schedule(np.zeros(64, np.int32), 1, False, 2048, 76)
    check_schedule(np.zeros(5, np.int32), 2, False, 100, 152)


def test_schedule_config_dense_v3_shape():
    m = check_schedule(np.full(64, 4096, np.int32), 1, True, 0, 76)
    hdr, prt, seq = parse_meta(m, 64, 76)
    assert hdr[10] == (64 * (32 + FIXED_COST) + 75) // 76   # balanced cost per part
    assert seq[:, 2].max() <= 3
    # 34 tiles per part unsplit against 29 split: the two-SM kernels (split
    # penalties 11 dense, 5 sparse) walk whole sequences, the one-SM kernel (4)
    # the balanced split
    assert walks_whole_sequences(m, 11) and walks_whole_sequences(m, 5)
    assert not walks_whole_sequences(m, 4)


def test_schedule_choice_prefers_splitting_long_uneven_batches():
    # 32 requests of 8192 keys over 76 parts: unsplit 66 tiles against 28
    m = check_schedule(np.full(32, 8192, np.int32), 1, True, 0, 76)
    assert not walks_whole_sequences(m, 11)
    # more sequences than parts: no schedule B at all
    m = check_schedule(np.full(80, 1000, np.int32), 1, True, 0, 76)
    assert not walks_whole_sequences(m, 1000)


def test_sparse_schedule_with_topk_length():
    """Sparse with per-token lengths (topk_length in place of cache_seqlens):
    each query token's key count is its length clamped to [0, topk], and the
    schedule covers exactly those tiles."""
    b, s_q, topk, parts = 5, 2, 700, 7
    lengths = np.array([0, 1, 127, 128, 129, 700, 701, -3, 640, 255], np.int32)
    m = binding.mla_get_metadata_host(lengths, b, s_q, False, topk, parts)
    hdr, prt, seq = parse_meta(m, b * s_q, parts)
    keys = np.clip(lengths, 0, topk)
    assert np.array_equal(seq[:, 3], keys) and np.array_equal(seq[:, 0], (keys + 127) // 128)
    covered = set()
    for p in range(parts):
        for (q, t0, t1, _) in walk_part(prt[p], seq):
            covered.update((q, t) for t in range(t0, t1))
    assert covered == {(q, t) for q in range(b * s_q) for t in range(int(seq[q, 0]))}
    assert np.array_equal(seq[:, 2] > 0, seq[:, 0] > 0)     # empty tokens have no split


def test_benchmark_workloads_walk_the_documented_schedules():
    """Dense b=64 t=4096 and DSA walk whole sequences on the two-SM kernels;
    FP8 t=8192 keeps the balanced split on the one-SM kernel; spec (256 query
    tokens over 76 parts) has only the balanced split, in two token groups."""
    from mla_decode_attention_gb300 import workloads
    dense = binding.mla_get_metadata_host(np.full(64, 4096, np.int32), 64, 1, True, 0, 76)
    assert walks_whole_sequences(dense, 11)
    dsa = binding.mla_get_metadata_host(None, 64, 1, False, 2048, 76)
    assert walks_whole_sequences(dsa, 5)
    fp8 = binding.mla_get_metadata_host(np.full(64, 8192, np.int32), 64, 1, True, 0, 76)
    assert not walks_whole_sequences(fp8, 4)
    w = workloads.WORKLOADS["spec"]
    sl = np.random.default_rng(3).integers(*w.seqlen_range, size=w.b, endpoint=True).astype(np.int32)
    spec = binding.mla_get_metadata_host(sl, w.b, w.s_q, True, 0, 76)
    assert not walks_whole_sequences(spec, 11) and spec[13] == 2


def _call_sparse(**over):
    """mla_sparse_decode with fake (never dereferenced) aligned pointers."""
    a = dict(q=0x10000, kv=0x20000, s_kv=1000, idx=0x30000, topk=64, batch=2, s_q=1, h=16,
             scale=0.07, sink=None, meta=0x50000, parts=4, ws=0x60000, out=0x70000, lse=0x80000,
             err=None, stream=None)
    a.update(over)
    return binding.lib().mla_sparse_decode(a["q"], a["kv"], a["s_kv"], a["idx"], a["topk"], a["batch"],
                                           a["s_q"], a["h"], a["scale"], a["sink"], a["meta"], a["parts"],
                                           a["ws"], a["out"], a["lse"], a["err"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(idx=None), -1), (dict(meta=None), -1), (dict(topk=0), -2), (dict(s_kv=0), -2),
    (dict(h=100), -2), (dict(scale=-1.0), -2), (dict(kv=0x20008), -3),
])
def test_sparse_decode_rejects_bad_arguments_before_launch(over, code):
    # the attention sink is optional: a NULL sink never fails validation
    assert _call_sparse(**over) == code


def test_binding_checks_the_attention_sink():
    import torch
    cpu = torch.zeros(16, dtype=torch.float32)
    with pytest.raises(ValueError):   # must live on the GPU
        binding.mla_combine(torch.zeros(4, dtype=torch.int32), 2, 1, 16, 4, cpu, cpu, cpu,
                            attn_sink=cpu)


def test_wait_timeout_check_rejects_a_null_error_word():
    assert binding.lib().mla_check_wait_timeout(None, None) == -1   # MLA_ERR_NULL


def test_binding_constants_match_the_header():
    """The binding's status, device-error and format constants are the
    header's #defines (a value the kernels OR into the error word must mean
    the same thing on both sides)."""
    import re
    text = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    defines = {m.group(1): int(m.group(2)) for m in
               re.finditer(r"#define (MLA_(?:DEVERR|KV)_\w+)\s+\(?(-?\d+)u?\)?", text)}
    assert {"MLA_DEVERR_BAD_PAGE", "MLA_DEVERR_BAD_INDEX", "MLA_DEVERR_TIMEOUT",
            "MLA_DEVERR_METADATA", "MLA_KV_BF16", "MLA_KV_FP8_656"} <= set(defines)
    for name, value in defines.items():
        assert getattr(binding, name) == value, name
