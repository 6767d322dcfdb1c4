"""Benchmark of MLA decode (absorbed, paged latent KV) on GB300.

Metric: decode TFLOP/s on the DeepSeek-V3-shaped dense workload (b=64, s_q=1,
h=128, 576/512, every request 4096 cached tokens, 64-token pages, shuffled
page table), with the effective KV GB/s and the fraction of the GB300
roofline min(bf16 peak, HBM BW x arithmetic intensity).

One step = one pass of the whole decode path on one batch: schedule metadata
(device kernel), split-KV kernel, combine kernel.  Steps are replayed from a
CUDA graph; two full input sets (each larger than L2) alternate so that every
step reads its KV cache from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only reference this
method has) on the host cores, on the same workload and metric.  Under
torchrun every rank runs its own replica of the batch (weak scaling, no
data-path collective); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode TFLOPS & KV GB/s (b=64,h=128,t=4096) as fraction of GB300 roofline"
UNIT = "TFLOP/s"
WORKLOAD = "dense_v3"
GRAPH_STEPS = 10
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}


# --------------------------------------------------------------------- utils

def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest per-rank value over all ranks (the slowest rank times the
    job); `x` itself when there is one rank.  Uses the default process group
    (NCCL on the GPU machine, gloo in the CPU tests)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, ms_per_step: float, world: int) -> float:
    """Whole-job rate: every rank processes `units_per_rank` per step (weak
    scaling), the step takes the slowest rank's `ms_per_step`."""
    return units_per_rank / (ms_per_step * 1e-3) * world


def check_world(gpus: int, world: int):
    """None when the launch matches --gpus, else why not.  Every GPU runs one
    process (one replica of the batch), so N > 1 needs a launcher that starts
    N ranks (torchrun) and sets WORLD_SIZE = N."""
    if gpus < 1:
        return f"--gpus must be >= 1 (got {gpus})"
    if gpus != world:
        return (f"--gpus {gpus} but WORLD_SIZE={world}: launch one process per GPU, e.g. "
                f"python -m torch.distributed.run --nproc-per-node {gpus} bench.py --gpus {gpus}")
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def kernel_source_hash():
    """Hash of the sources the decode kernels compile from (mla_decode.cu and
    every header); ncu traffic figures are valid only for it.  The schedule,
    combine and no-allocation translation units are not part of it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cuh", ".h")) or name == "mla_decode.cu":
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "mla_decode.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(kernel, {}).get(workload)
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms", str(self.period_ms)],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float, t_end: float):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        import datetime
        clocks, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        in_window = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, mx = float(r[2]), float(r[3])
            except ValueError:
                continue
            in_window.append((t_start - 0.06 <= ts <= t_end + 0.06, clk, mx, r[6:10]))
        chosen = [x for x in in_window if x[0]] or in_window
        for _, clk, mx, flags in chosen:
            clocks.append(clk)
            maxes.append(mx)
            for name, v in zip(names, flags):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(clocks) if clocks else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(clocks),
                "in_timed_window": sum(1 for x in in_window if x[0])}


# ---------------------------------------------------------------- ours (GPU)

def run_ours(args, rank, world, local_rank):
    import torch

    from mla_decode_attention_gb300 import binding, roofline, workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.config]
    peaks = load_peaks()

    # two input sets (each > L2), pinned host copies for the end-to-end leg
    sets_host = [workloads.make_inputs(w, seed=w.seed + 1000 * rank + k) for k in range(2)]
    for s in sets_host:
        for key, v in list(s.items()):
            if torch.is_tensor(v):
                s[key] = v.pin_memory()
    sets = [{k: (v.to(dev) if hasattr(v, "to") and hasattr(v, "pin_memory") else v)
             for k, v in s.items()} for s in sets_host]
    b, s_q, h = w.b, w.s_q, w.h
    parts = binding.mla_num_sm_parts(local_rank, h)
    # One set of schedule / workspace / output buffers reused every step, as a
    # serving loop reuses them; the inputs alternate between two sets.
    bufs = [binding.DecodeBuffers(b, s_q, h, dev, parts)]
    # the split-only timing replays the split kernel without the schedule
    # kernel, so it keeps one schedule per input set (lengths differ per set)
    split_meta = [torch.empty_like(bufs[0].metadata) for _ in range(2)]
    stream = torch.cuda.Stream(device=dev)
    scale = workloads.SOFTMAX_SCALE

    sparse = w.kind == "sparse"
    fmt = binding.MLA_KV_FP8_656 if w.kind == "fp8" else binding.MLA_KV_BF16
    in_keys = ("q", "kv", "indices") if sparse else ("q", "kv_cache", "block_table",
                                                      "cache_seqlens")

    def step(k, split_only=False):
        s, buf = sets[k % 2], bufs[0]
        meta = split_meta[k % 2] if split_only else buf.metadata
        if sparse:
            if not split_only:
                binding.mla_get_metadata(None, b, s_q, False, w.topk, parts, buf.metadata, stream)
            if w.prefill and not split_only:  # b query tokens in the prefill call's layouts
                binding.mla_sparse_prefill(s["q"][:, 0], s["kv"], s["indices"][:, 0], scale, meta, parts,
                                           buf.workspace, buf.out[:, 0], buf.lse[:, :, 0], buf.err, stream)
            else:
                fn = binding.mla_sparse_decode_splitkv if split_only else binding.mla_sparse_decode
                fn(s["q"], s["kv"], s["indices"], scale, meta, parts, buf.workspace, buf.out,
                   buf.lse, buf.err, stream)
        elif not split_only:
            binding.mla_get_metadata(s["cache_seqlens"], b, s_q, True, 0, parts, buf.metadata,
                                     stream)
            binding.mla_decode(s["q"], s["kv_cache"], fmt, s["block_table"],
                               s["cache_seqlens"], scale, True, buf.metadata, parts,
                               buf.workspace, buf.out, buf.lse, buf.err, stream)
        else:
            binding.mla_decode_splitkv(s["q"], s["kv_cache"], fmt,
                                       s["block_table"], s["cache_seqlens"], scale, True,
                                       meta, parts, buf.workspace, buf.out, buf.lse,
                                       buf.err, stream)

    # one schedule per input set for the split-only graph
    with torch.cuda.stream(stream):
        for k in range(2):
            if sparse:
                binding.mla_get_metadata(None, b, s_q, False, w.topk, parts, split_meta[k], stream)
            else:
                binding.mla_get_metadata(sets[k]["cache_seqlens"], b, s_q, True, 0, parts,
                                         split_meta[k], stream)
        for k in range(2):
            step(k)
    torch.cuda.synchronize(dev)
    if args.profile:
        # a few eager steps only: the command ncu captures
        with torch.cuda.stream(stream):
            for k in range(args.profile):
                step(k)
        torch.cuda.synchronize(dev)
        return {"profile_steps": args.profile, "errors": [int(bf.err.item()) for bf in bufs]}

    def capture(split_only):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for k in range(GRAPH_STEPS):
                step(k, split_only)
            g.capture_end()
        return g

    g_step = capture(False)
    g_split = capture(True)
    torch.cuda.synchronize(dev)

    def replay(g, n_steps):
        reps = n_steps // GRAPH_STEPS
        rest = n_steps - reps * GRAPH_STEPS
        for _ in range(reps):
            g.replay()
        with torch.cuda.stream(stream):
            for k in range(rest):
                step(k)

    # warm-up
    with torch.cuda.stream(stream):
        replay(g_step, max(args.warmup, 3))
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- timed region: exactly K steps
    sampler = ClockSampler(dev.index)
    with sampler:
        barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        e0.record(stream)
        with torch.cuda.stream(stream):
            replay(g_step, args.steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        t_wall1 = time.time()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    clocks = sampler.summary(t_wall0, t_wall1)
    ms_per_step = ms_total / args.steps

    # ---- dominant kernel alone: split-KV launches back to back, same stream
    n_split = max(GRAPH_STEPS, (min(args.steps, 2000) // GRAPH_STEPS) * GRAPH_STEPS)
    torch.cuda.synchronize(dev)
    k0 = torch.cuda.Event(enable_timing=True)
    k1 = torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(n_split // GRAPH_STEPS):
            g_split.replay()
    k1.record(stream)
    torch.cuda.synchronize(dev)
    split_ms = k0.elapsed_time(k1) / n_split

    errs = [int(bf.err.item()) for bf in bufs]

    # ---- end to end through the public API with host buffers
    n_e2e = max(3, min(args.steps, 50))
    h2d = sum(sets_host[0][k].numel() * sets_host[0][k].element_size() for k in in_keys)
    d2h = bufs[0].out.numel() * 2 + bufs[0].lse.numel() * 4
    out_host = [torch.empty(bufs[0].out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_host = [torch.empty(bufs[0].lse.shape, dtype=torch.float32).pin_memory() for _ in range(2)]

    # The inputs go up on a copy stream of their own, overlapping the previous
    # step's compute and read-back: a set's device buffers are rewritten only
    # once the step two back, which read them, has finished; the step waits
    # for its copies.  (Slicing the copies over 2 or 4 streams was no faster.)
    copy_stream = torch.cuda.Stream(device=dev)
    step_done = [torch.cuda.Event() for _ in range(2)]
    copied = torch.cuda.Event()

    def e2e_step(k):
        s_h, s_d, buf = sets_host[k % 2], sets[k % 2], bufs[0]
        copy_stream.wait_event(step_done[k % 2])
        with torch.cuda.stream(copy_stream):
            for key in in_keys:
                s_d[key].copy_(s_h[key], non_blocking=True)
        copied.record(copy_stream)
        stream.wait_event(copied)
        step(k)
        step_done[k % 2].record(stream)
        out_host[k % 2].copy_(buf.out, non_blocking=True)
        lse_host[k % 2].copy_(buf.lse, non_blocking=True)

    with torch.cuda.stream(stream):
        for k in range(3):
            e2e_step(k)
    torch.cuda.synchronize(dev)
    barrier()
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for ev in step_done:  # no copy of the timed steps starts before x0
        ev.record(stream)
    with torch.cuda.stream(stream):
        for k in range(n_e2e):
            e2e_step(k)
    x1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(x0.elapsed_time(x1) / n_e2e, world, dev)

    # ---- accounting
    flops_nominal = None
    if sparse:
        idx = sets_host[0]["indices"]
        valid = ((idx >= 0) & (idx < w.s_kv)).sum(dim=-1).flatten().tolist()
        flops, flops_nominal, bytes_, kv_bytes = roofline.sparse_counts(valid, h, w.topk)
        seqlens = [w.topk] * b
    else:
        seqlens = sets_host[0]["cache_seqlens"].tolist()
        flops, bytes_, kv_bytes = roofline.dense_counts(seqlens, s_q, h, causal=True,
                                                        fp8=(w.kind == "fp8"))
    tflops = job_rate(flops, ms_per_step, world) / 1e12
    kv_gbs = job_rate(kv_bytes, ms_per_step, world) / 1e9
    ai = flops / bytes_
    roof_tf = min(peaks["bf16_tflops"], peaks["hbm_gbs"] * ai / 1e3)
    split_gbs = bytes_ / (split_ms * 1e-3) / 1e9
    bound = "hbm" if peaks["hbm_gbs"] * ai / 1e3 < peaks["bf16_tflops"] else "tensor"
    if w.prefill:
        # sparse prefill: the pool is read again by every query token, mostly
        # from L2 (the byte count above counts each gathered row per token);
        # the pages quote this call in TFLOPS, as compute-bound work
        bound = "tensor"
        roof_tf = peaks["bf16_tflops"]
    if bound == "hbm":
        achieved, peak, unit = split_gbs, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = flops / (split_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    # the split kernel the library dispatches to: two-SM kernel for 128 bf16 query rows
    kernel_name = "mla_pair_kernel" if (w.kind in ("dense", "sparse") and h == 128) else "mla_splitkv_kernel"
    traffic = recorded_traffic(kernel_name, args.config)

    result = {
        "metric": METRIC, "value": round(tflops, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q and latent cache, shuffled page table)"
                if not sparse else "synthetic (seeded N(0,1) pool, top-k indices, peaked rows)",
        "config": {"workload": WORKLOAD if args.config == WORKLOAD else args.config,
                   "batch": b, "s_q": s_q, "h_q": h, "d_qk": 576, "d_v": 512,
                   "seqlen": seqlens[0] if len(set(seqlens)) == 1 else "mixed",
                   "page_block": 64, "num_sm_parts": parts,
                   "l2": ("inputs larger than L2 (KV per set > 129 MB, two sets alternate)"
                          if kv_bytes > 129e6 else
                          "KV working set fits in L2 (two sets alternate); effective GB/s may exceed HBM"),
                   "buffers": "schedule, workspace and outputs reused every step (as a serving loop)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_gbs": round(kv_gbs, 1),
        "roofline_fraction": round(tflops / world / roof_tf, 4),
        "roofline_tflops": round(roof_tf, 1),
        "arithmetic_intensity": round(ai, 1),
        "algorithmic": {"flops": flops, "bytes": bytes_, "kv_bytes": kv_bytes,
                        "flops_nominal_topk": flops_nominal},
        "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel_name, "kernel_ms": round(split_ms, 5),
                     "peak_source": f"{peaks.get('source')} (MEASURED_PEAKS.json "
                                    f"{'burst copy' if bound == 'hbm' else 'bf16 GEMM burst'})"},
        "e2e": {"value": round(job_rate(flops, e2e_ms, world) / 1e12, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "note": "all call inputs (" + ", ".join(in_keys) + ") copied from pinned "
                        "host memory on a copy stream (overlapping the previous step) and "
                        "out+lse copied back every step"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "device_error_word": errs,
    }
    return result


# ------------------------------------------------------------ oracle on CPU

def oracle_worker(argv):
    """Subprocess: time the fp64 oracle on `n_req` requests of the workload."""
    import numpy as np

    import oracle
    from mla_decode_attention_gb300 import roofline, workloads

    cfg, n_req, reps = argv[0], int(argv[1]), int(argv[2])
    w = workloads.WORKLOADS[cfg]
    inp = workloads.make_inputs(w)
    import torch
    if w.kind == "sparse":  # n_req query tokens of the top-k sparse workload
        q = inp["q"].contiguous().view(torch.int16).numpy().view(np.uint16)
        pool = inp["kv"].contiguous().view(torch.int16).numpy().view(np.uint16)
        idx = inp["indices"].numpy()
        toks = [(bi, j) for bi in range(w.b) for j in range(w.s_q)][:n_req]
        times = []
        for _ in range(reps):
            t0 = time.perf_counter()
            oracle.sparse_decode(q, pool, idx, inp["softmax_scale"], toks)
            times.append(time.perf_counter() - t0)
        valid = [int(((idx[bi, j] >= 0) & (idx[bi, j] < w.s_kv)).sum()) for bi, j in toks]
        flops, _, _, _ = roofline.sparse_counts(valid, w.h, w.topk)
        print(json.dumps({"times": times, "flops": flops, "requests": len(toks)}))
        return
    q = inp["q"].contiguous().view(torch.int16).numpy().view(np.uint16)
    kv = inp["kv_cache"].contiguous().view(torch.int16).numpy().view(np.uint16)
    bt = inp["block_table"].numpy()
    sl = inp["cache_seqlens"].numpy()
    rows = [(bi, j) for bi in range(min(n_req, w.b)) for j in range(w.s_q)]
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.dense_decode(q, kv, bt, sl, inp["softmax_scale"], True, rows)
        times.append(time.perf_counter() - t0)
    flops, _, _ = roofline.dense_counts(sl[:min(n_req, w.b)].tolist(), w.s_q, w.h)
    print(json.dumps({"times": times, "flops": flops, "requests": min(n_req, w.b)}))


def workloads_module():
    from mla_decode_attention_gb300 import workloads
    return workloads


def time_oracle(cfg, n_req, reps, threads):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker", cfg,
                        str(n_req), str(reps)], capture_output=True, text=True, env=env,
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(cfg):
    threads = os.cpu_count() or 1
    probe = time_oracle(cfg, 1, 1, threads)
    per_req = max(probe["times"][0], 1e-3)
    w = workloads_module().WORKLOADS[cfg]
    n_all = w.b * w.s_q if w.kind == "sparse" else w.b
    n_req = max(1, min(n_all, int(20.0 / per_req)))
    # repeat the sample until it is about 15 s of CPU work (the whole dense
    # workload takes well under a second in numpy), and take the median pass
    reps = max(1, min(30, int(15.0 / (per_req * n_req))))
    res = time_oracle(cfg, n_req, reps, threads)
    t = sorted(res["times"])[len(res["times"]) // 2]
    what = (f"{res['requests']} of {w.b * w.s_q} query tokens of the same workload (all {w.h} heads, "
            f"{w.topk} index slots each)" if w.kind == "sparse" else
            f"{res['requests']} of {w.b} requests of the same workload (all {w.h} heads)")
    return {"value": round(res["flops"] / t / 1e12, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{what}, fp64 numpy, median of {reps} passes of {t:.2f} s each"}


def run_reference(args):
    threads = os.cpu_count() or 1
    probe = time_oracle(args.config, 1, 1, threads)
    per_req = max(probe["times"][0], 1e-3)
    total_steps = args.steps + args.warmup
    n_req = max(1, min(64, int(150.0 / (per_req * max(total_steps, 1)))))
    res = time_oracle(args.config, n_req, total_steps, threads)
    times = res["times"][args.warmup:] or res["times"]
    t = sum(times) / len(times)
    v = res["flops"] / t / 1e12
    sample = (f"{res['requests']} of 64 requests per step (all 128 heads, 4096 keys), fp64 "
              f"numpy oracle")
    return {"metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded workload)", "impl": "reference",
            "config": {"workload": WORKLOAD if args.config == WORKLOAD else args.config},
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------- main

def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-worker":
        oracle_worker(sys.argv[2:])
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", type=int, default=0,
                    help="run only this many eager steps (for ncu captures) and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    problem = check_world(args.gpus, world)
    if problem:
        print(problem, file=sys.stderr, flush=True)
        sys.exit(2)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    result = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline and not args.profile:
            result["cpu_baseline"] = cpu_baseline(args.config)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
